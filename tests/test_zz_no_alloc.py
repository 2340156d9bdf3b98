"""w8a8_gemm_no_alloc against w8a8_gemm, through the C ABI.

The allocation-free entry point serves callers that cannot hand the library a workspace (a plugin
that sees only its input and output pointers, or a request path that must not call cudaMalloc);
it runs the same kernel on a scratch area held in the library's own device memory.  Its output
must equal the workspace entry point's bit for bit (the W8A8 tolerance), call after call, since
each call reuses the scratch the previous one left behind.

This file is collected last so that a run stopping at its first failure has already run every
other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import int8_weight_gemm_gb300 as lib8
import synth
from gpu_util import W8A8Case, bf16_bits

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _no_alloc(case, out, blocks=0, flags=0):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib8.lib().w8a8_gemm_no_alloc(_ptr(case.x), _ptr(case.xs), _ptr(case.Wp), _ptr(case.ws_scale), _ptr(out),
                                         case.M, case.K, case.N, blocks, flags, stream)


def _no_alloc_status():
    v = ctypes.c_uint32(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib8.lib().w8a8_gemm_no_alloc_status(stream, ctypes.byref(v)) == 0
    return int(v.value)


# M > 32 runs the tensor-memory arm (two launches; its scratch holds the fp16 activations too).
@pytest.mark.parametrize("M,K,N,blocks", [(16, 4096, 1536, 0), (5, 512, 200, 7), (32, 2048, 4096, 0),
                                          (64, 4096, 1536, 0), (100, 2048, 384, 7), (128, 2048, 4096, 0)])
def test_no_alloc_matches_workspace_entry_point_twice(M, K, N, blocks):
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=M + K + N)
    case = W8A8Case(x, xs, W, ws, blocks=blocks)
    ref = bf16_bits(case.run())
    for _ in range(2):   # the second call starts from the scratch the first one left behind
        out = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
        assert _no_alloc(case, out, blocks=blocks) == 0, lib8.lib().w8a8_last_error()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bf16_bits(out), ref)


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    # M = 32 at N = 131072 + 64 has 2049 tiles of 16 KiB of split-tile accumulators: more than the
    # 16 MiB area.
    M, K, N = 32, 32, 131136
    x = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    xs = torch.ones(M, dtype=torch.float32, device="cuda")
    wp = torch.zeros(lib8.w8a8_packed_weight_bytes(K, N), dtype=torch.uint8, device="cuda")
    wsc = torch.ones(N, dtype=torch.float32, device="cuda")
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert lib8.w8a8_workspace_bytes(M, K, N) > (16 << 20)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib8.lib().w8a8_gemm_no_alloc(_ptr(x), _ptr(xs), _ptr(wp), _ptr(wsc), _ptr(out), M, K, N, 0, 0, stream)
    assert rc == 4
    assert b"16 MiB" in lib8.lib().w8a8_last_error()


def test_no_alloc_calls_with_different_plans_in_a_row():
    # Each call starts from what a call with another plan left in the shared area: another word
    # format, another tile count, the tensor-memory arm's counters, planes and fp16 activations.
    shapes = [(128, 2048, 4096, 0), (16, 4096, 1536, 7), (5, 512, 200, 0), (64, 1024, 512, 16),
              (32, 65536, 64, 8), (1, 512, 256, 0)]
    cases = []
    for (M, K, N, blocks) in shapes:
        x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=2 * M + K)
        case = W8A8Case(x, xs, W, ws, blocks=blocks)
        cases.append((case, blocks, bf16_bits(case.run())))
    for _ in range(2):
        for case, blocks, ref in cases:
            out = torch.full((case.M, case.N), 7.0, dtype=torch.bfloat16, device="cuda")
            assert _no_alloc(case, out, blocks=blocks) == 0, lib8.lib().w8a8_last_error()
            torch.cuda.synchronize()
            np.testing.assert_array_equal(bf16_bits(out), ref)
    assert _no_alloc_status() == 0


def test_no_alloc_pdl_calls_replay_from_a_graph():
    # After a first eager call (the per-context set-up), calls with W8A8_FLAG_PDL are captured
    # into a CUDA graph and replayed: every replay gives the workspace entry point's bits.
    M, K, N = 16, 4096, 1536
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=99)
    case = W8A8Case(x, xs, W, ws)
    ref = bf16_bits(case.run())
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert _no_alloc(case, out, flags=lib8.W8A8_FLAG_PDL) == 0
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            assert _no_alloc(case, out, flags=lib8.W8A8_FLAG_PDL) == 0
    for _ in range(4):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bf16_bits(out), ref)
    assert _no_alloc_status() == 0


def test_no_alloc_status_reports_a_device_timeout_and_clears():
    # The test hook makes one warp's bounded wait run out: the status word of the area records
    # it, the status call clears it, and the next call is exact again (each call clears the
    # regions its kernel needs zeroed).
    M, K, N = 16, 512, 256
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=5)
    case = W8A8Case(x, xs, W, ws)
    ref = bf16_bits(case.run())
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert _no_alloc_status() == 0
    assert _no_alloc(case, out, flags=lib8.W8A8_FLAG_TEST_STALL) == 0
    torch.cuda.synchronize()
    assert _no_alloc_status() == lib8.W8A8_DEV_WAIT_TIMEOUT
    assert _no_alloc_status() == 0
    assert _no_alloc(case, out) == 0
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_bits(out), ref)
    assert _no_alloc_status() == 0

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

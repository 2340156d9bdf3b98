"""The device fault paths of both W8A8 arms, made to happen without faulting or hanging the GPU.

- W8A8_DEV_COUNTER_CORRUPT: an arrival count that no contributor can bring to its end is written
  into a zeroed workspace from the host.  Nothing waits on that word (the combine never waits for
  another CTA), so the call ends normally with the bit set, and no output of that tile is stored.
- W8A8_DEV_WAIT_TIMEOUT: W8A8_FLAG_TEST_STALL makes one warp wait, with a bound of a few
  milliseconds, on a barrier that nothing completes; the wait runs out and every role of the CTA
  returns through the same bounded exit a real timeout takes.

Each case then zeroes the workspace again and checks that the next call is bit-exact with a
clean status, so the context stays usable.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import int8_weight_gemm_gb300 as lib8
import oracle
import synth
from gpu_util import W8A8Case, bf16_bits

pytestmark = pytest.mark.gpu


def _clean_call_is_exact(case, x, xs, W, ws):
    lib8.w8a8_workspace_init(case.ws)
    out = case.run()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_bits(out), oracle.w8a8_gemm(x, xs, W, ws))
    assert case.status() == 0


@pytest.mark.parametrize("K,N,blocks,count_word", [
    (2048, 384, 64, 0xFFC0000000000000),    # two elements per word: the count is the top 10 bits
    (65536, 64, 8, 0xFFF0000000000000),     # one element per word: the count is bits 52 and up
])
def test_decode_arm_reports_a_dirty_combine_word(K, N, blocks, count_word):
    M = 16
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=K + N)
    case = W8A8Case(x, xs, W, ws, blocks=blocks)
    plan = lib8.w8a8_plan(M, K, N, blocks)
    assert plan["blocks"] > plan["n_tiles"] and plan["tensor_memory"] == 0   # every tile is split
    assert (plan["combine_pack_bits"] != 0) == (count_word == 0xFFC0000000000000)
    words = case.ws[256:].view(torch.int64)
    words[0] = np.int64(np.uint64(count_word).view(np.int64))   # first word of tile 0
    torch.cuda.synchronize()
    out = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    case.run(out=out)
    torch.cuda.synchronize()
    assert case.status() == lib8.W8A8_DEV_COUNTER_CORRUPT
    # the element(s) of that word were never finished; every other output is right
    got, ref = bf16_bits(out), oracle.w8a8_gemm(x, xs, W, ws)
    assert 1 <= np.count_nonzero(got != ref) <= 2
    _clean_call_is_exact(case, x, xs, W, ws)


def test_tensor_memory_arm_reports_a_dirty_counter():
    M, K, N, blocks = 64, 2048, 512, 16
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=77)
    case = W8A8Case(x, xs, W, ws, blocks=blocks)
    plan = lib8.w8a8_plan(M, K, N, blocks)
    assert plan["tensor_memory"] == 1 and plan["blocks"] > plan["n_tiles"]
    counters = case.ws[256:256 + 4 * plan["n_tiles"]].view(torch.int32)
    counters[0] = np.int32(np.uint32(0xFFFFFFF0).view(np.int32))
    torch.cuda.synchronize()
    case.run()
    torch.cuda.synchronize()
    assert case.status() == lib8.W8A8_DEV_COUNTER_CORRUPT
    _clean_call_is_exact(case, x, xs, W, ws)


@pytest.mark.parametrize("M,K,N,blocks", [
    (16, 512, 256, 0),       # one segment per CTA
    (16, 4096, 1536, 7),     # several segments per CTA: the combine warp gives up as well
    (64, 1024, 512, 0),      # the tensor-memory arm (forced): issuers, converters and producers
    (64, 1024, 512, -1),     # the same M through the automatic plan: 32-row decode chunks
])
def test_a_stalled_wait_times_out_and_the_call_returns(M, K, N, blocks):
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=M * K)
    forced = M > 32 and blocks == 0
    case = W8A8Case(x, xs, W, ws, blocks=max(blocks, 0))
    t0 = time.perf_counter()
    case.run(flags=lib8.W8A8_FLAG_TEST_STALL | (lib8.W8A8_FLAG_TENSOR_MEMORY_ARM if forced else 0))
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = case.status()
    if blocks < 0:
        # Row chunks: the first chunk's timeout leaves its split tiles' words unfinished, and the
        # next chunk, on the same workspace, finds them dirty and says so as well.
        assert status & lib8.W8A8_DEV_WAIT_TIMEOUT and not status & ~3
    else:
        assert status == lib8.W8A8_DEV_WAIT_TIMEOUT
    assert elapsed < 0.5, f"the stalled call took {elapsed:.3f} s"
    _clean_call_is_exact(case, x, xs, W, ws)

"""32 < M <= 128 through the automatic plan: where the cost model picks 32-row decode chunks (small
weights), the chunked call is bit-exact against the oracle, outputs and int32 accumulators, plain
and with PDL, repeated on one workspace; where it picks the tensor-memory arm (large weights), the
plan says so.  The tensor-memory arm itself is tested with the arm forced in test_w8a8_tc_gpu.py."""
import numpy as np
import pytest
import torch

import int8_weight_gemm_gb300 as lib8
import oracle
import synth
from gpu_util import W8A8Case, bf16_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,N", [(33, 4096, 1536), (40, 2048, 520), (64, 4096, 2560), (95, 2048, 4096),
                                   (96, 4096, 1536), (100, 1024, 200), (128, 1024, 512)])
def test_row_chunks_are_bit_exact(M, K, N):
    plan = lib8.w8a8_plan(M, K, N)
    assert plan["tensor_memory"] == 0 and plan["row_chunks"] == -(-M // 32)
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=M * 7 + N)
    case = W8A8Case(x, xs, W, ws)
    ref = oracle.w8a8_gemm(x, xs, W, ws)
    ref_acc = oracle.w8a8_acc(x, W)
    for flags in (0, lib8.W8A8_FLAG_PDL, 0):
        out, acc = case.run_acc(flags=flags)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bf16_bits(out), ref)
        np.testing.assert_array_equal(acc.cpu().numpy().astype(np.int64), ref_acc)
        assert case.status() == 0


def test_large_weights_keep_the_tensor_memory_arm():
    for M, K, N in ((128, 4096, 24576), (64, 12288, 4096), (96, 4096, 24576)):
        assert lib8.w8a8_plan(M, K, N)["tensor_memory"] == 1
    # an explicit CTA count selects the tensor-memory arm whatever the weight size
    assert lib8.w8a8_plan(64, 4096, 1536, blocks=76)["tensor_memory"] == 1

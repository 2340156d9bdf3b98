"""Quantisation kernels on the GPU against the oracle, bit for bit: the W8A8 activations' int8
quants and per-row scales, Q8_0 from BF16 weights, and the ggml-block <-> split re-layout; plus the
chains a caller runs (quantise, then the GEMM or the Q8_0 read)."""
import numpy as np
import pytest
import torch

import int8_weight_gemm_gb300 as lib8
import oracle
import synth
from gpu_util import W8A8Case, bf16_bits

pytestmark = pytest.mark.gpu


def _bf16(rng, shape, scale=1.0):
    return torch.tensor((rng.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _special_rows(K):
    # a zero row, exact ties of x / scale (halves away from zero), a negative amax, tiny values
    r_zero = torch.zeros(K)
    r_tie = torch.zeros(K)
    r_tie[:6] = torch.tensor([0.5, 1.5, 2.5, -0.5, -1.5, -126.5]) / 8
    r_tie[-1] = 127.0 / 8
    r_neg = torch.full((K,), 0.25)
    r_neg[3] = -127.0 / 4
    r_tiny = torch.full((K,), 3.0e-38)
    r_tiny[1] = -1.0e-37
    return torch.stack([r_zero, r_tie, r_neg, r_tiny]).to(torch.bfloat16)


@pytest.mark.parametrize("M,K", [(1, 512), (16, 4096), (32, 12288), (7, 136), (3, 8), (200, 2048)])
def test_quantize_activations_bit_exact(M, K):
    rng = np.random.default_rng(M * 7 + K)
    x = _bf16(rng, (M, K), 3.0)
    if M >= 4 and K >= 8:
        x[:4] = _special_rows(K)
    xq, xs = lib8.w8a8_quantize_activations(x.cuda())
    torch.cuda.synchronize()
    ref_q, ref_s = oracle.w8a8_quantize_rows(_bits(x))
    np.testing.assert_array_equal(xq.cpu().numpy(), ref_q)
    np.testing.assert_array_equal(xs.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


@pytest.mark.parametrize("N,K", [(320, 4096), (4096, 320), (33, 64), (1, 32), (100, 1024)])
def test_q8_0_quantize_bit_exact(N, K):
    rng = np.random.default_rng(N + 3 * K)
    w = _bf16(rng, (N, K), 0.02)
    if N >= 4:
        w[:4, :32] = _special_rows(32)          # zero block, ties, negative amax, tiny values
    q, d = lib8.q8_0_quantize(w.cuda())
    torch.cuda.synchronize()
    ref_q, ref_d = oracle.q8_0_quantize(_bits(w))
    np.testing.assert_array_equal(q.cpu().numpy(), ref_q)
    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint16), ref_d)


@pytest.mark.parametrize("N,K", [(320, 4096), (4096, 320), (3, 96)])
def test_relayout_both_ways(N, K):
    rng = np.random.default_rng(K + 2 * N)
    blocks = rng.integers(0, 256, (N, K // 32, 34)).astype(np.uint8)
    q, d = lib8.q8_0_split_from_blocks(torch.from_numpy(blocks).cuda(), K, N)
    torch.cuda.synchronize()
    ref_q, ref_d = oracle.q8_0_split_from_blocks(blocks, K, N)
    np.testing.assert_array_equal(q.cpu().numpy(), ref_q)
    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint16), ref_d)
    back = lib8.q8_0_blocks_from_split(q, d)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(back.cpu().numpy(), blocks)
    np.testing.assert_array_equal(oracle.q8_0_blocks_from_split(ref_q, ref_d), blocks)


def test_quantise_then_gemm_chain():
    # bf16 activations -> (x_q, x_scale) on the GPU -> the W8A8 GEMM; the oracle does both steps.
    M, K, N = 16, 4096, 1536
    rng = np.random.default_rng(5)
    x = _bf16(rng, (M, K))
    _, _, W, ws = synth.w8a8_inputs(M, K, N, seed=5)
    xq_d, xs_d = lib8.w8a8_quantize_activations(x.cuda())
    ref_q, ref_s = oracle.w8a8_quantize_rows(_bits(x))
    case = W8A8Case(ref_q, ref_s, W, ws)
    out = lib8.w8a8_gemm(xq_d, xs_d, case.Wp, case.ws_scale, case.ws, N)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_bits(out), oracle.w8a8_gemm(ref_q, ref_s, W, ws))


def test_quantise_then_q8_0_read_chain():
    # BF16 weights -> Q8_0 split layout on the GPU -> the Q8_0 read, within its tolerance of the
    # oracle's read of the oracle's quantisation (which the GPU's reproduces bit for bit).
    T, K, N = 6, 4096, 320
    rng = np.random.default_rng(6)
    w = _bf16(rng, (N, K), 0.02)
    x = _bf16(rng, (T, K))
    q, d = lib8.q8_0_quantize(w.cuda())
    ws = lib8.alloc_workspace(lib8.q8_0_workspace_bytes(T, K, N))
    y = lib8.q8_0_gemv(x.cuda(), q, d, ws)
    torch.cuda.synchronize()
    ref_q, ref_d = oracle.q8_0_quantize(_bits(w))
    xb = _bits(x)
    ref = oracle.q8_0_gemv(xb, ref_q, ref_d)
    bound = oracle.q8_0_bound(xb, ref_q, ref_d)
    got = oracle.bf16_to_f64(bf16_bits(y))
    assert (np.abs(got - ref) <= bound).all()

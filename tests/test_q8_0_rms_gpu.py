"""Q8_0 read with an RMS-norm prologue on the GPU against the oracle.

y = rs * (x * g) @ (d * q), rs the inverse RMS of each activation row.  Per output the error bound
is 8e-3 * rs[t] * ||x_t * g||_2 * ||w_n||_2: the staged product x * g is rounded once to bf16
(relative 2^-8 per term, bf16 having 8 significant bits: at most 2^-8 * ||x_t * g|| ||w_n|| over the
sum by Cauchy-Schwarz), the output is rounded once to bf16 (2^-8 |y| <= 2^-8 rs ||x_t * g|| ||w_n||),
and fp32 summation and rs add far less (2^-7 = 7.8e-3).  Cases cover the three combine paths of the read (one CTA per tile, a cluster per tile,
split CTAs with the last-arrival combine), ragged N, eps = 0 and large eps, a constant g against
the plain read, graph replay and programmatic dependent launch.
"""
import numpy as np
import pytest
import torch

import int8_weight_gemm_gb300 as lib8
import oracle
import synth
from gpu_util import bf16_bits

pytestmark = pytest.mark.gpu


def _inputs(T, K, N, seed, g_lo=0.5, g_hi=1.5, x_scale=1.0):
    x, q, d = synth.q8_0_inputs(T, K, N, seed=seed)
    x = (x.float() * x_scale).to(torch.bfloat16)
    g = torch.tensor(synth.uniform_f32(seed, "rms.g", (K,), g_lo, g_hi)).to(torch.bfloat16)
    return x, g, q, d


def _run(x, g, q, d, eps, flags=0):
    T, K = x.shape
    N = q.shape[0]
    ws = lib8.alloc_workspace(lib8.q8_0_workspace_bytes(T, K, N))
    dev = torch.device("cuda")
    y = lib8.q8_0_gemv_rms(x.to(dev), g.to(dev), eps, torch.from_numpy(q).to(dev),
                           torch.from_numpy(d.view(np.int16)).to(dev), ws, flags=flags)
    torch.cuda.synchronize()
    assert lib8.w8a8_workspace_status(ws) == 0
    return y, ws


def _check(x, g, q, d, eps):
    y, _ = _run(x, g, q, d, eps)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    gb = g.view(torch.int16).numpy().view(np.uint16)
    ref, _ = oracle.q8_0_rms_gemv(xb, gb, eps, q, d.view(np.uint16))
    bound = oracle.q8_0_rms_bound(xb, gb, eps, q, d.view(np.uint16))
    got = oracle.bf16_to_f64(bf16_bits(y))
    err = np.abs(got - ref)
    assert (err <= bound).all(), f"max err / bound {np.max(err / np.maximum(bound, 1e-300)):.3f}"
    return got, ref


# (K, N): one CTA per tile (K = 320), a cluster per tile (K = 4096), split CTAs (K = 12288, 65536)
@pytest.mark.parametrize("T", [1, 4, 6, 8])
@pytest.mark.parametrize("K,N", [(4096, 320), (320, 4096), (12288, 512), (2048, 100), (32, 8)])
def test_rms_read_within_bound(T, K, N):
    x, g, q, d = _inputs(T, K, N, seed=T * 131 + K + N)
    _check(x, g, q, d, 1e-6)


@pytest.mark.parametrize("eps", [0.0, 1e-6, 4.0])
def test_eps_values_and_the_longest_k(eps):
    x, g, q, d = _inputs(3, 65536, 64, seed=77, x_scale=3.0)
    _check(x, g, q, d, eps)


def test_constant_gamma_is_rs_times_the_plain_read():
    # g = 1: the staged product is x itself (no rounding), so the output is rs times the plain
    # read's sum, rounded once; compared against the plain read of the same bytes.
    T, K, N = 6, 4096, 320
    x, _, q, d = _inputs(T, K, N, seed=9)
    g = torch.ones(K, dtype=torch.bfloat16)
    got, ref = _check(x, g, q, d, 1e-6)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    plain = oracle.q8_0_gemv(xb, q, d.view(np.uint16))
    _, rs = oracle.q8_0_rms_gemv(xb, g.view(torch.int16).numpy().view(np.uint16), 1e-6, q[:1], d[:1].view(np.uint16))
    np.testing.assert_allclose(ref, rs[:, None] * plain, rtol=1e-12)


def test_scaling_x_leaves_the_output_nearly_unchanged():
    # RMS normalisation with eps = 0: doubling x doubles nothing the kernel rounds differently (x * g
    # doubles exactly, the squares quadruple exactly, rs halves exactly), so the bits are equal.
    T, K, N = 4, 4096, 320
    x, g, q, d = _inputs(T, K, N, seed=13)
    y1, _ = _run(x, g, q, d, 0.0)
    y2, _ = _run((x.float() * 2).to(torch.bfloat16), g, q, d, 0.0)
    np.testing.assert_array_equal(bf16_bits(y1), bf16_bits(y2))


@pytest.mark.parametrize("K,N", [(4096, 320), (12288, 512)])
def test_graph_replay_and_pdl_are_bitwise_the_direct_call(K, N):
    T = 6
    x, g, q, d = _inputs(T, K, N, seed=21)
    dev = torch.device("cuda")
    xd, gd = x.to(dev), g.to(dev)
    qd, dd = torch.from_numpy(q).to(dev), torch.from_numpy(d.view(np.int16)).to(dev)
    ws = lib8.alloc_workspace(lib8.q8_0_workspace_bytes(T, K, N))
    direct = bf16_bits(lib8.q8_0_gemv_rms(xd, gd, 1e-5, qd, dd, ws))
    outs = [lib8.q8_0_gemv_rms(xd, gd, 1e-5, qd, dd, ws, flags=lib8.W8A8_FLAG_PDL) for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs:
        np.testing.assert_array_equal(bf16_bits(o), direct)
    y = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lib8.q8_0_gemv_rms(xd, gd, 1e-5, qd, dd, ws, y=y)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        lib8.q8_0_gemv_rms(xd, gd, 1e-5, qd, dd, ws, y=y)
    for _ in range(2):
        y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bf16_bits(y), direct)
    assert lib8.w8a8_workspace_status(ws) == 0


def test_plain_and_rms_reads_share_a_workspace():
    T, K, N = 4, 12288, 512
    x, g, q, d = _inputs(T, K, N, seed=31)
    dev = torch.device("cuda")
    ws = lib8.alloc_workspace(lib8.q8_0_workspace_bytes(T, K, N))
    xd, gd = x.to(dev), g.to(dev)
    qd, dd = torch.from_numpy(q).to(dev), torch.from_numpy(d.view(np.int16)).to(dev)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    for _ in range(2):
        yp = lib8.q8_0_gemv(xd, qd, dd, ws)
        yr = lib8.q8_0_gemv_rms(xd, gd, 1e-6, qd, dd, ws)
        torch.cuda.synchronize()
        ref = oracle.q8_0_gemv(xb, q, d.view(np.uint16))
        assert (np.abs(oracle.bf16_to_f64(bf16_bits(yp)) - ref) <= oracle.q8_0_bound(xb, q, d.view(np.uint16))).all()
        gb = g.view(torch.int16).numpy().view(np.uint16)
        refr, _ = oracle.q8_0_rms_gemv(xb, gb, 1e-6, q, d.view(np.uint16))
        assert (np.abs(oracle.bf16_to_f64(bf16_bits(yr)) - refr) <= oracle.q8_0_rms_bound(xb, gb, 1e-6, q, d.view(np.uint16))).all()
    assert lib8.w8a8_workspace_status(ws) == 0

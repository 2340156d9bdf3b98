"""Q8_0 weight GEMV on the GPU against the fp64 oracle.

Two assertions per output (t, n):
- the stated tolerance, |y_gpu - y64| <= 2e-3 * ||x_t||_2 * ||w_n||_2 (w_n the dequantised weight
  row): the reading of "2e-3, row-norm scaled, per output" as the Cauchy-Schwarz scale of the
  dot product;
- a tight bound derived from the kernel's own arithmetic (tight_bound), far below the stated one,
  so that a defect confined to a few outputs or one block of K cannot hide under it.
"""
import numpy as np
import pytest
import torch

import int8_weight_gemm_gb300 as lib8
import oracle
import synth
from gpu_util import bf16_bits

pytestmark = pytest.mark.gpu

REL = 2e-3


def tight_bound(xb, q, db):
    """Per-output bound of |y_gpu - y64| from the read's arithmetic.  Every product x * q is exact in
    fp32 (bf16 times an int8 value held exactly in bf16); each 32-value block is summed by two
    chained MMAs from zero, scaled by its fp16 scale (exact in fp32) with one fused multiply-add
    per block into the warp's running sum, and the warps' and splits' partials are added in fp32.
    A term therefore passes through at most 32 + K/32 + (warps + splits) <= 32 + 3 K/32 + 8
    roundings, each of relative size at most 2^-23 (truncation as well as round-to-nearest), so
    the fp32 result is within E = 1.01 (32 + 3 K/32 + 8) 2^-23 sum_k |x_k w_k| of y64 (the factor
    1.01 covers the second-order terms); the final round-to-nearest into bf16 (8 significant bits)
    adds at most 2^-8 of the fp32 value's magnitude, plus half of bf16's smallest subnormal."""
    x = oracle.bf16_to_f64(xb)
    d = oracle.f16_to_f64(db)
    w = np.repeat(d, 32, axis=1) * q.astype(np.float64)
    K = x.shape[1]
    S = np.abs(x) @ np.abs(w).T
    y = x @ w.T
    E = 1.01 * (32 + 3 * (K // 32) + 8) * 2.0**-23 * S
    return E + 2.0**-8 * (np.abs(y) + E) + 2.0**-134


def _drop_one_block(xb, q, db):
    """The oracle's result with one block of K left out of every output (block n mod K/32 of row n):
    a planted mistake in a copy of the host-side reference."""
    x = oracle.bf16_to_f64(xb)
    d = oracle.f16_to_f64(db)
    w = np.repeat(d, 32, axis=1) * q.astype(np.float64)
    nb = x.shape[1] // 32
    y = x @ w.T
    for n in range(w.shape[0]):
        b = n % nb
        y[:, n] -= x[:, 32 * b:32 * b + 32] @ w[n, 32 * b:32 * b + 32]
    return y


class Q8Case:
    def __init__(self, T, K, N, seed, T_max=None):
        self.x, self.q, self.d = synth.q8_0_inputs(T, K, N, seed=seed)
        self.xd = self.x.cuda()
        self.qd = torch.from_numpy(self.q).cuda()
        self.dd = torch.from_numpy(self.d.view(np.int16)).cuda()
        self.ws = lib8.alloc_workspace(lib8.q8_0_workspace_bytes(T_max or T, K, N))

    def run(self, y=None, flags=0):
        return lib8.q8_0_gemv(self.xd, self.qd, self.dd, self.ws, y=y, flags=flags)

    def bits(self):
        return self.x.view(torch.int16).numpy().view(np.uint16), self.d.view(np.uint16)

    def reference(self):
        xb, db = self.bits()
        return oracle.q8_0_gemv(xb, self.q, db), oracle.q8_0_bound(xb, self.q, db, REL)


def _check(case):
    """Both assertions; returns (got, ref, max err / stated bound, max err / tight bound)."""
    y = case.run()
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().astype(np.float64)
    ref, bound = case.reference()
    xb, db = case.bits()
    tight = tight_bound(xb, case.q, db)
    err = np.abs(got - ref)
    worst, worst_tight = (err / bound).max(), (err / tight).max()
    assert (err <= bound).all(), f"max err/bound {worst:.3g}"
    assert (err <= tight).all(), f"max err/tight bound {worst_tight:.3g} (err/stated bound {worst:.3g})"
    assert lib8.w8a8_workspace_status(case.ws) == 0
    return got, ref, worst, worst_tight


@pytest.mark.parametrize("T", [1, 4, 6])
@pytest.mark.parametrize("K,N", [(4096, 320), (320, 4096)])
def test_verify_window_shapes(T, K, N):
    c = Q8Case(T, K, N, seed=100 * T + K)
    got, _, worst, worst_tight = _check(c)
    # The tight bound sits far below the stated one, and it catches a planted one-block drop in a
    # copy of the reference on most outputs of every case (the stated bound lets most through).
    xb, db = c.bits()
    tight = tight_bound(xb, c.q, db)
    assert (tight <= oracle.q8_0_bound(xb, c.q, db, REL)).all()
    caught = np.abs(got - _drop_one_block(xb, c.q, db)) > tight
    assert caught.mean() >= 0.85, f"the planted block drop is caught on {caught.mean():.1%} of outputs"


@pytest.mark.parametrize("T,K,N", [(8, 4096, 320), (2, 32, 16), (3, 64, 100), (5, 8192, 33), (7, 1024, 4096),
                                   (1, 65536, 16), (6, 320, 1)])
def test_edge_shapes(T, K, N):
    _check(Q8Case(T, K, N, seed=T + K + N))


def test_rows_beyond_t_untouched_and_replay_bitwise():
    c = Q8Case(4, 4096, 320, seed=9, T_max=8)
    y = torch.full((8, 320), 5.0, dtype=torch.bfloat16, device="cuda")
    c.run(y=y[:4])
    torch.cuda.synchronize()
    assert (y[4:] == 5.0).all()
    direct = bf16_bits(y[:4])
    out = torch.empty((4, 320), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        c.run(y=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        c.run(y=out)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bf16_bits(out), direct)


def test_the_quantised_bytes_are_read():
    # Changing one quant (or one scale) moves exactly the outputs of its row, by the predicted
    # amount: the kernel reads the Q8_0 bytes it is given.
    c = Q8Case(3, 4096, 320, seed=4)
    base = _check(c)[0]
    c.q[17, 1000] = np.int8(-c.q[17, 1000] if c.q[17, 1000] != 0 else 9)
    c.qd = torch.from_numpy(c.q).cuda()
    got = _check(c)[0]
    moved = np.nonzero((got != base).any(axis=0))[0]
    assert set(moved.tolist()) == {17}
    c.d[40, 3] = np.float16(c.d[40, 3] * 2)
    c.dd = torch.from_numpy(c.d.view(np.int16)).cuda()
    got2 = _check(c)[0]
    moved = np.nonzero((got2 != got).any(axis=0))[0]
    assert set(moved.tolist()) == {40}


def test_counters_reset_after_split_calls():
    c = Q8Case(6, 8192, 320, seed=1)      # 256 k-blocks: two CTAs per tile, combined by the last
    n_tiles = (320 + 15) // 16
    # the split layout's partials are in the workspace: per tile 2 splits x (32 lanes x 16 bytes of
    # sums + 32 bytes of the 8 rows' sums of squares, used by the RMS-norm variant)
    assert lib8.q8_0_workspace_bytes(6, 8192, 320) == 256 + 256 + n_tiles * 2 * 34 * 16
    for _ in range(3):
        _check(c)
    n_tiles = (320 + 15) // 16
    ctr = c.ws[256:256 + 4 * n_tiles].view(torch.int32).cpu().numpy()
    assert (ctr == 0).all()


@pytest.mark.parametrize("K,N", [(4096, 320), (320, 4096)])
def test_pdl_launch_matches_plain_launch_bitwise(K, N):
    c = Q8Case(6, K, N, seed=77)
    torch.cuda.synchronize()
    plain = bf16_bits(c.run())
    outs = [c.run(flags=lib8.W8A8_FLAG_PDL) for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs:
        np.testing.assert_array_equal(bf16_bits(o), plain)
    _check(c)


@pytest.mark.parametrize("K,N", [(4096, 320), (8192, 64)])
def test_weights_rewritten_just_before_a_read_are_the_ones_read(K, N):
    # Every read is launched as a programmatic dependent of the work before it; without
    # W8A8_FLAG_PDL it must still behave as plain stream order.  The quants, scales and activations
    # are overwritten on the stream right before each read, with no synchronisation: a read that
    # fetched its weights before those copies had finished would see the old values.  Each output
    # is checked against the oracle of the inputs it should have read (both bounds).
    a, b = Q8Case(4, K, N, seed=91), Q8Case(4, K, N, seed=92)
    dst = Q8Case(4, K, N, seed=93)
    bounds = []
    for src in (a, b):
        ref, stated = src.reference()
        xb, db = src.bits()
        bounds.append((ref, stated, tight_bound(xb, src.q, db)))
    torch.cuda.synchronize()
    outs = []
    for i in range(6):
        src = (a, b)[i % 2]
        dst.qd.copy_(src.qd)
        dst.dd.copy_(src.dd)
        dst.xd.copy_(src.xd)
        outs.append(dst.run())
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        ref, stated, tight = bounds[i % 2]
        err = np.abs(o.float().cpu().numpy().astype(np.float64) - ref)
        assert (err <= stated).all() and (err <= tight).all(), f"read {i}: max err/tight bound {(err / tight).max():.3g}"
        np.testing.assert_array_equal(bf16_bits(o), bf16_bits(outs[i % 2]))
    assert lib8.w8a8_workspace_status(dst.ws) == 0

"""Pins for the oracle: each check compares it with something other than itself.

Witnesses used here, none of which shares code with the oracle:
  * Python integers (exact, unbounded) for brute-force sums on tiny shapes;
  * closed forms (all-ones, int8 extremes, identity-like W, one-hot x, Q8_0 with x = q = 1);
  * invariants (the split-K partition of [0,K) does not change the int32 sums);
  * numpy's IEEE float32 / float16 arithmetic and torch's bfloat16 cast for rounding;
  * exact rational arithmetic (fractions.Fraction) for the Q8_0 fp64 sums;
  * hand-derived bit patterns in tests/golden/.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------------------------------
# IEEE scalars
# ------------------------------------------------------------------------------------------

def test_bf16_rne_golden_ties():
    for f32_hex, bf16_hex in _read_golden("bf16_rne_ties.txt"):
        f = np.array([int(f32_hex, 16)], dtype=np.uint32).view(np.float32)[0]
        assert int(oracle.bf16_from_f32(f)) == int(bf16_hex, 16), f32_hex


def test_bf16_rne_matches_torch_cast():
    # torch's float32 -> bfloat16 cast rounds to nearest even; an independent implementation.
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]            # finite values
    # add the exact halfway patterns, where a wrong tie rule shows up
    ties = (rng.integers(0, 2**16, size=2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    ties = ties[(ties & 0x7F800000) != 0x7F800000]
    bits = np.concatenate([bits, ties])
    f = bits.view(np.float32)
    ours = oracle.bf16_from_f32(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 97, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]
    ours = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    finite = (bits & 0x7C00) != 0x7C00
    ours = oracle.f16_to_f64(bits[finite])
    ref = bits[finite].view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(ours, ref)


def test_dequant_d_times_q_is_exact_in_fp32():
    # The Q8_0 page states that w = d * q is exact in FP32: an fp16 significand (11 bits) times an
    # int8 (8 bits) needs at most 19 bits.  Check it for every finite fp16 scale and every int8.
    d = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    d = d[(d & 0x7C00) != 0x7C00].view(np.float16)
    q = np.arange(-128, 128, dtype=np.int32)
    prod32 = d.astype(np.float32)[:, None] * q.astype(np.float32)[None, :]
    prod64 = d.astype(np.float64)[:, None] * q.astype(np.float64)[None, :]
    assert np.array_equal(prod32.astype(np.float64), prod64)


# ------------------------------------------------------------------------------------------
# W8A8 accumulation
# ------------------------------------------------------------------------------------------

def _brute_acc(x, W):
    M, K = x.shape
    N = W.shape[1]
    return [[sum(int(x[m, k]) * int(W[k, n]) for k in range(K)) for n in range(N)] for m in range(M)]


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (2, 3, 5), (4, 64, 16), (3, 32, 7)])
def test_w8a8_acc_brute_force(M, K, N):
    vals = np.array([-128, -127, -1, 0, 1, 127], dtype=np.int8)
    rng = np.random.default_rng(M * 1000 + K * 10 + N)
    for _ in range(4):
        x = vals[rng.integers(0, len(vals), size=(M, K))]
        W = vals[rng.integers(0, len(vals), size=(K, N))]
        assert oracle.w8a8_acc(x, W).tolist() == _brute_acc(x, W)


def test_w8a8_acc_exhaustive_pairs():
    # Every (x, w) int8 pair once: K = 1 products against Python integers.
    xs = np.arange(-128, 128, dtype=np.int8).reshape(256, 1)
    W = np.arange(-128, 128, dtype=np.int8).reshape(1, 256)
    acc = oracle.w8a8_acc(xs, W)
    ref = np.arange(-128, 128, dtype=np.int64)[:, None] * np.arange(-128, 128, dtype=np.int64)[None, :]
    np.testing.assert_array_equal(acc, ref)


@pytest.mark.parametrize("K", [32, 4096, 12288])
def test_w8a8_closed_forms_extremes(K):
    M, N = 2, 16
    ones_x = np.ones((M, K), np.int8)
    ones_w = np.ones((K, N), np.int8)
    assert (oracle.w8a8_acc(ones_x, ones_w) == K).all()
    x = np.full((M, K), 127, np.int8)
    w = np.full((K, N), -127, np.int8)
    assert (oracle.w8a8_acc(x, w) == -16129 * K).all()
    x = np.full((M, K), -128, np.int8)
    w = np.full((K, N), -128, np.int8)
    assert (oracle.w8a8_acc(x, w) == 16384 * K).all()


def test_w8a8_closed_form_identity_and_one_hot():
    K = N = 64
    x = synth.uniform_int8(3, "pin.x", (5, K))
    for c in (1, -1, 7, -128):
        W = (np.eye(K, dtype=np.int64) * c).astype(np.int8)
        np.testing.assert_array_equal(oracle.w8a8_acc(x, W), x.astype(np.int64) * c)
    W = synth.uniform_int8(4, "pin.W", (K, 48))
    for k0 in (0, 17, K - 1):
        xh = np.zeros((1, K), np.int8)
        xh[0, k0] = 1
        np.testing.assert_array_equal(oracle.w8a8_acc(xh, W)[0], W[k0].astype(np.int64))


def test_w8a8_acc_transposed_operand_is_caught():
    # A transposed W (or x) changes the sums for a non-symmetric case: the brute force sees it.
    x = np.array([[1, 2]], np.int8)
    W = np.array([[1, 2], [3, 4]], np.int8)
    assert oracle.w8a8_acc(x, W).tolist() == [[7, 10]]           # x @ W, not x @ W.T ([[5, 11]])


def test_w8a8_split_partition_invariance():
    M, K, N = 4, 512, 24
    x = synth.uniform_int8(5, "pin.x", (M, K))
    W = synth.uniform_int8(5, "pin.W", (K, N))
    ref = oracle.w8a8_acc(x, W)
    rng = np.random.default_rng(7)
    for parts in (1, 2, 3, 5, 16):
        for _ in range(3):
            cuts = np.sort(rng.choice(np.arange(1, K // 32), size=parts - 1, replace=False)) * 32
            bounds = [0, *cuts.tolist(), K]
            np.testing.assert_array_equal(oracle.w8a8_acc_split(x, W, bounds), ref)
    with pytest.raises(ValueError):
        oracle.w8a8_acc_split(x, W, [0, 64, 32, K])     # not ascending
    with pytest.raises(ValueError):
        oracle.w8a8_acc_split(x, W, [0, 64, K - 32])    # does not reach K


def test_w8a8_acc_overflow_is_reported():
    # 128 * 128 * 2^17 = 2^31 leaves int32: the oracle must refuse rather than wrap.
    K = 1 << 17
    x = np.full((1, K), -128, np.int8)
    W = np.full((K, 1), -128, np.int8)
    with pytest.raises(OverflowError):
        oracle.w8a8_acc(x, W)


# ------------------------------------------------------------------------------------------
# W8A8 epilogue
# ------------------------------------------------------------------------------------------

def test_w8a8_epilogue_golden():
    for acc, xs_hex, ws_hex, out_hex in _read_golden("w8a8_epilogue.txt"):
        xs = np.array([int(xs_hex, 16)], np.uint32).view(np.float32)
        ws = np.array([int(ws_hex, 16)], np.uint32).view(np.float32)
        out = oracle.w8a8_epilogue(np.array([[int(acc)]], np.int32), xs, ws)
        assert int(out[0, 0]) == int(out_hex, 16), (acc, xs_hex, ws_hex)


def test_w8a8_epilogue_matches_numpy_float32_and_torch_bf16():
    M, N = 16, 512
    rng = np.random.default_rng(11)
    acc = rng.integers(-200_000_000, 200_000_000, size=(M, N), dtype=np.int64).astype(np.int32)
    acc[0, :8] = [16777217, 16777219, -16777217, 2**31 - 1, -(2**31), 0, 1, -1]
    xs = synth.log_uniform_f32(1, "pin.xs", (M,), 1e-4, 1e-1)
    ws = synth.log_uniform_f32(1, "pin.ws", (N,), 1e-4, 1e-1)
    f = acc.astype(np.float32)                     # numpy: int32 -> float32 rounds to nearest even
    f = f * xs[:, None]                            # float32 * float32 -> float32 (IEEE RNE)
    f = f * ws[None, :]
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.w8a8_epilogue(acc, xs, ws), ref)


def test_w8a8_epilogue_order_is_x_scale_first():
    # Find inputs where (a*xs)*ws and a*(xs*ws) round to different bfloat16 values; the oracle must
    # take the first order.  numpy float32 arithmetic and torch's bf16 cast are the witnesses.
    rng = np.random.default_rng(5)
    checked = 0
    for _ in range(16):
        a = rng.integers(-(2**27), 2**27, size=1 << 21).astype(np.int32)
        xs = rng.uniform(1e-3, 2e-2, size=a.size).astype(np.float32)
        ws = rng.uniform(1e-3, 2e-2, size=a.size).astype(np.float32)
        first = (a.astype(np.float32) * xs) * ws
        other = a.astype(np.float32) * (xs * ws)
        b1 = torch.from_numpy(first).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        b2 = torch.from_numpy(other).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        idx = np.nonzero(b1 != b2)[0][:8]
        for i in idx:
            out = oracle.w8a8_epilogue(np.array([[a[i]]], np.int32), xs[i:i + 1], ws[i:i + 1])
            assert int(out[0, 0]) == int(b1[i])
            checked += 1
        if checked >= 10:
            break
    assert checked >= 10


def test_w8a8_gemm_small_against_python():
    M, K, N = 3, 64, 8
    x, xs, W, ws = synth.w8a8_inputs(M, K, N, seed=9)
    out, acc = oracle.w8a8_gemm(x, xs, W, ws, return_acc=True)
    assert acc.tolist() == _brute_acc(x, W)
    for m in range(M):
        for n in range(N):
            f = np.float32(np.float32(np.float32(acc[m, n]) * xs[m]) * ws[n])
            ref = torch.tensor([float(f)], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
            assert int(out[m, n]) == ref


# ------------------------------------------------------------------------------------------
# Q8_0
# ------------------------------------------------------------------------------------------

def _frac_from_bf16(b):
    return Fraction(float(torch.tensor([int(b)], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float().item()))


def test_q8_0_brute_force_rational():
    T, K, N = 2, 64, 3
    x, q, d = synth.q8_0_inputs(T, K, N, seed=2)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    db = d.view(np.uint16)
    y = oracle.q8_0_gemv(xb, q, db)
    xf = x.float().numpy()
    for t in range(T):
        for n in range(N):
            exact = sum(Fraction(float(xf[t, k])) * Fraction(float(d[n, k // 32])) * int(q[n, k]) for k in range(K))
            assert abs(float(exact) - y[t, n]) <= 1e-12 * max(1.0, abs(float(exact)))


def test_q8_0_closed_form_ones():
    T, K, N = 3, 320, 5
    x = torch.ones((T, K), dtype=torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    q = np.ones((N, K), np.int8)
    d = synth.uniform_f16(4, "pin.d", (N, K // 32), 1e-3, 1e-2)
    y = oracle.q8_0_gemv(xb, q, d.view(np.uint16))
    expect = 32.0 * d.astype(np.float64).sum(axis=1)       # exact: few terms, each exact in fp64
    for t in range(T):
        np.testing.assert_array_equal(y[t], expect)


def test_q8_0_one_hot_and_block_orientation():
    # One-hot activation at k0 picks d[n, k0 // 32] * q[n, k0]: pins the block index along K
    # (a block index along N, or a transposed q, gives another value).
    T, K, N = 1, 128, 6
    q = synth.uniform_int8(6, "pin.q", (N, K))
    d = synth.uniform_f16(6, "pin.d", (N, K // 32), 1e-3, 1e-2)
    for k0 in (0, 31, 32, 100):
        x = torch.zeros((T, K), dtype=torch.bfloat16)
        x[0, k0] = 1.0
        y = oracle.q8_0_gemv(x.view(torch.int16).numpy().view(np.uint16), q, d.view(np.uint16))
        np.testing.assert_array_equal(y[0], d[:, k0 // 32].astype(np.float64) * q[:, k0].astype(np.float64))


def test_q8_0_norms():
    T, K, N = 2, 96, 4
    x, q, d = synth.q8_0_inputs(T, K, N, seed=8)
    xn, wn = oracle.q8_0_norms(x.view(torch.int16).numpy().view(np.uint16), q, d.view(np.uint16))
    xf = x.double().numpy()
    w = d.astype(np.float64).repeat(32, axis=1) * q.astype(np.float64)
    np.testing.assert_allclose(xn, np.sqrt((xf * xf).sum(axis=1)), rtol=1e-14)
    np.testing.assert_allclose(wn, np.sqrt((w * w).sum(axis=1)), rtol=1e-14)


def test_q8_0_bound_is_the_cauchy_schwarz_scale():
    # The per-output bound is rel * ||x_t|| * ||w_n||: by Cauchy-Schwarz |y[t,n]| never exceeds
    # ||x_t|| ||w_n||, with equality when x_t is w_n.  Unit scales and small quants make w exact in
    # bf16, so rows of x can be set to rows of w: the equality pins the (t, n) orientation.
    T, K, N = 2, 64, 3
    q = synth.uniform_int8(12, "pin.cs.q", (N, K), lo=-20, hi=20)
    d = np.full((N, K // 32), 1.0, np.float16)
    x = torch.tensor(np.stack([q[2], q[0]]).astype(np.float32)).to(torch.bfloat16)
    xb = x.view(torch.int16).numpy().view(np.uint16)
    b = oracle.q8_0_bound(xb, q, d.view(np.uint16), 2e-3)
    y = oracle.q8_0_gemv(xb, q, d.view(np.uint16))
    assert b.shape == (T, N)
    assert (np.abs(y) <= b / 2e-3 * (1 + 1e-12)).all()
    for t, n in ((0, 2), (1, 0)):
        assert y[t, n] == pytest.approx(b[t, n] / 2e-3, rel=1e-12)
        assert y[t, n] == float((q[n].astype(np.int64) ** 2).sum())


def test_q8_0_split_layout_from_ggml_blocks():
    # The split layout is the same bytes as ggml's 34-byte blocks, reordered.
    K, N = 64, 3
    rng = np.random.default_rng(3)
    blocks = rng.integers(0, 256, size=(N, K // 32, 34), dtype=np.uint8)
    q, d = oracle.q8_0_split_from_blocks(blocks, K, N)
    for n in range(N):
        for b in range(K // 32):
            assert int(d[n, b]) == int(blocks[n, b, 0]) | (int(blocks[n, b, 1]) << 8)
            assert q[n, 32 * b:32 * b + 32].view(np.uint8).tolist() == blocks[n, b, 2:].tolist()


# ------------------------------------------------------------------------------------------
# Packed weight layout
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("K,N", [(32, 64), (64, 200), (96, 16)])
def test_pack_is_offset_binary_bijection(K, N):
    W = synth.uniform_int8(1, "pin.W", (K, N), lo=-128, hi=127)
    p = oracle.w8a8_pack(W)
    Np = -(-N // 64) * 64
    assert p.size == Np * K
    # Each padded (k, n) cell appears once: place distinct cell ids through a one-hot sweep of
    # rows, and check the multiset of stored values against W's.
    vals = (p ^ 0x80).view(np.int8)
    pad = Np * K - N * K
    expect = np.sort(np.concatenate([W.ravel(), np.zeros(pad, np.int8)]))
    np.testing.assert_array_equal(np.sort(vals), expect)


def test_pack_places_each_weight_once():
    K, N = 64, 128
    positions = {}
    for k in range(0, K, 7):
        for n in range(0, N, 5):
            W = np.zeros((K, N), np.int8)
            W[k, n] = 1
            p = oracle.w8a8_pack(W)
            hit = np.nonzero(p != 0x80)[0]
            assert hit.size == 1 and p[hit[0]] == 0x81
            assert hit[0] not in positions
            positions[hit[0]] = (k, n)
            # the stored cell lies in the 64-row tile of n and the 32-wide k block of k
            t, kb = hit[0] // (K // 32 * 2048), (hit[0] // 2048) % (K // 32)
            assert t == n // 64 and kb == k // 32


def test_pack_positions_golden():
    # Byte positions worked out by hand from the documented layout (tests/golden): a weight moved
    # to another byte of its slab, e.g. with the row and k halves of a chunk swapped, is caught.
    for K, N, off, k, n in _read_golden("w8a8_pack_positions.txt"):
        K, N, off = int(K), int(N), int(off)
        if k == "pad":
            p = oracle.w8a8_pack(np.full((K, N), 5, np.int8))
            assert p[off] == 0x80
            continue
        W = np.zeros((K, N), np.int8)
        W[int(k), int(n)] = -3
        p = oracle.w8a8_pack(W)
        assert np.nonzero(p != 0x80)[0].tolist() == [off]
        assert p[off] == (0xFD ^ 0x80)                     # -3 in offset binary


# --------------------------------------------------------------------------------------------
# Quantisation rows (activation quantisation in front of W8A8; Q8_0 from BF16 at load)
# --------------------------------------------------------------------------------------------

def _bf16_bits(values):
    """float values exactly representable in bf16 -> their bf16 bit patterns (via torch)."""
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.tensor(np.asarray(values, dtype=np.float32)))   # exact
    return t.view(torch.int16).numpy().view(np.uint16)


def test_f16_from_f32_matches_numpy():
    # Edges: largest half, the first value that rounds to infinity, subnormals, halfway cases
    # (low 13 bits exactly 0x1000, both parities), and random values over every exponent.
    edge = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 2.0**-14, 2.0**-24, 2.0**-25, 3 * 2.0**-25,
            2.0**-25 * 1.0001, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, 1.0 + 2.0**-11 + 2.0**-20, 1e-3, 1e-2, 0.1]
    rng = np.random.default_rng(3)
    rand = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 17, 20000))).astype(np.float32)
    vals = np.concatenate([np.array(edge, np.float32), rand])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(oracle.f16_from_f32(vals), ref)


def test_q8_0_quantize_exact_multiples_and_ties():
    # d = (127 / 8) / 127 = 1/8 exactly (fp16 0x3000).  Row 0: x = k/8 gives q = k.  Row 1:
    # x = (n + 1/2)/8 is a tie, rounded away from zero (ggml's roundf), not to even.  Row 2: a zero
    # block gives d = 0, q = 0.  Row 3: the amax element is negative and maps to -127.
    K = 32
    k = np.array(list(range(-15, 16)) + [127], dtype=np.float64)
    ties = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, -126.5] + [0.0] * 23 + [127.0])
    rows = np.stack([k / 8, ties / 8, np.zeros(K), np.array([-127.0] + [3.0] * 31) / 8])
    q, d = oracle.q8_0_quantize(_bf16_bits(rows))
    assert d.tolist() == [[0x3000], [0x3000], [0], [0x3000]]
    np.testing.assert_array_equal(q[0], k.astype(np.int8))
    np.testing.assert_array_equal(q[1, :8], [1, 2, 3, -1, -2, -3, 127, -127])
    assert q[1, -1] == 127 and (q[2] == 0).all()
    assert q[3, 0] == -127 and (q[3, 1:] == 3).all()         # (3/8) / (1/8) = 3


def test_q8_0_quantize_invariants_random():
    # Random bf16 weights: |x - q d| <= d / 2 (rounding to the nearest integer, d the float32
    # amax / 127), |q| <= 127 with the amax element at +-127, and the stored scale is numpy's
    # float16 of that float32 quotient.
    rng = np.random.default_rng(11)
    N, K = 24, 256
    w = torch.tensor(rng.standard_normal((N, K)).astype(np.float32) * 0.02).to(torch.bfloat16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    wf = w.float().numpy().reshape(N, K // 32, 32)
    q, d = oracle.q8_0_quantize(wb)
    amax = np.abs(wf).max(axis=2).astype(np.float32)
    d32 = amax / np.float32(127)
    np.testing.assert_array_equal(d, d32.astype(np.float16).view(np.uint16))
    qb = q.reshape(N, K // 32, 32).astype(np.float64)
    err = np.abs(wf.astype(np.float64) - qb * d32[..., None].astype(np.float64))
    assert (err <= d32[..., None] * (0.5 + 2.0**-16)).all()      # x / d rounds once in fp32 (|x / d| <= 127)
    assert np.abs(q).max() <= 127
    at = np.argmax(np.abs(wf), axis=2)
    np.testing.assert_array_equal(np.abs(np.take_along_axis(qb, at[..., None], axis=2)[..., 0]), 127)


def test_w8a8_quantize_rows_closed_forms_and_invariants():
    # Row-wise: same closed forms as a Q8_0 block spanning the whole row, plus random rows.
    K = 64
    r0 = np.array(list(range(-31, 32)) + [127], dtype=np.float64) / 4           # scale 1/4: q = 4x
    r1 = np.zeros(K)
    r2 = np.array([2.5, -2.5, 0.5] + [0.0] * 60 + [-127.0]) / 4                 # ties away from zero
    xq, xs = oracle.w8a8_quantize_rows(_bf16_bits(np.stack([r0, r1, r2])))
    assert xs.tolist() == [0.25, 0.0, 0.25]
    np.testing.assert_array_equal(xq[0], (r0 * 4).astype(np.int8))
    assert (xq[1] == 0).all()
    assert xq[2, :3].tolist() == [3, -3, 1] and xq[2, -1] == -127
    rng = np.random.default_rng(12)
    x = torch.tensor(rng.standard_normal((16, 4096)).astype(np.float32)).to(torch.bfloat16)
    xq, xs = oracle.w8a8_quantize_rows(x.view(torch.int16).numpy().view(np.uint16))
    xf = x.float().numpy().astype(np.float64)
    np.testing.assert_array_equal(xs, (np.abs(x.float().numpy()).max(axis=1) / np.float32(127)).astype(np.float32))
    assert (np.abs(xf - xq * xs[:, None].astype(np.float64)) <= xs[:, None] * (0.5 + 2.0**-16)).all()
    assert (np.abs(xq).max(axis=1) == 127).all()


def test_q8_0_blocks_and_split_layout_are_inverse():
    rng = np.random.default_rng(13)
    N, K = 5, 96
    q = rng.integers(-128, 128, (N, K)).astype(np.int8)
    d = rng.integers(0, 1 << 16, (N, K // 32)).astype(np.uint16)
    blocks = oracle.q8_0_blocks_from_split(q, d)
    assert blocks.shape == (N, K // 32, 34)
    # byte-level check of one block from the definition: little-endian scale, then the 32 quants
    assert blocks[2, 1, 0] == d[2, 1] & 0xFF and blocks[2, 1, 1] == d[2, 1] >> 8
    np.testing.assert_array_equal(blocks[2, 1, 2:].view(np.int8), q[2, 32:64])
    q2, d2 = oracle.q8_0_split_from_blocks(blocks, K, N)
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(d2, d)


# --------------------------------------------------------------------------------------------
# Q8_0 read with an RMS-norm prologue (rs * (x * g) @ w, rs the inverse RMS of x's row)
# --------------------------------------------------------------------------------------------

def _xg_inputs(T, K, N, seed):
    x, q, d = synth.q8_0_inputs(T, K, N, seed=seed)
    g = torch.tensor(synth.uniform_f32(seed, "pin.g", (K,), 0.5, 1.5)).to(torch.bfloat16)
    return (x.view(torch.int16).numpy().view(np.uint16), g.view(torch.int16).numpy().view(np.uint16), q,
            d.view(np.uint16), x, g, d)


def test_q8_0_rms_brute_force_with_python_floats():
    # Independent restatement: Python floats from torch's bf16 decoding, math.fsum for the sums.
    import math
    T, K, N = 2, 64, 3
    xb, gb, q, db, x, g, d = _xg_inputs(T, K, N, seed=3)
    eps = 1e-5
    y, rs = oracle.q8_0_rms_gemv(xb, gb, eps, q, db)
    xf, gf = x.double().numpy(), g.double().numpy()
    for t in range(T):
        r = 1.0 / math.sqrt(math.fsum(float(v) * float(v) for v in xf[t]) / K + eps)
        assert abs(r - rs[t]) <= 1e-14 * r
        for n in range(N):
            s = math.fsum(float(xf[t, k]) * float(gf[k]) * float(d[n, k // 32]) * int(q[n, k]) for k in range(K))
            assert abs(r * s - y[t, n]) <= 1e-12 * max(1.0, abs(r * s))


def test_q8_0_rms_gamma_one_reduces_to_the_plain_read():
    T, K, N = 3, 320, 7
    xb, _, q, db, *_ = _xg_inputs(T, K, N, seed=4)
    ones = _bf16_bits(np.ones(K))
    y, rs = oracle.q8_0_rms_gemv(xb, ones, 1e-6, q, db)
    np.testing.assert_array_equal(y, rs[:, None] * oracle.q8_0_gemv(xb, q, db))


def test_q8_0_rms_is_scale_invariant_without_eps():
    # RMS normalisation: doubling x (exact in bf16 and fp64) leaves every output bit unchanged when
    # eps = 0; a missing rs, rs from x * g, or a wrong power would not.
    T, K, N = 2, 128, 5
    xb, gb, q, db, x, g, d = _xg_inputs(T, K, N, seed=5)
    x2 = (x.float() * 2).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    y1, rs1 = oracle.q8_0_rms_gemv(xb, gb, 0.0, q, db)
    y2, rs2 = oracle.q8_0_rms_gemv(x2, gb, 0.0, q, db)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(rs2, rs1 / 2)


def test_q8_0_rms_closed_forms():
    # Constant rows: x = c, g = 1, q = 1: rs = 1 / sqrt(c^2 + eps), y = rs * c * 32 * sum_b d[n, b].
    T, K, N = 2, 96, 4
    d = synth.uniform_f16(9, "pin.d", (N, K // 32), 1e-3, 1e-2)
    q = np.ones((N, K), np.int8)
    eps = 0.25
    for c in (0.5, -3.0):
        xb = _bf16_bits(np.full((T, K), c))
        y, rs = oracle.q8_0_rms_gemv(xb, _bf16_bits(np.ones(K)), eps, q, d.view(np.uint16))
        r = 1.0 / np.sqrt(c * c + eps)
        np.testing.assert_allclose(rs, r, rtol=1e-15)
        np.testing.assert_allclose(y, np.broadcast_to(r * c * 32.0 * d.astype(np.float64).sum(axis=1), (T, N)),
                                   rtol=1e-14)
    # One-hot x at k0 with weight g[k0]: rs = 1 / sqrt(x^2 / K + eps), y = rs * x * g[k0] * d q.
    K, N = 64, 3
    q = synth.uniform_int8(10, "pin.q", (N, K))
    d = synth.uniform_f16(10, "pin.d", (N, K // 32), 1e-3, 1e-2)
    g = np.array([0.5 + k / 64 for k in range(K)])
    for k0 in (0, 33, 63):
        xv = np.zeros((1, K))
        xv[0, k0] = 4.0
        y, rs = oracle.q8_0_rms_gemv(_bf16_bits(xv), _bf16_bits(g), 1e-3, q, d.view(np.uint16))
        r = 1.0 / np.sqrt(16.0 / K + 1e-3)
        np.testing.assert_allclose(rs[0], r, rtol=1e-15)
        np.testing.assert_allclose(y[0], r * 4.0 * g[k0] * d[:, k0 // 32].astype(np.float64) * q[:, k0], rtol=1e-14)


def test_q8_0_rms_bound_scales_with_rs_and_the_norms():
    T, K, N = 2, 64, 3
    xb, gb, q, db, x, g, d = _xg_inputs(T, K, N, seed=11)
    b = oracle.q8_0_rms_bound(xb, gb, 1e-6, q, db)
    _, rs = oracle.q8_0_rms_gemv(xb, gb, 1e-6, q, db)
    xg = (x.double() * g.double()).numpy()
    w = d.astype(np.float64).repeat(32, axis=1) * q.astype(np.float64)
    expect = 8e-3 * rs[:, None] * np.sqrt((xg * xg).sum(axis=1))[:, None] * np.sqrt((w * w).sum(axis=1))[None, :]
    np.testing.assert_allclose(b, expect, rtol=1e-13)

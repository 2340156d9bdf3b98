"""The seeded input generators on the CPU: the counter-based SplitMix64 stream pinned to the
generator's published check values, random access into a stream, and each distribution the
workloads name (range, ends, moments, exact representability in its storage type)."""
import numpy as np
import pytest
import torch

import synth


def test_mix64_reproduces_the_splitmix64_check_values():
    # SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) started from state 1234567: the state
    # advances by the golden-ratio increment and each output is the mix of the new state.  These
    # five outputs are the check values commonly quoted for that state.
    expect = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
              16408922859458223821]
    with np.errstate(over="ignore"):
        idx = np.arange(1, 6, dtype=np.uint64)
        got = synth._mix64(np.uint64(1234567) + idx * synth.GAMMA)
    assert [int(v) for v in got] == expect


def test_streams_are_random_access_and_keyed_by_seed_and_tag():
    whole = synth.raw_u64(7, "x", 1000)
    assert np.array_equal(synth.raw_u64(7, "x", 300, start=500), whole[500:800])
    assert np.array_equal(synth.raw_u64(7, "x", 1000), whole)                 # deterministic
    assert not np.array_equal(synth.raw_u64(8, "x", 1000), whole)
    assert not np.array_equal(synth.raw_u64(7, "y", 1000), whole)
    # 1000 draws of 64 bits: every bit position is set in roughly half of them
    bits = np.unpackbits(whole.view(np.uint8)).reshape(1000, 64).mean(axis=0)
    assert bits.min() > 0.4 and bits.max() < 0.6


def test_uniform_int8_covers_its_inclusive_range_evenly():
    v = synth.uniform_int8(3, "u", (200000,))
    assert v.dtype == np.int8 and v.min() == -127 and v.max() == 127
    counts = np.bincount(v.astype(np.int64) + 127, minlength=255)
    assert counts.min() > 0.8 * 200000 / 255 and counts.max() < 1.2 * 200000 / 255
    w = synth.uniform_int8(3, "u", (10000,), lo=-2, hi=3)
    assert set(np.unique(w).tolist()) == {-2, -1, 0, 1, 2, 3}


def test_clipped_gaussian_has_its_sigma_and_clip():
    v = synth.clipped_gaussian_int8(4, "g", (200000,), sigma=40.0, clip=127)
    assert v.dtype == np.int8 and v.min() >= -127 and v.max() <= 127
    assert abs(v.astype(np.float64).mean()) < 0.5
    assert 39.0 < v.astype(np.float64).std() < 41.0        # ~1.5 % of the mass is clipped at 3.2 sigma
    assert (np.abs(v) == 127).any()


def test_uniform_and_log_uniform_floats():
    u = synth.uniform_f32(5, "s", (100000,), 1e-3, 2e-2)
    assert u.dtype == np.float32 and u.min() >= np.float32(1e-3) and u.max() <= np.float32(2e-2)
    assert abs(u.astype(np.float64).mean() - 0.5 * (1e-3 + 2e-2)) < 1e-4
    lg = synth.log_uniform_f32(5, "l", (100000,), 1e-4, 1e-1)
    assert lg.min() >= np.float32(1e-4) * (1 - 1e-6) and lg.max() <= np.float32(1e-1) * (1 + 1e-6)
    # uniform in log: the mean of ln x is the midpoint of the logs
    assert abs(np.log(lg.astype(np.float64)).mean() - 0.5 * (np.log(1e-4) + np.log(1e-1))) < 0.02


def test_half_and_bfloat16_draws_are_exact_in_their_types():
    h = synth.uniform_f16(6, "d", (5000,), 1e-3, 1e-2)
    assert np.array_equal(h.astype(np.float16).astype(h.dtype), h)
    assert h.min() >= np.float16(1e-3) and h.max() <= np.float16(1e-2)
    b = synth.normal_bf16(6, "x", (4, 4096))
    assert b.dtype == torch.bfloat16
    f = b.float()
    assert torch.equal(f.to(torch.bfloat16), b)
    assert abs(float(f.mean())) < 0.05 and 0.95 < float(f.std()) < 1.05


@pytest.mark.parametrize("dist", ["uniform", "mlp"])
def test_w8a8_inputs_shapes_and_types(dist):
    x, xs, W, ws = synth.w8a8_inputs(16, 512, 256, seed=9, dist=dist)
    assert x.shape == (16, 512) and x.dtype == np.int8 and x.flags["C_CONTIGUOUS"]
    assert xs.shape == (16,) and xs.dtype == np.float32 and (xs > 0).all()
    assert W.shape == (512, 256) and W.dtype == np.int8 and W.flags["C_CONTIGUOUS"]
    assert ws.shape == (256,) and ws.dtype == np.float32 and (ws > 0).all()
    again = synth.w8a8_inputs(16, 512, 256, seed=9, dist=dist)
    assert all(np.array_equal(a, b) for a, b in zip((x, xs, W, ws), again))


def test_q8_0_inputs_shapes_and_types():
    x, q, d = synth.q8_0_inputs(6, 320, 4096, seed=2)
    assert x.shape == (6, 320) and x.dtype == torch.bfloat16
    assert q.shape == (4096, 320) and q.dtype == np.int8
    assert d.shape == (4096, 10) and d.dtype == np.float16 and (d > 0).all()

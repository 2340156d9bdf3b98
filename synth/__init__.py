"""Seeded synthetic inputs for the small-M quantized weight GEMM workloads.

This module only draws numbers. It holds none of the arithmetic of the
operators: the CUDA path and the oracle both take their inputs from here and
compute everything else on their own.

Every stream is a counter-based SplitMix64 sequence (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014): output i of
stream (seed, tag) is mix64(key + (i + 1) * GAMMA) with GAMMA the 64-bit
golden-ratio increment and key = mix64(mix64(seed) ^ tag_hash).  The whole
array is produced with vectorised numpy uint64 arithmetic, so any element can
be regenerated without producing the ones before it and the result is the same
on x86-64 and AArch64 hosts.

The distributions are the ones the workloads name:
  * int8 uniform on an inclusive range            (uniform_int8)
  * int8 from a clipped, rounded Gaussian         (clipped_gaussian_int8)
  * float32 uniform on [lo, hi]                   (uniform_f32)
  * float32 log-uniform on [lo, hi]               (log_uniform_f32)
  * float16 values drawn uniform then rounded     (uniform_f16)
  * bfloat16 values drawn N(0, 1) then rounded    (normal_bf16)
"""
from __future__ import annotations

import hashlib

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _key(seed: int, tag: str) -> np.uint64:
    h = int.from_bytes(hashlib.sha256(tag.encode()).digest()[:8], "little")
    with np.errstate(over="ignore"):
        s = _mix64(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))
        k = _mix64(s ^ np.uint64(h))
    return k[0]


def raw_u64(seed: int, tag: str, count: int, start: int = 0) -> np.ndarray:
    """Elements [start, start + count) of the (seed, tag) stream as uint64."""
    key = _key(seed, tag)
    out = np.empty(count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for lo in range(0, count, _CHUNK):
            hi = min(count, lo + _CHUNK)
            idx = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            out[lo:hi] = _mix64(key + idx * GAMMA)
    return out


def _unit_open(u: np.ndarray) -> np.ndarray:
    """uint64 -> float64 in (0, 1]: top 53 bits, shifted off zero."""
    return ((u >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def _unit24(u: np.ndarray) -> np.ndarray:
    """uint64 -> float64 in [0, 1) with 24 bits of resolution."""
    return (u >> np.uint64(40)).astype(np.float64) * (1.0 / 16777216.0)


def uniform_int8(seed: int, tag: str, shape, lo: int = -127, hi: int = 127) -> np.ndarray:
    """int8 uniform on the inclusive range [lo, hi] (Lemire's multiply-shift)."""
    n = int(np.prod(shape))
    span = np.uint64(hi - lo + 1)
    out = np.empty(n, dtype=np.int8)
    with np.errstate(over="ignore"):
        for a in range(0, n, _CHUNK):
            b = min(n, a + _CHUNK)
            u = raw_u64(seed, tag, b - a, start=a) >> np.uint64(32)
            out[a:b] = ((u * span) >> np.uint64(32)).astype(np.int64) + lo
    return out.reshape(shape)


def _normal(seed: int, tag: str, n: int, start: int = 0) -> np.ndarray:
    """Standard normal float64 samples, one Box-Muller cosine branch per pair of draws."""
    u = raw_u64(seed, tag, 2 * n, start=2 * start)
    u1 = _unit_open(u[0::2])
    u2 = _unit_open(u[1::2])
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def clipped_gaussian_int8(seed: int, tag: str, shape, sigma: float = 40.0, clip: int = 127) -> np.ndarray:
    """int8 from sigma * N(0,1), rounded half to even, clipped to [-clip, clip]."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.int8)
    for a in range(0, n, _CHUNK):
        b = min(n, a + _CHUNK)
        z = np.rint(sigma * _normal(seed, tag, b - a, start=a))
        out[a:b] = np.clip(z, -clip, clip).astype(np.int8)
    return out.reshape(shape)


def uniform_f32(seed: int, tag: str, shape, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape))
    u = _unit24(raw_u64(seed, tag, n))
    return (lo + (hi - lo) * u).astype(np.float32).reshape(shape)


def log_uniform_f32(seed: int, tag: str, shape, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape))
    u = _unit24(raw_u64(seed, tag, n))
    return np.exp(np.log(lo) + u * (np.log(hi) - np.log(lo))).astype(np.float32).reshape(shape)


def uniform_f16(seed: int, tag: str, shape, lo: float, hi: float) -> np.ndarray:
    """float16 values: float32 uniform on [lo, hi], then numpy's round-to-nearest-even cast."""
    return uniform_f32(seed, tag, shape, lo, hi).astype(np.float16)


def normal_bf16(seed: int, tag: str, shape):
    """bfloat16 N(0,1) values as a CPU torch tensor (torch's round-to-nearest-even cast)."""
    import torch

    n = int(np.prod(shape))
    z = _normal(seed, tag, n).astype(np.float32).reshape(shape)
    return torch.from_numpy(z).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# Workload recipes.  Each returns plain arrays; nothing here computes a result.
# ---------------------------------------------------------------------------

def w8a8_inputs(M: int, K: int, N: int, seed: int = 0, dist: str = "uniform"):
    """Inputs of the W8A8 decode GEMM.

    dist="uniform": x_q, W int8 uniform [-127, 127]; x_scale, w_scale float32 uniform [1e-3, 2e-2].
    dist="mlp":     x_q, W int8 from a Gaussian with sigma 40 clipped to +-127;
                    x_scale, w_scale float32 log-uniform [1e-4, 1e-1].
    Returns (x_q [M,K] int8, x_scale [M] f32, W [K,N] int8, w_scale [N] f32).
    """
    if dist == "uniform":
        x_q = uniform_int8(seed, "w8a8.x_q", (M, K))
        W = uniform_int8(seed, "w8a8.W", (K, N))
        x_scale = uniform_f32(seed, "w8a8.x_scale", (M,), 1e-3, 2e-2)
        w_scale = uniform_f32(seed, "w8a8.w_scale", (N,), 1e-3, 2e-2)
    elif dist == "mlp":
        x_q = clipped_gaussian_int8(seed, "w8a8.x_q", (M, K))
        W = clipped_gaussian_int8(seed, "w8a8.W", (K, N))
        x_scale = log_uniform_f32(seed, "w8a8.x_scale", (M,), 1e-4, 1e-1)
        w_scale = log_uniform_f32(seed, "w8a8.w_scale", (N,), 1e-4, 1e-1)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x_q, x_scale, W, w_scale


def q8_0_inputs(T: int, K: int, N: int, seed: int = 0):
    """Inputs of the Q8_0 weight GEMV in the split layout.

    x bf16 [T,K] ~ N(0,1) (CPU torch tensor); q int8 [N,K] uniform [-127,127];
    d float16 [N, K/32] uniform [1e-3, 1e-2] rounded to fp16.
    """
    x = normal_bf16(seed, "q8_0.x", (T, K))
    q = uniform_int8(seed, "q8_0.q", (N, K))
    d = uniform_f16(seed, "q8_0.d", (N, K // 32), 1e-3, 1e-2)
    return x, q, d

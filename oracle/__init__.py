"""Oracle for the small-M quantized weight GEMMs (numpy front end of oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU-baseline leg may import this package; the library's compute
path never does, and this package never imports the library.

Every function takes and returns numpy arrays (bf16 / fp16 as uint16 bit
patterns) and forwards to the plain C definitions in oracle.c, which cite the
passages they follow.  Pins: tests/test_oracle_pins.py checks each function
against values fixed by the pages or by the mathematics (brute force with
Python integers, closed forms, invariants, and bit patterns of IEEE rounding).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        c_p = ctypes.c_void_p
        c_i = ctypes.c_int
        L.oracle_bf16_from_f32.argtypes = [ctypes.c_float]
        L.oracle_bf16_from_f32.restype = ctypes.c_uint16
        L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f64.restype = ctypes.c_double
        L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_f64.restype = ctypes.c_double
        L.oracle_w8a8_acc.argtypes = [c_p, c_p, c_i, c_i, c_i, c_p]
        L.oracle_w8a8_acc.restype = c_i
        L.oracle_w8a8_acc_split.argtypes = [c_p, c_p, c_i, c_i, c_i, c_p, c_i, c_p]
        L.oracle_w8a8_acc_split.restype = c_i
        L.oracle_w8a8_epilogue.argtypes = [c_p, c_p, c_p, c_i, c_i, c_p]
        L.oracle_w8a8_epilogue.restype = None
        L.oracle_w8a8_gemm.argtypes = [c_p, c_p, c_p, c_p, c_i, c_i, c_i, c_p, c_p]
        L.oracle_w8a8_gemm.restype = c_i
        L.oracle_q8_0_gemv.argtypes = [c_p, c_p, c_p, c_i, c_i, c_i, c_p]
        L.oracle_q8_0_gemv.restype = None
        L.oracle_q8_0_norms.argtypes = [c_p, c_p, c_p, c_i, c_i, c_i, c_p, c_p]
        L.oracle_q8_0_norms.restype = None
        L.oracle_q8_0_rms_gemv.argtypes = [c_p, c_p, ctypes.c_double, c_p, c_p, c_i, c_i, c_i, c_p, c_p]
        L.oracle_q8_0_rms_gemv.restype = None
        L.oracle_q8_0_rms_xg_norms.argtypes = [c_p, c_p, c_i, c_i, c_p]
        L.oracle_q8_0_rms_xg_norms.restype = None
        L.oracle_q8_0_split_from_blocks.argtypes = [c_p, c_i, c_i, c_p, c_p]
        L.oracle_q8_0_split_from_blocks.restype = None
        L.oracle_w8a8_packed_bytes.argtypes = [c_i, c_i]
        L.oracle_w8a8_packed_bytes.restype = ctypes.c_size_t
        L.oracle_w8a8_pack.argtypes = [c_p, c_i, c_i, c_p]
        L.oracle_w8a8_pack.restype = None
        L.oracle_f16_from_f32.argtypes = [ctypes.c_float]
        L.oracle_f16_from_f32.restype = ctypes.c_uint16
        L.oracle_q8_0_quantize.argtypes = [c_p, c_i, c_i, c_p, c_p]
        L.oracle_q8_0_quantize.restype = None
        L.oracle_w8a8_quantize_rows.argtypes = [c_p, c_i, c_i, c_p, c_p]
        L.oracle_w8a8_quantize_rows.restype = None
        L.oracle_q8_0_blocks_from_split.argtypes = [c_p, c_p, c_i, c_i, c_p]
        L.oracle_q8_0_blocks_from_split.restype = None
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --- scalars ------------------------------------------------------------------------------

def bf16_from_f32(values) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (uint16)."""
    v = np.asarray(values, dtype=np.float32).ravel()
    L = lib()
    out = np.array([L.oracle_bf16_from_f32(float(f)) for f in v], dtype=np.uint16)
    return out.reshape(np.shape(values))


def bf16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).ravel()
    L = lib()
    return np.array([L.oracle_bf16_to_f64(int(x)) for x in b], dtype=np.float64).reshape(np.shape(bits))


def f16_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).ravel()
    L = lib()
    return np.array([L.oracle_f16_to_f64(int(x)) for x in b], dtype=np.float64).reshape(np.shape(bits))


# --- W8A8 -----------------------------------------------------------------------------------

def w8a8_acc(x_q: np.ndarray, W: np.ndarray) -> np.ndarray:
    """int32 [M,N] = x_q[M,K] @ W[K,N] (int64 sums, checked to fit int32)."""
    x_q = _c(x_q, np.int8)
    W = _c(W, np.int8)
    M, K = x_q.shape
    K2, N = W.shape
    assert K == K2
    acc = np.zeros((M, N), dtype=np.int32)
    rc = lib().oracle_w8a8_acc(_ptr(x_q), _ptr(W), M, K, N, _ptr(acc))
    if rc != 0:
        raise OverflowError("accumulator leaves the int32 range")
    return acc


def w8a8_acc_split(x_q: np.ndarray, W: np.ndarray, bounds) -> np.ndarray:
    """int32 sums taken slice by slice (k-ascending), slices added in ascending order."""
    x_q = _c(x_q, np.int8)
    W = _c(W, np.int8)
    M, K = x_q.shape
    N = W.shape[1]
    b = np.ascontiguousarray(bounds, dtype=np.int32)
    acc = np.zeros((M, N), dtype=np.int32)
    rc = lib().oracle_w8a8_acc_split(_ptr(x_q), _ptr(W), M, K, N, _ptr(b), len(b) - 1, _ptr(acc))
    if rc != 0:
        raise ValueError("bounds do not cover [0, K) in ascending order")
    return acc


def w8a8_epilogue(acc: np.ndarray, x_scale: np.ndarray, w_scale: np.ndarray) -> np.ndarray:
    """bf16 bits [M,N] = bf16_rne((float(acc) * x_scale[m]) * w_scale[n])."""
    acc = _c(acc, np.int32)
    xs = _c(x_scale, np.float32)
    ws = _c(w_scale, np.float32)
    M, N = acc.shape
    out = np.zeros((M, N), dtype=np.uint16)
    lib().oracle_w8a8_epilogue(_ptr(acc), _ptr(xs), _ptr(ws), M, N, _ptr(out))
    return out


def w8a8_gemm(x_q, x_scale, W, w_scale, return_acc: bool = False):
    """The whole W8A8 operator: returns bf16 bits [M,N] (and the int32 accumulators)."""
    x_q = _c(x_q, np.int8)
    W = _c(W, np.int8)
    xs = _c(x_scale, np.float32)
    ws = _c(w_scale, np.float32)
    M, K = x_q.shape
    N = W.shape[1]
    out = np.zeros((M, N), dtype=np.uint16)
    acc = np.zeros((M, N), dtype=np.int32)
    rc = lib().oracle_w8a8_gemm(_ptr(x_q), _ptr(xs), _ptr(W), _ptr(ws), M, K, N, _ptr(out), _ptr(acc))
    if rc != 0:
        raise OverflowError("accumulator leaves the int32 range")
    return (out, acc) if return_acc else out


def w8a8_packed_bytes(K: int, N: int) -> int:
    return int(lib().oracle_w8a8_packed_bytes(K, N))


def w8a8_pack(W: np.ndarray) -> np.ndarray:
    """The documented packed layout of w8a8_pack_weights, as uint8 bytes."""
    W = _c(W, np.int8)
    K, N = W.shape
    out = np.zeros(w8a8_packed_bytes(K, N), dtype=np.uint8)
    lib().oracle_w8a8_pack(_ptr(W), K, N, _ptr(out))
    return out


# --- Q8_0 -----------------------------------------------------------------------------------

def q8_0_gemv(x_bits: np.ndarray, q: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """float64 [T,N]: y[t,n] = sum_k x[t,k] * (d[n,k/32] * q[n,k])."""
    x_bits = _c(x_bits, np.uint16)
    q = _c(q, np.int8)
    d_bits = _c(d_bits, np.uint16)
    T, K = x_bits.shape
    N = q.shape[0]
    y = np.zeros((T, N), dtype=np.float64)
    lib().oracle_q8_0_gemv(_ptr(x_bits), _ptr(q), _ptr(d_bits), T, K, N, _ptr(y))
    return y


def q8_0_norms(x_bits: np.ndarray, q: np.ndarray, d_bits: np.ndarray):
    """(||x_t||_2 [T], ||w_n||_2 [N]) with w_n the dequantised weight row."""
    x_bits = _c(x_bits, np.uint16)
    q = _c(q, np.int8)
    d_bits = _c(d_bits, np.uint16)
    T, K = x_bits.shape
    N = q.shape[0]
    xn = np.zeros(T, dtype=np.float64)
    wn = np.zeros(N, dtype=np.float64)
    lib().oracle_q8_0_norms(_ptr(x_bits), _ptr(q), _ptr(d_bits), T, K, N, _ptr(xn), _ptr(wn))
    return xn, wn


def q8_0_bound(x_bits, q, d_bits, rel: float = 2e-3) -> np.ndarray:
    """Per-output error bound [T,N]: rel * ||x_t||_2 * ||w_n||_2."""
    xn, wn = q8_0_norms(x_bits, q, d_bits)
    return rel * np.outer(xn, wn)


def q8_0_rms_gemv(x_bits: np.ndarray, g_bits: np.ndarray, eps: float, q: np.ndarray, d_bits: np.ndarray):
    """(y float64 [T,N], rs float64 [T]): y[t,n] = rs[t] * sum_k (x[t,k] g[k]) (d[n,k/32] q[n,k]),
    rs[t] = 1 / sqrt(sum_k x[t,k]^2 / K + eps) (oracle.c: oracle_q8_0_rms_gemv)."""
    x_bits = _c(x_bits, np.uint16)
    g_bits = _c(g_bits, np.uint16)
    q = _c(q, np.int8)
    d_bits = _c(d_bits, np.uint16)
    T, K = x_bits.shape
    N = q.shape[0]
    assert g_bits.shape == (K,)
    y = np.zeros((T, N), dtype=np.float64)
    rs = np.zeros(T, dtype=np.float64)
    lib().oracle_q8_0_rms_gemv(_ptr(x_bits), _ptr(g_bits), float(eps), _ptr(q), _ptr(d_bits), T, K, N, _ptr(y),
                               _ptr(rs))
    return y, rs


def q8_0_rms_bound(x_bits, g_bits, eps, q, d_bits, rel: float = 8e-3) -> np.ndarray:
    """Per-output error bound of the RMS-norm read: rel * rs[t] * ||x_t * g||_2 * ||w_n||_2."""
    x_bits = _c(x_bits, np.uint16)
    g_bits = _c(g_bits, np.uint16)
    T, K = x_bits.shape
    xg = np.zeros(T, dtype=np.float64)
    lib().oracle_q8_0_rms_xg_norms(_ptr(x_bits), _ptr(g_bits), T, K, _ptr(xg))
    _, wn = q8_0_norms(x_bits, q, d_bits)
    _, rs = q8_0_rms_gemv(x_bits, g_bits, eps, q[:1], d_bits[:1])
    return rel * (rs * xg)[:, None] * wn[None, :]


def q8_0_split_from_blocks(blocks: np.ndarray, K: int, N: int):
    """ggml 34-byte Q8_0 blocks [N, K/32, 34] -> (q int8 [N,K], d fp16 bits [N,K/32])."""
    blocks = _c(blocks, np.uint8)
    q = np.zeros((N, K), dtype=np.int8)
    d = np.zeros((N, K // 32), dtype=np.uint16)
    lib().oracle_q8_0_split_from_blocks(_ptr(blocks), K, N, _ptr(q), _ptr(d))
    return q, d


def f16_from_f32(values) -> np.ndarray:
    """float32 values -> IEEE half bit patterns, round to nearest even (oracle.c)."""
    v = np.asarray(values, dtype=np.float32).ravel()
    L = lib()
    return np.array([L.oracle_f16_from_f32(float(f)) for f in v], dtype=np.uint16).reshape(np.shape(values))


def q8_0_quantize(w_bits: np.ndarray):
    """BF16 weights [N, K] (uint16 bits) -> (q [N, K] int8, d [N, K/32] fp16 bits), ggml's
    rounding as the Q8_0 page states it (oracle.c: oracle_q8_0_quantize)."""
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    q = np.empty((N, K), dtype=np.int8)
    d = np.empty((N, K // 32), dtype=np.uint16)
    lib().oracle_q8_0_quantize(_ptr(w), K, N, _ptr(q), _ptr(d))
    return q, d


def w8a8_quantize_rows(x_bits: np.ndarray):
    """BF16 activations [M, K] (uint16 bits) -> (x_q [M, K] int8, x_scale [M] float32), one
    symmetric scale per row (oracle.c: oracle_w8a8_quantize_rows)."""
    x = _c(x_bits, np.uint16)
    M, K = x.shape
    xq = np.empty((M, K), dtype=np.int8)
    xs = np.empty(M, dtype=np.float32)
    lib().oracle_w8a8_quantize_rows(_ptr(x), M, K, _ptr(xq), _ptr(xs))
    return xq, xs


def q8_0_blocks_from_split(q: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """Split layout -> ggml-style 34-byte blocks [N, K/32, 34] (oracle.c)."""
    qc = _c(q, np.int8)
    dc = _c(d_bits, np.uint16)
    N, K = qc.shape
    out = np.empty((N, K // 32, 34), dtype=np.uint8)
    lib().oracle_q8_0_blocks_from_split(_ptr(qc), _ptr(dc), K, N, _ptr(out))
    return out

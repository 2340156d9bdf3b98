"""Python binding of libw8a8_gb300.so, the GB300 small-M quantized weight GEMM library.

Argument marshalling only: every function forwards to the C ABI of the same name declared in
include/w8a8.h, passing device pointers taken from torch tensors and the current CUDA stream.
Since the C side sees bare pointers, the binding first checks each tensor it passes (contiguous,
the element size the call reads, long enough, in CUDA memory) and raises ValueError otherwise.
All arithmetic runs in the library's CUDA kernels; there is no fallback path, and a missing or
unloadable library raises at the first call.
"""
from __future__ import annotations

import ctypes
import functools
import os

from . import build as _build

__all__ = [
    "W8A8Error",
    "lib",
    "w8a8_version",
    "w8a8_packed_weight_bytes",
    "w8a8_workspace_bytes",
    "q8_0_workspace_bytes",
    "w8a8_workspace_init",
    "w8a8_workspace_status",
    "w8a8_pack_weights",
    "w8a8_gemm",
    "w8a8_gemm_acc",
    "q8_0_gemv",
    "q8_0_gemv_rms",
    "w8a8_plan",
    "w8a8_split_bounds",
    "w8a8_read_probe",
    "w8a8_quantize_activations",
    "q8_0_quantize",
    "q8_0_split_from_blocks",
    "q8_0_blocks_from_split",
    "alloc_workspace",
]

W8A8_OK = 0
W8A8_FLAG_PDL = 1
W8A8_FLAG_TENSOR_MEMORY_ARM = 2
W8A8_FLAG_TEST_STALL = 0x100
W8A8_DEV_WAIT_TIMEOUT = 1
W8A8_DEV_COUNTER_CORRUPT = 2

# Every symbol include/w8a8.h declares, with its ctypes signature.
_c_p = ctypes.c_void_p
_c_i = ctypes.c_int
_c_sz = ctypes.c_size_t


class PlanT(ctypes.Structure):
    _fields_ = [
        ("n8_tiles", ctypes.c_int),
        ("n_tiles", ctypes.c_int),
        ("k_blocks", ctypes.c_int),
        ("slabs", ctypes.c_longlong),
        ("blocks", ctypes.c_int),
        ("threads", ctypes.c_int),
        ("stage_slabs", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("smem_bytes", ctypes.c_size_t),
        ("workspace_bytes", ctypes.c_size_t),
        ("combine_pack_bits", ctypes.c_int),
        ("tile_rows", ctypes.c_int),
        ("tensor_memory", ctypes.c_int),
        ("row_chunks", ctypes.c_int),
        ("split_unit", ctypes.c_int),
    ]


SIGNATURES = {
    "w8a8_version": ([], _c_i),
    "w8a8_status_string": ([_c_i], ctypes.c_char_p),
    "w8a8_last_error": ([], ctypes.c_char_p),
    "w8a8_workspace_init": ([_c_p, _c_sz, _c_p], _c_i),
    "w8a8_workspace_status": ([_c_p, _c_sz, _c_p, ctypes.POINTER(ctypes.c_uint32)], _c_i),
    "w8a8_packed_weight_bytes": ([_c_i, _c_i], _c_sz),
    "w8a8_workspace_bytes": ([_c_i, _c_i, _c_i, _c_i], _c_sz),
    "w8a8_pack_weights": ([_c_p, _c_i, _c_i, _c_p, _c_p, _c_sz, _c_p], _c_i),
    "w8a8_gemm": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i, ctypes.c_uint, _c_p, _c_sz, _c_p], _c_i),
    "w8a8_gemm_acc": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i, ctypes.c_uint, _c_p, _c_sz, _c_p],
                      _c_i),
    "w8a8_gemm_no_alloc": ([_c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i, ctypes.c_uint, _c_p], _c_i),
    "w8a8_gemm_no_alloc_status": ([_c_p, ctypes.POINTER(ctypes.c_uint32)], _c_i),
    "w8a8_plan": ([_c_i, _c_i, _c_i, _c_i, ctypes.POINTER(PlanT)], _c_i),
    "w8a8_plan_flags": ([_c_i, _c_i, _c_i, _c_i, ctypes.c_uint, ctypes.POINTER(PlanT)], _c_i),
    "w8a8_split_bounds": ([_c_i, _c_i, _c_i, ctypes.POINTER(ctypes.c_longlong), _c_i], _c_i),
    "w8a8_split_bounds_m": ([_c_i, _c_i, _c_i, _c_i, ctypes.POINTER(ctypes.c_longlong), _c_i], _c_i),
    "q8_0_workspace_bytes": ([_c_i, _c_i, _c_i], _c_sz),
    "w8a8_read_probe": ([_c_p, _c_sz, _c_p, _c_p], _c_i),
    "w8a8_mma_rate_probe": ([_c_i, _c_i, _c_p, _c_p], _c_i),
    "w8a8_quantize_activations": ([_c_p, _c_p, _c_p, _c_i, _c_i, _c_p], _c_i),
    "q8_0_quantize": ([_c_p, _c_p, _c_p, _c_i, _c_i, _c_p], _c_i),
    "q8_0_split_from_blocks": ([_c_p, _c_p, _c_p, _c_i, _c_i, _c_p], _c_i),
    "q8_0_blocks_from_split": ([_c_p, _c_p, _c_p, _c_i, _c_i, _c_p], _c_i),
    "q8_0_gemv": ([_c_p, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, ctypes.c_uint, _c_p, _c_sz, _c_p], _c_i),
    "q8_0_gemv_rms": ([_c_p, _c_p, ctypes.c_float, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, ctypes.c_uint, _c_p, _c_sz, _c_p],
                      _c_i),
}

_lib = None


class W8A8Error(RuntimeError):
    def __init__(self, name, status, detail=""):
        self.status = status
        text = lib().w8a8_status_string(status).decode()
        super().__init__(f"{name} failed: {text} ({status}){': ' + detail if detail else ''}")


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded C library (built in-tree on first use if absent or stale)."""
    global _lib
    if _lib is None:
        path = _build.build()
        try:
            L = ctypes.CDLL(path)
        except OSError as e:  # no silent fallback: the CUDA path is the product
            raise RuntimeError(f"cannot load the CUDA library {path}: {e}") from e
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(name, rc):
    if rc != W8A8_OK:
        detail = lib().w8a8_last_error().decode()
        raise W8A8Error(name, rc, detail)


def _stream(stream):
    if stream is None:
        import torch

        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _nbytes(t):
    return t.numel() * t.element_size()


def _dev(t, name, nbytes=0, esize=None):
    """Layout check of a tensor whose pointer crosses the C ABI: contiguous, of element size
    `esize` where the call reads the tensor's shape, and at least `nbytes` long (the C side sees a
    bare pointer and cannot check).  Raises ValueError before any library call."""
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor (strides {tuple(t.stride())})")
    if esize is not None and t.element_size() != esize:
        raise ValueError(f"{name}: expected {esize}-byte elements, got {t.dtype}")
    if nbytes and t.nbytes < nbytes:
        raise ValueError(f"{name}: {t.nbytes} bytes, the call needs {nbytes}")


def _on_cuda(**tensors):
    """Every tensor of a call in CUDA memory (a host pointer handed to a kernel would fault):
    checked after the layout checks, just before the library call."""
    for name, t in tensors.items():
        if t is not None and not t.is_cuda:
            raise ValueError(f"{name}: expected a CUDA tensor, got device {t.device}")


# ---------------------------------------------------------------------------------------------

def w8a8_version() -> int:
    return lib().w8a8_version()


@functools.lru_cache(maxsize=1024)
def w8a8_packed_weight_bytes(K: int, N: int) -> int:
    return int(lib().w8a8_packed_weight_bytes(K, N))


def w8a8_workspace_bytes(M_max: int, K: int, N: int, blocks: int = 0) -> int:
    return int(lib().w8a8_workspace_bytes(M_max, K, N, blocks))


def q8_0_workspace_bytes(T_max: int, K: int, N: int) -> int:
    return int(lib().q8_0_workspace_bytes(T_max, K, N))


def w8a8_plan(M: int, K: int, N: int, blocks: int = 0, flags: int = 0) -> dict:
    p = PlanT()
    _check("w8a8_plan_flags", lib().w8a8_plan_flags(M, K, N, blocks, flags, ctypes.byref(p)))
    return {f: getattr(p, f) for f, _ in PlanT._fields_}


def w8a8_split_bounds(K: int, N: int, blocks: int, M: int = 1) -> list:
    n = blocks + 1
    arr = (ctypes.c_longlong * n)()
    if M == 1:
        _check("w8a8_split_bounds", lib().w8a8_split_bounds(K, N, blocks, arr, n))
    else:
        _check("w8a8_split_bounds_m", lib().w8a8_split_bounds_m(M, K, N, blocks, arr, n))
    return list(arr)


def w8a8_workspace_init(ws, stream=None) -> None:
    _dev(ws, "ws")
    _on_cuda(ws=ws)
    _check("w8a8_workspace_init", lib().w8a8_workspace_init(_ptr(ws), _nbytes(ws), _stream(stream)))


def w8a8_workspace_status(ws, stream=None) -> int:
    _dev(ws, "ws")
    _on_cuda(ws=ws)
    v = ctypes.c_uint32(0)
    _check("w8a8_workspace_status", lib().w8a8_workspace_status(_ptr(ws), _nbytes(ws), _stream(stream), ctypes.byref(v)))
    return int(v.value)


def alloc_workspace(nbytes: int, device="cuda", stream=None):
    """A zeroed workspace tensor (uint8) of at least nbytes (torch allocations are 512-B aligned)."""
    import torch

    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    w8a8_workspace_init(ws, stream)
    return ws


def w8a8_pack_weights(W, W_packed=None, ws=None, stream=None):
    """Pack W [K,N] int8 (device) into the kernel layout; returns the packed uint8 tensor."""
    import torch

    K, N = W.shape
    _dev(W, "W", esize=1)
    if W_packed is None:
        W_packed = torch.empty(w8a8_packed_weight_bytes(K, N), dtype=torch.uint8, device=W.device)
    _dev(W_packed, "W_packed", w8a8_packed_weight_bytes(K, N))
    if ws is not None:
        _dev(ws, "ws")
    _on_cuda(W=W, W_packed=W_packed, ws=ws)
    rc = lib().w8a8_pack_weights(_ptr(W), K, N, _ptr(W_packed), _ptr(ws), _nbytes(ws) if ws is not None else 0,
                                 _stream(stream))
    _check("w8a8_pack_weights", rc)
    return W_packed


def w8a8_gemm(x_q, x_scale, W_packed, w_scale, ws, N: int, out=None, blocks: int = 0, flags: int = 0,
              stream=None):
    """out[M,N] bf16 = bf16((float(x_q @ W) * x_scale) * w_scale) through the C ABI."""
    import torch

    M, K = x_q.shape
    _dev(x_q, "x_q", esize=1)
    _dev(x_scale, "x_scale", 4 * M)
    _dev(W_packed, "W_packed", w8a8_packed_weight_bytes(K, N))
    _dev(w_scale, "w_scale", 4 * N)
    _dev(ws, "ws")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x_q.device)
    _dev(out, "out", 2 * M * N)
    _on_cuda(x_q=x_q, x_scale=x_scale, W_packed=W_packed, w_scale=w_scale, ws=ws, out=out)
    rc = lib().w8a8_gemm(_ptr(x_q), _ptr(x_scale), _ptr(W_packed), _ptr(w_scale), _ptr(out), M, K, N, blocks,
                         flags, _ptr(ws), _nbytes(ws), _stream(stream))
    _check("w8a8_gemm", rc)
    return out


def w8a8_gemm_acc(x_q, x_scale, W_packed, w_scale, ws, N: int, out=None, acc=None, blocks: int = 0, flags: int = 0,
                  stream=None):
    """w8a8_gemm that also returns the exact int32 sums: (out [M,N] bf16, acc [M,N] int32)."""
    import torch

    M, K = x_q.shape
    _dev(x_q, "x_q", esize=1)
    _dev(x_scale, "x_scale", 4 * M)
    _dev(W_packed, "W_packed", w8a8_packed_weight_bytes(K, N))
    _dev(w_scale, "w_scale", 4 * N)
    _dev(ws, "ws")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x_q.device)
    if acc is None:
        acc = torch.empty((M, N), dtype=torch.int32, device=x_q.device)
    _dev(out, "out", 2 * M * N)
    _dev(acc, "acc", 4 * M * N, esize=4)
    _on_cuda(x_q=x_q, x_scale=x_scale, W_packed=W_packed, w_scale=w_scale, ws=ws, out=out, acc=acc)
    rc = lib().w8a8_gemm_acc(_ptr(x_q), _ptr(x_scale), _ptr(W_packed), _ptr(w_scale), _ptr(out), _ptr(acc), M, K, N,
                             blocks, flags, _ptr(ws), _nbytes(ws), _stream(stream))
    _check("w8a8_gemm_acc", rc)
    return out, acc


def _q8_args(x, q, d, ws, K, N):
    _dev(x, "x", esize=2)
    if q.dim() != 2 or q.shape[1] != K:
        raise ValueError(f"q: expected shape [N, {K}], got {tuple(q.shape)}")
    _dev(q, "q", esize=1)
    _dev(d, "d", 2 * N * (K // 32))
    _dev(ws, "ws")


def q8_0_gemv(x, q, d, ws, y=None, flags: int = 0, stream=None):
    """y[T,N] bf16 = x[T,K] (bf16) times the Q8_0 weights (q [N,K] int8, d [N,K/32] fp16)."""
    import torch

    T, K = x.shape
    N = q.shape[0]
    _q8_args(x, q, d, ws, K, N)
    if y is None:
        y = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    _dev(y, "y", 2 * T * N)
    _on_cuda(x=x, q=q, d=d, ws=ws, y=y)
    rc = lib().q8_0_gemv(_ptr(x), _ptr(q), _ptr(d), _ptr(y), T, K, N, flags, _ptr(ws), _nbytes(ws),
                         _stream(stream))
    _check("q8_0_gemv", rc)
    return y


def q8_0_gemv_rms(x, gamma, eps: float, q, d, ws, y=None, flags: int = 0, stream=None):
    """y[T,N] bf16 = rs * (x * gamma) [T,K] times the Q8_0 weights, rs[t] = 1 / sqrt(mean_k x[t,k]^2 + eps)."""
    import torch

    T, K = x.shape
    N = q.shape[0]
    _q8_args(x, q, d, ws, K, N)
    _dev(gamma, "gamma", 2 * K)
    if y is None:
        y = torch.empty((T, N), dtype=torch.bfloat16, device=x.device)
    _dev(y, "y", 2 * T * N)
    _on_cuda(x=x, gamma=gamma, q=q, d=d, ws=ws, y=y)
    rc = lib().q8_0_gemv_rms(_ptr(x), _ptr(gamma), float(eps), _ptr(q), _ptr(d), _ptr(y), T, K, N, flags, _ptr(ws),
                             _nbytes(ws), _stream(stream))
    _check("q8_0_gemv_rms", rc)
    return y


def w8a8_read_probe(buf, sink, stream=None) -> None:
    """Read the whole device tensor `buf` once (16-byte loads) and discard it: the HBM read-rate
    probe.  `sink` is an 8-byte device tensor the kernel may write."""
    _dev(buf, "buf")
    _dev(sink, "sink", 8)
    _on_cuda(buf=buf, sink=sink)
    _check("w8a8_read_probe", lib().w8a8_read_probe(_ptr(buf), _nbytes(buf), _ptr(sink), _stream(stream)))


def w8a8_mma_rate_probe(kind: int, iters: int, sink, stream=None) -> None:
    """Launch the tensor-pipe rate probe (kind 0: fp16 m16n8k16, kind 1: int8 m16n8k32); the
    caller times it.  `sink` is an 8-byte device tensor the kernel may write."""
    _dev(sink, "sink", 8)
    _on_cuda(sink=sink)
    _check("w8a8_mma_rate_probe", lib().w8a8_mma_rate_probe(kind, iters, _ptr(sink), _stream(stream)))


def w8a8_quantize_activations(x, x_q=None, x_scale=None, stream=None):
    """bf16 x [M, K] -> (x_q [M, K] int8, x_scale [M] fp32), one symmetric scale per row."""
    import torch

    M, K = x.shape
    _dev(x, "x", esize=2)
    if x_q is None:
        x_q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if x_scale is None:
        x_scale = torch.empty(M, dtype=torch.float32, device=x.device)
    _dev(x_q, "x_q", M * K)
    _dev(x_scale, "x_scale", 4 * M)
    _on_cuda(x=x, x_q=x_q, x_scale=x_scale)
    _check("w8a8_quantize_activations",
           lib().w8a8_quantize_activations(_ptr(x), _ptr(x_q), _ptr(x_scale), M, K, _stream(stream)))
    return x_q, x_scale


def q8_0_quantize(w, q=None, d=None, stream=None):
    """bf16 weights w [N, K] -> Q8_0 split layout (q [N, K] int8, d [N, K/32] fp16 bits as int16)."""
    import torch

    N, K = w.shape
    _dev(w, "w", esize=2)
    if q is None:
        q = torch.empty((N, K), dtype=torch.int8, device=w.device)
    if d is None:
        d = torch.empty((N, K // 32), dtype=torch.int16, device=w.device)
    _dev(q, "q", N * K)
    _dev(d, "d", 2 * N * (K // 32))
    _on_cuda(w=w, q=q, d=d)
    _check("q8_0_quantize", lib().q8_0_quantize(_ptr(w), _ptr(q), _ptr(d), K, N, _stream(stream)))
    return q, d


def q8_0_split_from_blocks(blocks, K: int, N: int, q=None, d=None, stream=None):
    """ggml Q8_0 blocks (uint8, N * K/32 * 34 bytes) -> (q [N, K] int8, d [N, K/32] int16 bits)."""
    import torch

    _dev(blocks, "blocks", 34 * N * (K // 32))
    if q is None:
        q = torch.empty((N, K), dtype=torch.int8, device=blocks.device)
    if d is None:
        d = torch.empty((N, K // 32), dtype=torch.int16, device=blocks.device)
    _dev(q, "q", N * K)
    _dev(d, "d", 2 * N * (K // 32))
    _on_cuda(blocks=blocks, q=q, d=d)
    _check("q8_0_split_from_blocks", lib().q8_0_split_from_blocks(_ptr(blocks), _ptr(q), _ptr(d), K, N, _stream(stream)))
    return q, d


def q8_0_blocks_from_split(q, d, blocks=None, stream=None):
    """(q [N, K] int8, d [N, K/32] fp16 bits) -> ggml Q8_0 blocks (uint8 [N, K/32, 34])."""
    import torch

    N, K = q.shape
    _dev(q, "q", esize=1)
    _dev(d, "d", 2 * N * (K // 32))
    if blocks is None:
        blocks = torch.empty((N, K // 32, 34), dtype=torch.uint8, device=q.device)
    _dev(blocks, "blocks", 34 * N * (K // 32))
    _on_cuda(q=q, d=d, blocks=blocks)
    _check("q8_0_blocks_from_split", lib().q8_0_blocks_from_split(_ptr(q), _ptr(d), _ptr(blocks), K, N, _stream(stream)))
    return blocks

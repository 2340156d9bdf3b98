"""The Python binding's marshalling checks, on the CPU: every tensor whose pointer crosses the C ABI
is checked for layout, element size, length and device before any library call, so that a host
tensor, a strided view or a short buffer is a ValueError and never a kernel reading past a bare
pointer.  Host (CPU) tensors of the right size fail the device check, which comes last: reaching
it shows every earlier check passed."""
import pytest
import torch

import int8_weight_gemm_gb300 as lib8


def _raises(fragment, fn, *args, **kw):
    with pytest.raises(ValueError, match=fragment):
        fn(*args, **kw)


def _w8a8(M=16, K=512, N=256):
    return dict(x_q=torch.zeros((M, K), dtype=torch.int8), x_scale=torch.zeros(M),
                W_packed=torch.zeros(lib8.w8a8_packed_weight_bytes(K, N), dtype=torch.uint8),
                w_scale=torch.zeros(N), ws=torch.zeros(1 << 16, dtype=torch.uint8), N=N)


def test_w8a8_gemm_arguments():
    a = _w8a8()
    _raises("x_q: expected a CUDA tensor", lib8.w8a8_gemm, **a)
    _raises("x_q: expected a contiguous", lib8.w8a8_gemm, **dict(a, x_q=torch.zeros((512, 16), dtype=torch.int8).t()))
    _raises("x_q: expected 1-byte", lib8.w8a8_gemm, **dict(a, x_q=torch.zeros((16, 512), dtype=torch.int16)))
    _raises("x_scale: 60 bytes, the call needs 64", lib8.w8a8_gemm, **dict(a, x_scale=torch.zeros(15)))
    _raises("W_packed: .* the call needs 131072", lib8.w8a8_gemm,
            **dict(a, W_packed=torch.zeros(131071, dtype=torch.uint8)))
    _raises("w_scale: .* the call needs 1024", lib8.w8a8_gemm, **dict(a, w_scale=torch.zeros(128)))
    _raises("out: .* the call needs 8192", lib8.w8a8_gemm, **a, out=torch.zeros((16, 255), dtype=torch.bfloat16))
    _raises("out: expected a contiguous", lib8.w8a8_gemm,
            **a, out=torch.zeros((256, 16), dtype=torch.bfloat16).t())


def test_pack_and_workspace_arguments():
    _raises("W: expected 1-byte", lib8.w8a8_pack_weights, torch.zeros((512, 256), dtype=torch.float32))
    _raises("W: expected a CUDA tensor", lib8.w8a8_pack_weights, torch.zeros((512, 256), dtype=torch.int8))
    _raises("W_packed: .* the call needs 131072", lib8.w8a8_pack_weights, torch.zeros((512, 256), dtype=torch.int8),
            W_packed=torch.zeros(1024, dtype=torch.uint8))
    _raises("ws: expected a CUDA tensor", lib8.w8a8_workspace_init, torch.zeros(256, dtype=torch.uint8))
    _raises("ws: expected a CUDA tensor", lib8.w8a8_workspace_status, torch.zeros(256, dtype=torch.uint8))
    _raises("sink: 4 bytes, the call needs 8", lib8.w8a8_read_probe, torch.zeros(64, dtype=torch.uint8),
            torch.zeros(1, dtype=torch.int32))


def _q8(T=4, K=4096, N=320):
    return dict(x=torch.zeros((T, K), dtype=torch.bfloat16), q=torch.zeros((N, K), dtype=torch.int8),
                d=torch.zeros((N, K // 32), dtype=torch.int16), ws=torch.zeros(1 << 16, dtype=torch.uint8))


def test_q8_0_gemv_arguments():
    a = _q8()
    _raises("x: expected a CUDA tensor", lib8.q8_0_gemv, **a)
    _raises("x: expected 2-byte", lib8.q8_0_gemv, **dict(a, x=torch.zeros((4, 4096))))
    _raises(r"q: expected shape \[N, 4096\]", lib8.q8_0_gemv, **dict(a, q=torch.zeros((320, 2048), dtype=torch.int8)))
    _raises("q: expected 1-byte", lib8.q8_0_gemv, **dict(a, q=torch.zeros((320, 4096), dtype=torch.int16)))
    _raises("d: .* the call needs 81920", lib8.q8_0_gemv, **dict(a, d=torch.zeros((320, 127), dtype=torch.int16)))
    _raises("y: .* the call needs 2560", lib8.q8_0_gemv, **a, y=torch.zeros((3, 320), dtype=torch.bfloat16))
    g = torch.ones(4096, dtype=torch.bfloat16)
    _raises("x: expected a CUDA tensor", lib8.q8_0_gemv_rms, a["x"], g, 1e-6, a["q"], a["d"], a["ws"])
    _raises("gamma: .* the call needs 8192", lib8.q8_0_gemv_rms, a["x"], g[:4000], 1e-6, a["q"], a["d"], a["ws"])


def test_quantisation_arguments():
    x = torch.zeros((8, 512), dtype=torch.bfloat16)
    _raises("x: expected a CUDA tensor", lib8.w8a8_quantize_activations, x)
    _raises("x: expected 2-byte", lib8.w8a8_quantize_activations, x.float())
    _raises("x_q: .* the call needs 4096", lib8.w8a8_quantize_activations, x, x_q=torch.zeros((8, 511), dtype=torch.int8))
    _raises("x_scale: .* the call needs 32", lib8.w8a8_quantize_activations, x, x_scale=torch.zeros(7))
    w = torch.zeros((320, 4096), dtype=torch.bfloat16)
    _raises("w: expected a CUDA tensor", lib8.q8_0_quantize, w)
    _raises("d: .* the call needs 81920", lib8.q8_0_quantize, w, d=torch.zeros((320, 64), dtype=torch.int16))
    blocks = torch.zeros((320, 128, 34), dtype=torch.uint8)
    _raises("blocks: expected a CUDA tensor", lib8.q8_0_split_from_blocks, blocks, 4096, 320)
    _raises("blocks: .* the call needs 1392640", lib8.q8_0_split_from_blocks, blocks[:100], 4096, 320)
    q, d = torch.zeros((320, 4096), dtype=torch.int8), torch.zeros((320, 128), dtype=torch.int16)
    _raises("q: expected a CUDA tensor", lib8.q8_0_blocks_from_split, q, d)
    _raises("blocks: .* the call needs 1392640", lib8.q8_0_blocks_from_split, q, d,
            blocks=torch.zeros(1000, dtype=torch.uint8))

"""Helpers shared by the GPU tests: run the library on seeded inputs and return host arrays."""
import numpy as np
import torch

import int8_weight_gemm_gb300 as lib8


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


class W8A8Case:
    """Device copies of one W8A8 problem (packed weight, scales, workspace).  base_flags are OR-ed
    into every call's flags."""

    base_flags = 0

    def __init__(self, x_q, x_scale, W, w_scale, M_max=None, blocks=0):
        dev = torch.device("cuda")
        self.M, self.K = x_q.shape
        self.N = W.shape[1]
        self.x = torch.from_numpy(np.ascontiguousarray(x_q)).to(dev)
        self.xs = torch.from_numpy(np.ascontiguousarray(x_scale)).to(dev)
        self.W = torch.from_numpy(np.ascontiguousarray(W)).to(dev)
        self.ws_scale = torch.from_numpy(np.ascontiguousarray(w_scale)).to(dev)
        self.ws = lib8.alloc_workspace(lib8.w8a8_workspace_bytes(M_max or self.M, self.K, self.N, blocks))
        self.Wp = lib8.w8a8_pack_weights(self.W, ws=self.ws)
        self.blocks = blocks

    def run(self, out=None, blocks=None, flags=0):
        return lib8.w8a8_gemm(self.x, self.xs, self.Wp, self.ws_scale, self.ws, self.N, out=out,
                              blocks=self.blocks if blocks is None else blocks, flags=flags | self.base_flags)

    def run_acc(self, blocks=None, flags=0):
        """The same call through w8a8_gemm_acc: (out bf16, acc int32) as device tensors."""
        return lib8.w8a8_gemm_acc(self.x, self.xs, self.Wp, self.ws_scale, self.ws, self.N,
                                  blocks=self.blocks if blocks is None else blocks, flags=flags | self.base_flags)

    def status(self):
        return lib8.w8a8_workspace_status(self.ws)

"""Device-resident operands for the tkg GEMMs (torch is used for device
memory, pinned host buffers and streams only; the GEMM itself is one call into
the C library).
"""
from __future__ import annotations

import numpy as np
import torch

from . import tkg


def _to_dev(arr: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(arr))
    return t.to(device)


class DeviceGemm:
    """Holds A, B (and scales) of one problem on a CUDA device plus an output
    buffer, and launches the matching tkg entry point."""

    def __init__(self, ops, device="cuda", out: torch.Tensor | None = None):
        self.kind = ops.kind
        self.M, self.N, self.K = ops.M, ops.N, ops.K
        self.device = torch.device(device)
        self.a = _to_dev(ops.a, self.device)
        self.b = _to_dev(ops.b, self.device)
        self.scale_a = self.scale_b = self.sfa = self.sfb = None
        if ops.kind in ("fp8", "nvfp4"):
            self.scale_a = torch.tensor([ops.scale_a], dtype=torch.float32, device=self.device)
            self.scale_b = torch.tensor([ops.scale_b], dtype=torch.float32, device=self.device)
        if ops.kind == "nvfp4":
            self.sfa = _to_dev(ops.sfa, self.device)
            self.sfb = _to_dev(ops.sfb, self.device)
        self.c = out if out is not None else torch.empty((self.M, self.N), dtype=torch.bfloat16, device=self.device)

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def scales(self):
        if self.kind == "bf16":
            return None
        return (self.scale_a, self.scale_b, self.sfa, self.sfb)

    def run(self, stream=None, check=True) -> int:
        fn = {"bf16": tkg.tkg_gemm_bf16, "fp8": tkg.tkg_gemm_fp8, "nvfp4": tkg.tkg_gemm_nvfp4}[self.kind]
        return fn(self.M, self.N, self.K, self.a, self.b, self.c, self.scales(), stream=stream, check=check)

    def c_bits(self) -> np.ndarray:
        """Output as raw bf16 bit patterns (uint16) on the host."""
        return self.c.view(torch.int16).cpu().numpy().view(np.uint16)

    def input_bytes(self) -> int:
        n = self.a.numel() * self.a.element_size() + self.b.numel() * self.b.element_size()
        for t in (self.scale_a, self.scale_b, self.sfa, self.sfb):
            if t is not None:
                n += t.numel() * t.element_size()
        return n

    def output_bytes(self) -> int:
        return self.c.numel() * self.c.element_size()

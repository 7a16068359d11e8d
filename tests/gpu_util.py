"""Helpers for the GPU parity tests: strided device buffers with NaN
sentinels in their padding, and one call per operation through the C ABI
binding that returns every output."""
from __future__ import annotations

import numpy as np
import torch

import oracle

NAN_BITS = {torch.bfloat16: 0x7FC0, torch.float16: 0x7E00}


class Strided:
    """A [M, N] view inside a NaN-filled buffer with row stride `stride` and
    `lead` spare elements before row 0 (to misalign the base) and 64 after."""

    def __init__(self, M, N, dtype, stride=None, lead=0, device="cuda"):
        self.M, self.N, self.dtype = M, N, dtype
        self.stride = stride or N
        self.lead = lead
        total = lead + (M * self.stride if M else 0) + 64
        self.buf = torch.full((total,), float("nan"), dtype=dtype, device=device)
        self.view = self.buf.as_strided((M, N), (self.stride, 1), lead)

    @classmethod
    def of(cls, t_cpu, stride=None, lead=0):
        s = cls(t_cpu.shape[0], t_cpu.shape[1], t_cpu.dtype, stride, lead)
        s.view.copy_(t_cpu)
        return s

    def padding_intact(self) -> bool:
        """Every element outside the view still holds the NaN sentinel."""
        mask = torch.ones(self.buf.numel(), dtype=torch.bool, device=self.buf.device)
        if self.M:
            mask.as_strided((self.M, self.N), (self.stride, 1), self.lead).fill_(False)
        pad = self.buf[mask]
        if self.dtype in NAN_BITS:
            return bool((pad.view(torch.int16) == NAN_BITS[self.dtype]).all())
        return bool(torch.isnan(pad).all())


def f64(t):
    return t.detach().double().cpu().numpy()


def unit_xhat(x64, ln: bool, eps: float):
    """xhat of every element (oracle forward with unit weight, no bias)."""
    N = x64.shape[1]
    if ln:
        return oracle.ln_fwd(x64, np.ones(N), None, 0.0, eps)[0]
    return oracle.rms_fwd(x64, np.ones(N), 0.0, eps)[0]


def dw_scale(dy64, xhat64):
    """Magnitude of the terms summed into each dW column."""
    return np.abs(dy64 * xhat64).sum(axis=0)


def bits_equal(a, b) -> bool:
    if a.dtype != b.dtype or a.shape != b.shape:
        return False
    if a.dtype in (torch.bfloat16, torch.float16):
        return bool(torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16)))
    return bool(torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32)))


def workspace(g, M, N, dw, db=False):
    nb = g.norm_bwd_workspace_bytes(M, N, dw, db)
    if nb == 0:
        return None
    return torch.empty(nb, dtype=torch.uint8, device="cuda")

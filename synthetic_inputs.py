"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers; it holds none of the normalisation
arithmetic.  Both the CUDA path and the FP64 oracle consume the exact bytes
produced here.

Recipe (the workloads on "perf(norm): skip dW/dB calculation when parameters
are frozen", Benchmark Results, and "fix(cutedsl): fuse Gemma RMSNorm weight
offset in FP32", PyTorch accuracy comparison and minimal reproduction):

* every tensor is drawn from its own torch CPU generator seeded with
  ``seed * 1000 + k`` (k fixed per role below), in float32, then scaled and
  rounded once to its storage dtype;
* activations x, upstream gradients dy, residuals and residual-output
  gradients ~ N(0, 1) (stress: x ~ N(0, 3) with an i.i.d. 1 % of entries
  multiplied by 100);
* plain weights w = 1 + 0.1 * N(0, 1); Gemma weights w = 0.01 * N(0, 1)
  (used with offset 1); LayerNorm bias b = 0.1 * N(0, 1).
"""
from __future__ import annotations

import torch

# Sub-stream index of each tensor role.
ROLE = {"x": 0, "dy": 1, "w": 2, "b": 3, "residual": 4, "dh_out": 5,
        "outlier_mask": 6}

TORCH_DTYPES = {"float32": torch.float32, "float16": torch.float16,
                "bfloat16": torch.bfloat16}


def _gen(seed: int, role: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1000 + ROLE[role])
    return g


def normal(shape, seed: int, role: str, dtype="bfloat16", scale=1.0, shift=0.0):
    """``shift + scale * N(0,1)`` drawn in float32, rounded once to ``dtype``."""
    t = torch.randn(*shape, generator=_gen(seed, role), dtype=torch.float32)
    if scale != 1.0:
        t = t * scale
    if shift != 0.0:
        t = t + shift
    return t.to(TORCH_DTYPES[dtype])


def activations(M, N, seed, role="x", dtype="bfloat16", outliers=False):
    """Activation-like rows. ``outliers``: N(0,3) with 1 % of entries x100."""
    if not outliers:
        return normal((M, N), seed, role, dtype)
    t = torch.randn(M, N, generator=_gen(seed, role), dtype=torch.float32) * 3.0
    u = torch.rand(M, N, generator=_gen(seed, "outlier_mask"), dtype=torch.float32)
    t = torch.where(u < 0.01, t * 100.0, t)
    return t.to(TORCH_DTYPES[dtype])


def weight(N, seed, dtype="bfloat16", gemma=False):
    """Plain weight 1 + 0.1 N(0,1), or Gemma weight 0.01 N(0,1)."""
    if gemma:
        return normal((N,), seed, "w", dtype, scale=0.01)
    return normal((N,), seed, "w", dtype, scale=0.1, shift=1.0)


def bias(N, seed, dtype="bfloat16"):
    return normal((N,), seed, "b", dtype, scale=0.1)


def norm_case(M, N, seed=0, dtype="bfloat16", w_dtype=None, gemma=False,
              outliers=False, with_bias=True, fused_add=False):
    """All inputs of one forward+backward case as CPU tensors.

    Keys: x, dy, w, b (LayerNorm bias), and for fused_add also residual and
    dh_out.
    """
    w_dtype = w_dtype or dtype
    case = {
        "x": activations(M, N, seed, "x", dtype, outliers=outliers),
        "dy": normal((M, N), seed, "dy", dtype),
        "w": weight(N, seed, w_dtype, gemma=gemma),
    }
    if with_bias:
        case["b"] = bias(N, seed, w_dtype)
    if fused_add:
        case["residual"] = normal((M, N), seed, "residual", dtype)
        case["dh_out"] = normal((M, N), seed, "dh_out", dtype)
    return case

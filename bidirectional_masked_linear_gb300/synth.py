"""Seeded synthetic inputs shaped like the LION pages' workloads.

This module only draws random numbers: it holds none of the operator's
arithmetic, so the CUDA path and the float64 oracle can both be fed from it.

Recipe (every workload):

* ``q, k, v`` ~ N(0, 1) from ``numpy.random.default_rng(seed)`` (PCG64,
  standard normal), drawn in float32 and then rounded to the compute dtype
  (bf16 by round-to-nearest-even through ``torch.Tensor.to``) -- the rounded
  values are the exact inputs both sides see.
* decays are passed to the operator as ``log_lambda = log(lambda) <= 0``:

  - LION-LIT: none (all-ones mask);
  - LION-D: one lambda per head, ``lambda = sigmoid(u)``, ``u ~ U(2, 5)`` for the
    tiny case, or ``lambda ~ U(0.9, 0.999)`` for the vision/MLM shapes;
  - LION-S: per (batch, head, token) ``lambda_i = sigmoid(a_i)``, ``a_i ~ N(3, 1)``.

  ``log(sigmoid(a))`` is evaluated as ``-log1p(exp(-a))`` in float64 and stored
  as float32.

The shapes stand in for the pages' ImageNet (ViT-T / ViT-B patch sequences),
C4 MLM (BERT-large), 2496-px image and Long-Range-Arena text (length 4096)
workloads, whose data are not available.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

MASK_NAMES = {"lit": 0, "d": 1, "s": 2}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d: int
    dtype: str          # "bf16" or "fp32"
    masks: tuple        # mask names the workload is run with
    chunks: tuple       # chunk lengths the workload is run with
    lam: str            # "u25" (sigmoid(U(2,5))), "u09" (U(0.9,0.999)) for LION-D
    seed: int


WORKLOADS = {
    "tiny_d_fp32": Workload("tiny_d_fp32", 1, 2, 64, 16, "fp32", ("d",), (16,), "u25", 1001),
    "vit_t_s": Workload("vit_t_s", 64, 3, 197, 64, "bf16", ("s",), (64,), "u09", 1002),
    "vit_b": Workload("vit_b", 64, 12, 197, 64, "bf16", ("lit", "d", "s"), (32, 64, 128), "u09", 1003),
    "bert_large": Workload("bert_large", 32, 16, 512, 64, "bf16", ("d", "s"), (64, 128), "u09", 1004),
    "hires_2496": Workload("hires_2496", 2, 12, 24337, 64, "bf16", ("d", "s"), (64, 128), "u09", 1005),
    "lra_4096": Workload("lra_4096", 16, 8, 4096, 64, "bf16", ("d", "s"), (64, 128), "u09", 1006),
}


def _round(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    if dtype == "fp32":
        return t
    raise ValueError(f"unknown dtype {dtype!r}")


def _log_sigmoid(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return -np.log1p(np.exp(-a))


def make_inputs(B: int, H: int, L: int, d: int, mask: str, dtype: str = "bf16",
                seed: int = 0, lam: str = "u09") -> dict:
    """Return CPU tensors ``q, k, v`` ([B, H, L, d], ``dtype``) and ``log_lambda``
    (float32; ``None`` for LIT, ``[H]`` for D, ``[B, H, L]`` for S)."""
    if mask not in MASK_NAMES:
        raise ValueError(f"unknown mask {mask!r}")
    rng = np.random.default_rng(seed)
    shape = (B, H, L, d)
    q = _round(rng.standard_normal(shape, dtype=np.float32), dtype)
    k = _round(rng.standard_normal(shape, dtype=np.float32), dtype)
    v = _round(rng.standard_normal(shape, dtype=np.float32), dtype)
    if mask == "lit":
        ll = None
    elif mask == "d":
        if lam == "u25":
            lamv = 1.0 / (1.0 + np.exp(-rng.uniform(2.0, 5.0, size=H)))
            ll = np.log(lamv)
        else:
            ll = np.log(rng.uniform(0.9, 0.999, size=H))
        ll = torch.from_numpy(ll.astype(np.float32))
    else:
        a = rng.normal(3.0, 1.0, size=(B, H, L))
        ll = torch.from_numpy(_log_sigmoid(a).astype(np.float32))
    return {"q": q, "k": k, "v": v, "log_lambda": ll, "mask": MASK_NAMES[mask]}


def workload_inputs(name: str, mask: str) -> dict:
    w = WORKLOADS[name]
    return make_inputs(w.B, w.H, w.L, w.d, mask, w.dtype, w.seed, w.lam)


def as_f64(t):
    """Exact float64 copy (numpy) of a tensor's values, or ``None``."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()

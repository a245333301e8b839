"""Seeded synthetic tensors for the attention workloads.

Q, K, V and dO are drawn from N(0, 1) with one torch CPU generator seeded
once, in the order Q, K, V, dO, each as float32 and then rounded to bf16.
Layout is BSHD ([batch][seq][head][head_dim], head_dim contiguous), the layout
the attention library takes.  Nothing here computes attention.
"""
from __future__ import annotations

import numpy as np
import torch

from .masks import make_mask


def qkv_do(B: int, Sq: int, Skv: int, H: int, d: int, seed: int = 0,
           device: str = "cpu", dtype=torch.bfloat16):
    """Return (q, k, v, do) as bf16 tensors in BSHD layout.

    The draws happen on the CPU generator (so the values are the same whatever
    the device) and the tensors are then moved to ``device``.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn(B, Sq, H, d, generator=g, dtype=torch.float32).to(dtype)
    k = torch.randn(B, Skv, H, d, generator=g, dtype=torch.float32).to(dtype)
    v = torch.randn(B, Skv, H, d, generator=g, dtype=torch.float32).to(dtype)
    do = torch.randn(B, Sq, H, d, generator=g, dtype=torch.float32).to(dtype)
    if device != "cpu":
        q, k, v, do = (t.to(device) for t in (q, k, v, do))
    return q, k, v, do


def randn_bf16(*shape, seed: int, device: str = "cpu") -> torch.Tensor:
    """One N(0, 1) bf16 tensor of ``shape`` from a torch CPU generator seeded
    with ``seed`` (float32 draws rounded to bf16), moved to ``device``; the
    values do not depend on the device."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    t = torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return t.to(device) if device != "cpu" else t


def bounds_tensor(masks_per_batch, device: str = "cpu") -> torch.Tensor:
    """Stack per-(batch, mask-head) bound vectors into one int32 tensor of shape
    [4][B][Hm][Skv] (LTS, LTE, UTS, UTE), the layout the library reads.

    ``masks_per_batch`` is a list over b of lists over hm of (lts, lte, uts, ute).
    """
    B = len(masks_per_batch)
    Hm = len(masks_per_batch[0])
    S = len(masks_per_batch[0][0][0])
    out = np.empty((4, B, Hm, S), dtype=np.int32)
    for b in range(B):
        for hm in range(Hm):
            for t in range(4):
                out[t, b, hm] = masks_per_batch[b][hm][t]
    return torch.from_numpy(out).to(device)


def mask_bounds(name: str, B: int, S: int, seed: int = 0, per_batch_seed: bool = True,
                device: str = "cpu", **params) -> torch.Tensor:
    """Bounds of a named mask for every batch entry, one mask head (Hm = 1).

    With ``per_batch_seed`` batch entry b uses seed ``seed + b`` (documents differ
    across the batch); otherwise all entries share one draw.
    """
    per_b = []
    for b in range(B):
        s = seed + b if per_batch_seed else seed
        per_b.append([make_mask(name, S, s, **params)])
    return bounds_tensor(per_b, device=device)

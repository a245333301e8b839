"""A model of the forward kernel's rounding steps, for tests.

Not the oracle (``oracle/`` holds the plain definition in fp64); this is the
streaming softmax of the FlashAttention-2 page («Блочная обработка сохраняет
общую нормализацию»: running maximum and sum over key blocks, partial outputs
rescaled) written with the precision of each step of the CUDA forward pass:

  S        fp32 (exact bf16 products, one rounding of the row . key sum)
  m        fp32 row maximum of S * scale * log2(e), per 128-key tile; the
           reference maximum moves only when a tile's maximum exceeds it by
           more than 8 (factor 256), and O and l are rescaled then
  p        exp2(S * scale * log2(e) - m) in fp32
  l        fp32 sum of the fp32 p
  P        p rounded to bf16 (round to nearest even) for the P V product
  O        fp32 accumulation of bf16(P) V
  output   O / l in fp32, rounded to bf16

It lets a test separate the rounding that this design implies from a defect:
the kernel's output should equal the model's up to an ulp in a few elements,
and the model's own error against the fp64 oracle shows how much of a
parity difference the bf16 rounding accounts for.
"""
from __future__ import annotations

import numpy as np
import torch

LOG2E = 1.4426950408889634


def bf16(x) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.bfloat16().float().numpy().astype(np.float64)


def f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def bf16_half_ulp(x) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) at |x|."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def forward_head(q, k, v, hidden, scale, tile=128):
    """Model of the kernel's O for one head: q [Sq][d], k, v [Skv][d] (float64
    holding bf16 values), ``hidden`` the dense [Sq][Skv] mask (True = hidden).
    Returns (O as delivered in bf16, O in fp32 before the output rounding)."""
    Sq, Skv = q.shape[0], k.shape[0]
    c = float(np.float32(scale * LOG2E))
    s_all = np.where(hidden, -np.inf, f32(q @ k.T))
    m_used = np.full(Sq, -np.inf)
    l = np.zeros(Sq)
    O = np.zeros((Sq, v.shape[1]))
    for k0 in range(0, Skv, tile):
        s = s_all[:, k0:k0 + tile]
        m_tile = f32(s.max(axis=1) * c)
        grow = m_tile > m_used + 8
        m_new = np.where(grow, m_tile, m_used)
        with np.errstate(invalid="ignore"):
            alpha = np.where(grow, np.where(np.isneginf(m_used), 0.0, f32(np.exp2(m_used - m_new))), 1.0)
        l = f32(l * alpha)
        O = f32(O * alpha[:, None])
        m_used = m_new
        m_ref = np.where(np.isneginf(m_used), 0.0, m_used)
        p = f32(np.exp2(f32(s * c - m_ref[:, None])))
        l = f32(l + p.sum(axis=1))
        O = f32(O + bf16(p) @ v[k0:k0 + tile])
    inv = f32(np.where(l > 0, 1.0 / np.where(l > 0, l, 1.0), 0.0))
    o32 = f32(O * inv[:, None])
    return bf16(o32), o32

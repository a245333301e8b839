"""FP8 (e4m3) forward oracle: per-tile quantisation and the attention it
computes, in float64.  Test infrastructure only (see ``oracle/__init__.py``).

The ROCm page («Современное состояние Flash Attention на ROCm») reports an
FP8 FlashAttention as the fastest of its comparison and gives no formula.
The reading written here (and in the library's header):

* e4m3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; normals
  (1 + m/8) 2^(e-7) for e = 1..15 (e = 15, m = 7 is NaN, so the largest
  finite value is 448), subnormals (m/8) 2^-6.  Conversion rounds to the
  nearest value, ties to even, and saturates at +-448.
* Per-tile quantisation of a [rows][d] head slice: tile t = rows
  [128 t, 128 t + 128); scale s_t = amax_t / 448 and its reciprocal
  r_t = 448 / amax_t, each one float32 division (both 1 when the tile is all
  zero); code = e4m3(x * r_t) with the product in float32.  (The page gives
  no formula; a reciprocal computed once per tile and multiplied in is the
  plainest reading that costs one division per tile, not one per element.)
* Attention on codes and scales, one query row i at a time, over the k-tiles
  in ascending order (a streaming pass, as FlashAttention-2 computes it:
  FlashAttention-2 page, «Блочная обработка сохраняет общую нормализацию»):
      s_ij = scale * sq_t(i) * sk_t(j) * (q8_i . k8_j),   c_ij = s_ij log2 e
  The row keeps an integral reference exponent M (from -inf), a sum l and an
  accumulator a.  For tile t with maximum m_t of c over its visible keys: if
  m_t > M + 8, M moves to ceil(m_t) and l, a are multiplied by 2^(M_old -
  M_new) (0 from -inf).  Then, for the tile's visible keys,
      p_ij = 2^(c_ij - M),  l += sum p_ij,  a += sum e4m3(p_ij r_t) v8_j,
  with r_t = sv_t / sv_head (sv_head = max_t sv_t).  Finally
      o_i = sv_head a / l,   lse_i = (M + log2 l) ln 2.
  Rows that see no key: o = 0, lse = -inf.  P is rounded after the V tile's
  scale ratio is folded into it, so P8 V8 needs one scale per head.  The
  reference exponent is part of the definition: e4m3 rounding commutes with
  power-of-two scaling only outside its subnormal range, which small P r_t
  reach.
"""
from __future__ import annotations

import numpy as np

from .masks import dense_mask

E4M3_MAX = 448.0
TILE = 128


def e4m3(x) -> np.ndarray:
    """Nearest e4m3 value (ties to even), saturating at +-448; float64 out."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))          # a = m 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)                          # binade; subnormals share 2^-6's
    q = np.ldexp(1.0, (e - 3).astype(np.int64))         # spacing of 3 mantissa bits there
    r = np.round(a / q) * q                             # exact quotient; half to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(a > 0, np.sign(x) * r, 0.0)


def quantize_tiles(x) -> tuple[np.ndarray, np.ndarray]:
    """Codes (as float64 values) and float32 scales of a [rows][d] slice,
    per 128-row tile (the last tile may be short)."""
    x32 = np.asarray(x, dtype=np.float32)
    rows = x32.shape[0]
    nt = -(-rows // TILE)
    codes = np.zeros(x32.shape, dtype=np.float64)
    scales = np.ones(nt, dtype=np.float32)
    for t in range(nt):
        blk = x32[t * TILE:(t + 1) * TILE]
        amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
        s = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1)
        r = np.float32(np.float32(E4M3_MAX) / amax) if amax > 0 else np.float32(1)
        scales[t] = s
        codes[t * TILE:(t + 1) * TILE] = e4m3((blk * r).astype(np.float32))
    return codes, scales


def forward_head_fp8(q8, sq, k8, sk, v8, sv, mvec, scale, rows=None):
    """O rows and LSE of one head from codes and per-tile scales (see the
    module docstring); q8 [Sq][d], k8 and v8 [Skv][d] as float64 values."""
    Sq, Skv = q8.shape[0], k8.shape[0]
    rows = np.arange(Sq) if rows is None else np.asarray(rows)
    hidden = dense_mask(*mvec, Sq, rows=rows)               # [len(rows)][Skv]
    svh = float(np.max(sv))
    qs = np.asarray(sq, np.float64)[rows // TILE]
    ks = np.asarray(sk, np.float64)[np.arange(Skv) // TILE]
    c = (q8[rows] @ k8.T) * qs[:, None] * ks[None, :] * scale * np.log2(np.e)
    c = np.where(hidden, -np.inf, c)
    n = len(rows)
    M = np.full(n, -np.inf)
    l = np.zeros(n)
    a = np.zeros((n, v8.shape[1]))
    for t in range(-(-Skv // TILE)):
        cols = slice(t * TILE, min(Skv, (t + 1) * TILE))
        ct = c[:, cols]
        mt = ct.max(axis=1)
        grow = mt > M + 8
        Mn = np.where(grow, np.ceil(np.where(grow, mt, 0.0)), M)
        finite = np.isfinite(M)
        alpha = np.where(grow & finite, np.exp2(np.where(finite, M, 0.0) - Mn), 0.0)
        alpha = np.where(grow, alpha, 1.0)
        l *= alpha
        a *= alpha[:, None]
        M = Mn
        live = np.isfinite(M)
        p = np.where(live[:, None], np.exp2(ct - np.where(live, M, 0.0)[:, None]), 0.0)
        l += p.sum(axis=1)
        a += e4m3(p * (float(sv[t]) / svh)) @ v8[cols]
    dead = ~np.isfinite(M)
    o = svh * a / np.where(dead, 1.0, l)[:, None]
    o[dead] = 0.0
    lse = np.where(dead, -np.inf, (np.where(dead, 0.0, M) + np.log2(np.where(dead, 1.0, l)))
                   * np.log(2.0))
    return o, lse


"""Attention-side oracle: exact masked scaled-dot-product attention and its
gradients in float64.  Test infrastructure only (see ``oracle/__init__.py``).

The method is exact attention computed faster (FlashAttention-2 page,
«Блочная обработка сохраняет общую нормализацию»: streaming softmax with
rescaling keeps the normalisation over the whole row and the result is exact
attention; outputs and gradients differ only by floating-point order).  So the
oracle is the plain definition, one (batch, head) at a time:

  s_ij = scale * q_i . k_j                    for visible (i, j)
  lse_i = log sum_j exp(s_ij)                 (natural log; -inf if row i sees nothing)
  p_ij = exp(s_ij - lse_i)                    (0 for hidden entries, 0 on a row that sees nothing)
  o_i = sum_j p_ij v_j
  dV_j = sum_i p_ij dO_i,  dP_ij = dO_i . v_j,  D_i = sum_j p_ij dP_ij
  dS_ij = p_ij (dP_ij - D_i),  dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i

Tensors are BSHD ([batch][seq][head][d]) float64 arrays holding the bf16
values exactly; bounds are [4][B][Hm][Skv] (head h uses mask head 0 when
Hm == 1, else h).

Grouped-query attention (the ROCm page lists GQA among the key features of
current attention kernels; it gives no formula): K and V may have Hkv heads
with H = G * Hkv query heads; query head h attends with K/V head h // G
(consecutive query heads share one K/V head), and, since a shared head enters
G per-query-head losses, its gradients dK and dV are the sums of the G
per-head gradients (chain rule).  Hkv = H is ordinary multi-head attention.  Rows are independent: ``slice_rows`` only bounds the size of
the dense score block held at once; with it the row sums in dK and dV are
accumulated one row group after another.
"""
from __future__ import annotations

import numpy as np

from .masks import dense_mask


def to64(t) -> np.ndarray:
    """A torch tensor or array as float64 numpy (exact for bf16 inputs)."""
    if hasattr(t, "detach"):
        t = t.detach().to("cpu").float().numpy()
    return np.asarray(t, dtype=np.float64)


def _mask_vectors(bounds, b, h):
    bounds = np.asarray(bounds)
    Hm = bounds.shape[2]
    hm = 0 if Hm == 1 else h
    return tuple(bounds[t, b, hm] for t in range(4))


def columns_seen(mvec, r0: int, r1: int) -> np.ndarray:
    """Indices of the key columns that at least one query row of [r0, r1)
    sees.  A column is dropped only when its two hidden intervals together
    cover all of [r0, r1); such a column contributes exactly zero to every
    sum of the definition for those rows, so leaving it out changes nothing."""
    lts, lte, uts, ute = (np.asarray(x, dtype=np.int64) for x in mvec)
    if r0 >= r1:
        return np.zeros(0, dtype=np.int64)
    a_cov = (lts <= r0) & (lte >= r1)
    b_cov = (uts <= r0) & (ute >= r1)
    a_ne = lts < lte
    b_ne = uts < ute
    touch = a_ne & b_ne & (np.maximum(lts, uts) <= np.minimum(lte, ute))
    union_cov = touch & (np.minimum(lts, uts) <= r0) & (np.maximum(lte, ute) >= r1)
    return np.nonzero(~(a_cov | b_cov | union_cov))[0]


def probabilities_head(q, k, mvec, scale, rows=None, cols=None):
    """Scores, lse and probabilities for one head; q [Sq][d], k [Skv][d].
    Returns (p [R][len(cols)], lse [R]) for the selected rows (default all)
    over the selected key columns (default all; pass ``columns_seen`` to skip
    columns the rows cannot see)."""
    Sq = q.shape[0]
    rows = np.arange(Sq) if rows is None else np.asarray(rows)
    cols = np.arange(k.shape[0]) if cols is None else np.asarray(cols)
    if len(cols) == 0:                           # no row of the group sees any key
        return np.zeros((len(rows), 0)), np.full(len(rows), -np.inf)
    M = dense_mask(*(np.asarray(x)[cols] for x in mvec), Sq, rows=rows)
    s = scale * (q[rows] @ k[cols].T)
    s = np.where(M, -np.inf, s)
    m = s.max(axis=1)
    dead = ~np.isfinite(m)                       # the row sees no key at all
    m0 = np.where(dead, 0.0, m)
    with np.errstate(divide="ignore"):
        lse = np.where(dead, -np.inf, m0 + np.log(np.exp(s - m0[:, None]).sum(axis=1)))
    p = np.where(dead[:, None], 0.0, np.exp(s - np.where(dead, 0.0, lse)[:, None]))
    return p, lse


def forward_head(q, k, v, mvec, scale, rows=None, slice_rows=None, skip_hidden=False):
    """O rows and LSE for one head (fully hidden row: o = 0, lse = -inf).
    With ``skip_hidden`` each row group only touches ``columns_seen``."""
    Sq = q.shape[0]
    rows = np.arange(Sq) if rows is None else np.asarray(rows)
    step = len(rows) if not slice_rows else slice_rows
    o = np.zeros((len(rows), v.shape[1]))
    lse = np.zeros(len(rows))
    for a in range(0, len(rows), max(step, 1)):
        r = rows[a:a + step]
        cols = columns_seen(mvec, int(r.min()), int(r.max()) + 1) if skip_hidden and len(r) else None
        p, l = probabilities_head(q, k, mvec, scale, rows=r, cols=cols)
        o[a:a + len(r)] = p @ (v if cols is None else v[cols])
        lse[a:a + len(r)] = l
    return o, lse


def backward_head(q, k, v, do, mvec, scale, slice_rows=None, skip_hidden=False):
    """dQ, dK, dV (and O, LSE, D) for one head, from the definitions above.
    With ``skip_hidden`` each row group only touches ``columns_seen``."""
    Sq, Skv = q.shape[0], k.shape[0]
    step = Sq if not slice_rows else slice_rows
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.zeros((Sq, v.shape[1]))
    lse = np.zeros(Sq)
    D = np.zeros(Sq)
    for a in range(0, Sq, max(step, 1)):
        r = np.arange(a, min(Sq, a + step))
        cols = columns_seen(mvec, a, int(r[-1]) + 1) if skip_hidden else np.arange(Skv)
        kc, vc = k[cols], v[cols]
        p, l = probabilities_head(q, k, mvec, scale, rows=r, cols=cols)
        o[r] = p @ vc
        lse[r] = l
        dP = do[r] @ vc.T
        Dr = (p * dP).sum(axis=1)
        dS = p * (dP - Dr[:, None])
        dq[r] = scale * (dS @ kc)
        dk[cols] += scale * (dS.T @ q[r])
        dv[cols] += p.T @ do[r]
        D[r] = Dr
    return dq, dk, dv, o, lse, D


def kv_head(h: int, H: int, Hkv: int) -> int:
    """The K/V head query head h reads: h // G with G = H / Hkv."""
    if Hkv < 1 or H % Hkv:
        raise ValueError("the K/V head count must divide the query head count")
    return h // (H // Hkv)


def forward(q, k, v, bounds, scale, slice_rows=None):
    """O [B][Sq][H][d] and LSE [B][H][Sq] for BSHD float64 inputs (k, v may
    have fewer heads than q: grouped-query attention)."""
    B, Sq, H, d = q.shape
    Hkv = k.shape[2]
    o = np.zeros((B, Sq, H, v.shape[3]))
    lse = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, Hkv)
            ob, lb = forward_head(q[b, :, h], k[b, :, hk], v[b, :, hk],
                                  _mask_vectors(bounds, b, h), scale, slice_rows=slice_rows)
            o[b, :, h] = ob
            lse[b, h] = lb
    return o, lse


def backward(q, k, v, do, bounds, scale, slice_rows=None):
    """(dq, dk, dv, o, lse, D) for BSHD float64 inputs; D is [B][H][Sq].  With
    fewer K/V heads than query heads, dk and dv of a K/V head sum over the
    query heads that read it."""
    B, Sq, H, d = q.shape
    Hkv = k.shape[2]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    o = np.zeros((B, Sq, H, v.shape[3]))
    lse = np.zeros((B, H, Sq))
    D = np.zeros((B, H, Sq))
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, Hkv)
            r = backward_head(q[b, :, h], k[b, :, hk], v[b, :, hk], do[b, :, h],
                              _mask_vectors(bounds, b, h), scale, slice_rows=slice_rows)
            dq[b, :, h], gk, gv, o[b, :, h], lse[b, h], D[b, h] = r
            dk[b, :, hk] += gk
            dv[b, :, hk] += gv
    return dq, dk, dv, o, lse, D

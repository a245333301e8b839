"""Shared parity helpers: run the CUDA path through the binding and compare
with the oracle on the same seeded inputs.

Tolerances (written here once, used by every parity test):
  O:     max (|O - O_ref| - u(O_ref)) <= 1e-2, u(x) = half a bf16 ulp at |x|:
         the 1e-2 budget is for the computation, and the rounding to the bf16
         output (up to 2^-7 for |O_ref| in [2, 4)) comes on top of it
  LSE:   max |LSE - LSE_ref| <= 1e-3 on rows that see a key, exactly -inf otherwise
  grads: max |G - G_ref| <= 2e-2 * max(max |G_ref|, 1e-4)
         (the floor only matters when the reference gradient is identically
         zero, e.g. a row that sees a single key: D is formed from the bf16
         output, so dP - D is a rounding residual instead of an exact 0)
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention as oa
from rounding_model import bf16_half_ulp

O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_REL = 2e-2
GRAD_FLOOR = 1e-4


def o_excess(got, ref):
    """|O - O_ref| beyond the unavoidable rounding of O_ref to bf16, elementwise."""
    return np.abs(got - ref) - bf16_half_ulp(ref)


def head_slice(t, b, h):
    """One (batch, head) slice of a BSHD tensor as float64 numpy."""
    return oa.to64(t[b, :, h])


def mask_vec(bounds, b, h):
    bnd = bounds.detach().cpu().numpy()
    Hm = bnd.shape[2]
    hm = 0 if Hm == 1 else h
    return tuple(bnd[t, b, hm] for t in range(4))


def sample_rows(Sq, n, seed):
    if n is None or n >= Sq:
        return np.arange(Sq)
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(Sq, size=n, replace=False).tolist())
    rows.update({0, Sq - 1, min(Sq - 1, 127), min(Sq - 1, 128)})
    return np.array(sorted(rows))


def compare_fwd(q, k, v, bounds, scale, o, lse, heads=None, rows=None, seed=0, slice_rows=4096):
    """Check O and LSE of the given (b, h) pairs (default all) on ``rows``
    sampled query rows per head (default all).  Returns the worst errors."""
    B, Sq, H, _ = q.shape
    Hkv = k.shape[2]
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    worst_o = worst_l = 0.0
    for n, (b, h) in enumerate(heads):
        r = sample_rows(Sq, rows, seed + n)
        hk = oa.kv_head(h, H, Hkv)
        ro, rl = oa.forward_head(head_slice(q, b, h), head_slice(k, b, hk), head_slice(v, b, hk),
                                 mask_vec(bounds, b, h), scale, rows=r, slice_rows=slice_rows,
                                 skip_hidden=True)
        go = o[b, r, h].float().cpu().numpy()
        gl = lse[b, h, r].cpu().numpy().astype(np.float64)
        eo = float(o_excess(go, ro).max()) if len(r) else 0.0
        dead = np.isneginf(rl)
        assert np.array_equal(np.isneginf(gl), dead), f"-inf LSE rows differ at (b={b}, h={h})"
        el = float(np.abs(gl[~dead] - rl[~dead]).max()) if (~dead).any() else 0.0
        assert np.all(go[dead] == 0), "rows that see no key must have O = 0"
        worst_o, worst_l = max(worst_o, eo), max(worst_l, el)
        assert eo <= O_TOL, f"O error {eo} beyond the bf16 output rounding at (b={b}, h={h})"
        assert el <= LSE_TOL, f"LSE error {el} at (b={b}, h={h})"
    return worst_o, worst_l


def compare_bwd(q, k, v, do, bounds, scale, dq, dk, dv, heads=None, slice_rows=1024):
    """Check dQ of the given (b, h) query-head pairs (default all), and dK, dV
    of the K/V heads they read, in full against the oracle.  With fewer K/V
    heads than query heads, a K/V head's reference gradients sum over all the
    query heads that read it (oracle.attention, grouped-query attention)."""
    B, Sq, H, _ = q.shape
    Hkv = k.shape[2]
    G = H // Hkv
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    worst = {"dq": 0.0, "dk": 0.0, "dv": 0.0}

    def check(name, g, ref, b, h):
        err = float(np.abs(g - ref).max())
        scale_ref = float(np.abs(ref).max())
        rel = err / scale_ref if scale_ref > 0 else err
        worst[name] = max(worst[name], rel)
        assert err <= GRAD_REL * max(scale_ref, GRAD_FLOOR), \
            f"{name} error {err} vs max|ref| {scale_ref} at (b={b}, head={h})"

    for b, hk in sorted({(b, oa.kv_head(h, H, Hkv)) for b, h in heads}):
        sk = sv = 0.0
        for h in range(hk * G, hk * G + G):
            rq, rk, rv, *_ = oa.backward_head(head_slice(q, b, h), head_slice(k, b, hk),
                                              head_slice(v, b, hk), head_slice(do, b, h),
                                              mask_vec(bounds, b, h), scale, slice_rows=slice_rows,
                                              skip_hidden=True)
            if (b, h) in heads:
                check("dq", dq[b, :, h].float().cpu().numpy(), rq, b, h)
            sk, sv = sk + rk, sv + rv
        check("dk", dk[b, :, hk].float().cpu().numpy(), sk, b, hk)
        check("dv", dv[b, :, hk].float().cpu().numpy(), sv, b, hk)
    return worst

"""Pins for the attention side of the oracle (no GPU).

The oracle is checked against: torch's own scaled_dot_product_attention in
float64 (a library special case: no mask, causal, boolean masks), scipy's
logsumexp, central finite differences of the loss sum(O * dO), the identity
D_i = dO_i . o_i, a permutation invariance, row-sum and fully-masked-row
invariants, and a planted mistake (per-tile normalisation) that must fail the
output tolerance.
"""
import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from fm_inputs import masks as gen
from fm_inputs.configs import TINY, TINY_DOCS
from fm_inputs.tensors import qkv_do
from oracle import attention as oa
from oracle import masks as om


def _bounds(b):
    return np.stack([np.asarray(x)[None, None] for x in b])  # [4][1][1][S]


def _rand(S, d, seed, Skv=None):
    rng = np.random.default_rng(seed)
    Skv = S if Skv is None else Skv
    q = rng.standard_normal((1, S, 1, d))
    k = rng.standard_normal((1, Skv, 1, d))
    v = rng.standard_normal((1, Skv, 1, d))
    do = rng.standard_normal((1, S, 1, d))
    return q, k, v, do


def _sdpa(q, k, v, scale, visible=None, causal=False):
    qt = torch.from_numpy(q[0].transpose(1, 0, 2).copy())  # [H][S][d]
    kt = torch.from_numpy(k[0].transpose(1, 0, 2).copy())
    vt = torch.from_numpy(v[0].transpose(1, 0, 2).copy())
    m = None if visible is None else torch.from_numpy(visible)
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, is_causal=causal, scale=scale)
    return o.numpy().transpose(1, 0, 2)[None]


def test_unmasked_equals_sdpa():
    S, d = 96, 16
    q, k, v, _ = _rand(S, d, 0)
    o, lse = oa.forward(q, k, v, _bounds(gen.full(S)), 0.3)
    assert np.abs(o - _sdpa(q, k, v, 0.3)).max() < 1e-12
    s = 0.3 * q[0, :, 0] @ k[0, :, 0].T
    assert np.abs(lse[0, 0] - scipy.special.logsumexp(s, axis=1)).max() < 1e-12


def test_causal_equals_sdpa():
    S, d = 128, 8
    q, k, v, _ = _rand(S, d, 1)
    o, _ = oa.forward(q, k, v, _bounds(gen.causal(S)), d ** -0.5)
    assert np.abs(o - _sdpa(q, k, v, d ** -0.5, causal=True)).max() < 1e-12


@pytest.mark.parametrize("name", ["causal_document", "share_question", "sliding_window",
                                  "global_sliding", "prefix_document", "random_eviction"])
def test_masked_equals_sdpa_with_boolean_mask(name):
    S, d = 192, 16
    q, k, v, _ = _rand(S, d, 2)
    b = gen.make_mask(name, S, seed=3, window=40, n_global=4) if name in ("sliding_window", "global_sliding") \
        else gen.make_mask(name, S, seed=3)
    vis = ~om.dense_mask(*b, S)
    assert vis.any(axis=1).all()
    o, _ = oa.forward(q, k, v, _bounds(b), 0.25)
    assert np.abs(o - _sdpa(q, k, v, 0.25, visible=vis)).max() < 1e-12


def test_rows_sum_to_one_and_dead_rows():
    S, d = 256, 8
    q, k, v, _ = _rand(S, d, 4)
    b = gen.qk_sparse(S)
    p, lse = oa.probabilities_head(q[0, :, 0], k[0, :, 0], b, 0.5)
    vis = ~om.dense_mask(*b, S)
    live = vis.any(axis=1)
    assert (~live).sum() == S // 16                      # the dropped query rows
    assert np.abs(p[live].sum(axis=1) - 1).max() < 1e-12
    assert np.all(p[~vis] == 0)
    o, lse = oa.forward(q, k, v, _bounds(b), 0.5)
    assert np.all(o[0, ~live] == 0)
    assert np.all(np.isneginf(lse[0, 0, ~live]))
    dq, dk, dv, *_ = oa.backward(q, k, v, _rand(S, d, 5)[3], _bounds(b), 0.5)
    assert np.all(dq[0, ~live] == 0)
    dead_cols = ~vis.any(axis=0)
    assert dead_cols.sum() == S // 16
    assert np.all(dk[0, dead_cols] == 0) and np.all(dv[0, dead_cols] == 0)


@pytest.mark.parametrize("name", ["causal_document", "qk_sparse", "full"])
def test_gradients_by_finite_differences(name):
    S, d, scale = 32, 8, 0.7
    q, k, v, do = _rand(S, d, 6)
    b = _bounds(gen.causal_document(S, [9, 14, 9]) if name == "causal_document" else gen.make_mask(name, S))
    dq, dk, dv, *_ = oa.backward(q, k, v, do, b, scale)

    def loss(qq, kk, vv):
        o, _ = oa.forward(qq, kk, vv, b, scale)
        return float((o * do).sum())

    eps = 1e-6
    for X, G, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = Xp, Xm
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        rel = np.abs(num - G).max() / max(np.abs(G).max(), 1e-30)
        assert rel < 1e-6, (which, rel)


def test_D_two_ways():
    S, d = 200, 16
    q, k, v, do = _rand(S, d, 7)
    b = _bounds(gen.make_mask("share_question", S, seed=0))
    *_, o, lse, D = oa.backward(q, k, v, do, b, 0.25)
    assert np.abs(D[0, 0] - (do[0, :, 0] * o[0, :, 0]).sum(axis=1)).max() < 1e-12


def test_key_permutation_invariance():
    S, d = 160, 8
    q, k, v, do = _rand(S, d, 8)
    b = _bounds(gen.make_mask("random_eviction", S, seed=1))
    perm = np.random.default_rng(0).permutation(S)
    r0 = oa.backward(q, k, v, do, b, 0.4)
    r1 = oa.backward(q, k[:, perm], v[:, perm], do, b[..., perm], 0.4)
    assert np.abs(r0[0] - r1[0]).max() < 1e-12                # dq
    assert np.abs(r0[1][:, perm] - r1[1]).max() < 1e-12       # dk permuted
    assert np.abs(r0[2][:, perm] - r1[2]).max() < 1e-12       # dv permuted
    assert np.abs(r0[3] - r1[3]).max() < 1e-12                # o


def test_slice_rows_changes_nothing():
    S, d = 300, 8
    q, k, v, do = _rand(S, d, 9)
    b = _bounds(gen.make_mask("causal_document", S, seed=2))
    a = oa.backward(q, k, v, do, b, 0.3)
    c = oa.backward(q, k, v, do, b, 0.3, slice_rows=37)
    for x, y in zip(a, c):
        assert np.allclose(x, y, rtol=0, atol=1e-12, equal_nan=True)


def test_per_tile_normalisation_fails_tolerance():
    """Normalising each key tile on its own and adding the pieces is not
    attention (FlashAttention-2 page, «Блочная обработка сохраняет общую
    нормализацию»); such a mistake must break the 1e-2 output tolerance on the
    tiny workload, which shows the tolerance discriminates."""
    q, k, v, _ = qkv_do(TINY.B, TINY.S, TINY.S, TINY.H, TINY.d, seed=0)
    q, k, v = oa.to64(q), oa.to64(k), oa.to64(v)
    b = _bounds(gen.causal_document(TINY.S, TINY_DOCS))
    o, _ = oa.forward(q, k, v, b, TINY.scale)
    bad = np.zeros_like(o)
    for h in range(TINY.H):
        M = om.dense_mask(*(b[t, 0, 0] for t in range(4)), TINY.S)
        s = TINY.scale * q[0, :, h] @ k[0, :, h].T
        s = np.where(M, -np.inf, s)
        for kj in range(2):
            c = slice(kj * 128, kj * 128 + 128)
            blk = s[:, c]
            m = blk.max(axis=1, keepdims=True)
            ok = np.isfinite(m[:, 0])
            e = np.where(ok[:, None], np.exp(blk - np.where(ok[:, None], m, 0)), 0)
            z = e.sum(axis=1, keepdims=True)
            bad[0, :, h] += np.where(ok[:, None], e / np.where(z == 0, 1, z), 0) @ v[0, c, h]
    assert np.abs(bad - o).max() > 1e-2


@pytest.mark.parametrize("name", ["causal_document", "qk_sparse", "global_sliding", "random_eviction",
                                  "share_question", "block_sparse", "causal_blockwise"])
def test_skip_hidden_columns_changes_nothing(name):
    """Leaving out the columns a row group cannot see is exact: compare with
    the plain dense path (and check the skipped columns really are hidden)."""
    S, d = 700, 8
    q, k, v, do = _rand(S, d, 10)
    b = gen.make_mask(name, S, seed=3, window=50, n_global=3) if name == "global_sliding" \
        else gen.make_mask(name, S, seed=3)
    M = om.dense_mask(*b, S)
    for r0, r1 in ((0, 64), (100, 228), (640, 700), (333, 334)):
        seen = oa.columns_seen(b, r0, r1)
        hidden = np.setdiff1d(np.arange(S), seen)
        assert M[r0:r1][:, hidden].all()
        assert not M[r0:r1][:, seen].all(axis=0).any()
    a = oa.backward_head(q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0], b, 0.3, slice_rows=64)
    c = oa.backward_head(q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0], b, 0.3, slice_rows=64,
                         skip_hidden=True)
    for x, y in zip(a, c):
        assert np.allclose(x, y, rtol=0, atol=1e-12, equal_nan=True)
    fo = oa.forward_head(q[0, :, 0], k[0, :, 0], v[0, :, 0], b, 0.3, slice_rows=50, skip_hidden=True)
    assert np.allclose(fo[0], a[3], rtol=0, atol=1e-12)


def _gqa_inputs(S, H, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, S, H, d))
    k = rng.standard_normal((1, S, Hkv, d))
    v = rng.standard_normal((1, S, Hkv, d))
    do = rng.standard_normal((1, S, H, d))
    # a different mask per query head, so a wrong mask-head mapping shows too
    names = ["causal", "sliding_window", "full", "prefix_lm", "causal", "full"]
    b = np.stack([np.stack([np.asarray(x) for x in gen.make_mask(names[h % len(names)], S)])
                  for h in range(H)], axis=1)[:, None]  # [4][1][H][S]
    return q, k, v, do, b


def test_gqa_equals_mha_with_repeated_kv():
    """Grouped-query attention equals multi-head attention on K/V repeated so
    that query head h sees copy h // G (consecutive query heads share a K/V
    head); dQ agrees, and a K/V head's dK, dV are the sums of its copies'."""
    S, H, Hkv, d, scale = 48, 6, 2, 8, 0.5
    G = H // Hkv
    q, k, v, do, b = _gqa_inputs(S, H, Hkv, d, 11)
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    o_g, l_g = oa.forward(q, k, v, b, scale)
    o_m, l_m = oa.forward(q, kr, vr, b, scale)
    assert np.allclose(o_g, o_m, rtol=0, atol=1e-13) and np.allclose(l_g, l_m, rtol=0, atol=1e-13)
    dq_g, dk_g, dv_g, *_ = oa.backward(q, k, v, do, b, scale)
    dq_m, dk_m, dv_m, *_ = oa.backward(q, kr, vr, do, b, scale)
    assert np.allclose(dq_g, dq_m, rtol=0, atol=1e-12)
    assert np.allclose(dk_g, dk_m.reshape(1, S, Hkv, G, d).sum(axis=3), rtol=0, atol=1e-12)
    assert np.allclose(dv_g, dv_m.reshape(1, S, Hkv, G, d).sum(axis=3), rtol=0, atol=1e-12)
    # the other plausible mapping (h % Hkv) differs on this input
    kw = np.concatenate([k] * G, axis=2)
    o_w, _ = oa.forward(q, kw, np.concatenate([v] * G, axis=2), b, scale)
    assert not np.allclose(o_g, o_w, atol=1e-6)


def test_gqa_gradients_by_finite_differences():
    """dK and dV of shared K/V heads against central differences of
    sum(O * dO): independent of the group-sum rule."""
    S, H, Hkv, d, scale = 16, 4, 2, 4, 0.6
    q, k, v, do, b = _gqa_inputs(S, H, Hkv, d, 12)
    _, dk, dv, *_ = oa.backward(q, k, v, do, b, scale)

    def loss(kk, vv):
        o, _ = oa.forward(q, kk, vv, b, scale)
        return float((o * do).sum())

    eps = 1e-6
    for X, Gr, which in ((k, dk, 0), (v, dv, 1)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            num[idx] = ((loss(Xp, v) - loss(Xm, v)) if which == 0 else
                        (loss(k, Xp) - loss(k, Xm))) / (2 * eps)
        rel = np.abs(num - Gr).max() / np.abs(Gr).max()
        assert rel < 1e-6, (which, rel)

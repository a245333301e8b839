"""Mask-analysis kernels against the oracle, bit for bit (GPU).

Block summary + tile classification + work lists (per q-tile row, per
q-tile pair, per k-tile column) + longest-first orders (forward pairs, dK/dV
columns, dQ rows) + the partial tiles' visibility bit masks (fm_plan), bound
validation, and localisation (fm_localize).
"""
import numpy as np
import pytest
import torch

import masked_attention_bound_gb300 as fm
from fm_inputs import masks as gen
from fm_inputs.configs import TINY_DOCS, dual_chunk_map
from fm_inputs.tensors import bounds_tensor, mask_bounds
from oracle import masks as om

pytestmark = pytest.mark.gpu


def _bounds_from(b_list, Hm=1):
    return bounds_tensor([[b] * Hm for b in b_list], device="cuda")


def _ws_view(ws, off, n, dtype):
    itemsize = torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + n * itemsize].view(dtype)


def _check_tile_masks(ws, L, bounds, Sq, ref_rl, sample=40, seed=0):
    """The forward plan's visibility bit masks: every row with partial tiles
    (class PARTIAL, or the ragged last k-tile) owns consecutive slots, one per
    such tile in list order, disjoint from other rows' and inside the region
    (rows may go without when the region is full); sampled tiles match the
    oracle's dense mask bit for bit (rows below Sq; columns past Skv set)."""
    _, B, Hm, Skv = bounds.shape
    nQ, nK = -(-Sq // 128), -(-Skv // 128)
    cap = (L.total - L.masks) // 2048
    rowm = _ws_view(ws, L.row_mask, B * Hm * nQ, torch.int32).view(B, Hm, nQ).cpu().numpy()
    ragged = Skv % 128 != 0
    parts = {}
    for key, ent in ref_rl.items():
        p = [kj for kj, c in ent if c == 1 or (ragged and kj == nK - 1)]
        if p:
            parts[key] = p
    for b in range(B):
        for hm in range(Hm):
            for qi in range(nQ):
                if (b, hm, qi) not in parts:
                    assert rowm[b, hm, qi] == -1
    spans = sorted((int(rowm[key]), len(p)) for key, p in parts.items() if rowm[key] >= 0)
    for (f0, n0), (f1, _) in zip(spans, spans[1:]):
        assert f0 + n0 <= f1
    if spans:
        assert spans[0][0] >= 0 and spans[-1][0] + spans[-1][1] <= cap
    if sum(len(p) for p in parts.values()) <= cap:
        assert len(spans) == len(parts)
    owned = [(key, o) for key, p in parts.items() if rowm[key] >= 0 for o in range(len(p))]
    if not owned:
        return
    words = _ws_view(ws, L.masks, cap * 512, torch.int32).cpu().numpy().view(np.uint32).reshape(cap, 128, 4)
    bnp = bounds.cpu().numpy()
    rng = np.random.default_rng(seed)
    pick = rng.choice(len(owned), size=min(sample, len(owned)), replace=False)
    shifts = np.arange(32, dtype=np.uint32)
    for n in pick:
        (b, hm, qi), o = owned[n]
        kj = parts[(b, hm, qi)][o]
        got = ((words[rowm[b, hm, qi] + o][:, :, None] >> shifts) & 1).reshape(128, 128).astype(bool)
        rows = np.arange(qi * 128, min(qi * 128 + 128, Sq))
        cols = np.arange(kj * 128, kj * 128 + 128)
        want = np.ones((len(rows), 128), dtype=bool)
        live = cols < Skv
        want[:, live] = om.dense_mask(*(bnp[t, b, hm, cols[live]] for t in range(4)), Sq, rows=rows)
        assert np.array_equal(got[:len(rows)], want), ((b, hm, qi), kj)


def _check_plan(bounds, Sq, H=2, d=64):
    _, B, Hm, Skv = bounds.shape
    q = torch.empty(B, Sq, H, d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(B, Skv, H, d, dtype=torch.bfloat16, device="cuda")
    nQ, nK = -(-Sq // 128), -(-Skv // 128)
    ref_table = om.tile_table(bounds.cpu().numpy(), Sq)
    ref_rc, ref_rl = om.row_lists(ref_table)
    ref_cc, ref_cl = om.col_lists(ref_table)
    for for_bwd in (False, True):
        ws, L = fm.plan(q, k, bounds, for_bwd=for_bwd)
        torch.cuda.synchronize()
        assert fm.device_status(ws) == 0
        table = _ws_view(ws, L.table, B * Hm * nQ * nK, torch.uint8).view(B, Hm, nQ, nK).cpu().numpy()
        assert np.array_equal(table, ref_table)
        # q-tile rows and their partial tiles' bit masks: the forward builds
        # its pairs from them, the backward's dQ pass walks them
        cnt = _ws_view(ws, L.row_count, B * Hm * nQ, torch.int32).view(B, Hm, nQ).cpu().numpy()
        lst = _ws_view(ws, L.row_list, B * Hm * nQ * nK, torch.int32).view(B, Hm, nQ, nK).cpu().numpy()
        assert np.array_equal(cnt, ref_rc)
        for (b, hm, qi), ent in ref_rl.items():
            want = [(kj << 2) | c for kj, c in ent]
            assert lst[b, hm, qi, :len(want)].tolist() == want
        _check_tile_masks(ws, L, bounds, Sq, ref_rl)
        if not for_bwd:
            nP = (nQ + 1) // 2
            ref_pc, ref_cost, ref_pl = om.pair_lists(ref_table, Skv)
            info = _ws_view(ws, L.pair_info, B * Hm * nP * 4, torch.int32).view(B, Hm, nP, 4).cpu().numpy()
            plst = _ws_view(ws, L.pair_list, B * Hm * nP * nK, torch.int32).view(B, Hm, nP, nK).cpu().numpy()
            assert np.array_equal(info[..., 0], ref_pc)
            assert np.array_equal(info[..., 3], ref_cost)
            for (b, hm, p), ent in ref_pl.items():
                want = [(kj << 4) | (ca << 2) | cb for kj, ca, cb in ent]
                assert plst[b, hm, p, :len(want)].tolist() == want
                assert info[b, hm, p, 1] == sum(ca != 0 for _, ca, _ in ent)
                assert info[b, hm, p, 2] == sum(cb != 0 for _, _, cb in ent)
            order = _ws_view(ws, L.fwd_order, B * H * nP, torch.int32).cpu().numpy()
            assert np.array_equal(order, om.unit_order(ref_cost, H))
        else:
            cnt = _ws_view(ws, L.col_count, B * Hm * nK, torch.int32).view(B, Hm, nK).cpu().numpy()
            lst = _ws_view(ws, L.col_list, B * Hm * nK * nQ, torch.int32).view(B, Hm, nK, nQ).cpu().numpy()
            assert np.array_equal(cnt, ref_cc)
            for (b, hm, kj), ent in ref_cl.items():
                want = [(qi << 2) | c for qi, c in ent]
                assert lst[b, hm, kj, :len(want)].tolist() == want
            order = _ws_view(ws, L.bwd_order, B * H * nK, torch.int32).cpu().numpy()
            assert np.array_equal(order, om.unit_order(ref_cc, H))
            order = _ws_view(ws, L.row_order, B * H * nQ, torch.int32).cpu().numpy()
            assert np.array_equal(order, om.unit_order(ref_rc, H))


def test_plan_tiny():
    _check_plan(_bounds_from([gen.causal_document(256, TINY_DOCS)]), 256)


@pytest.mark.parametrize("name", ["full", "causal", "sliding_window", "causal_document", "prefix_lm"])
def test_plan_4k_masks(name):
    _check_plan(mask_bounds(name, 4, 4096, device="cuda"), 4096, H=16, d=128)


@pytest.mark.parametrize("name", gen.MASKS_32K)
def test_plan_32k_suite(name):
    _check_plan(mask_bounds(name, 1, 32768, device="cuda"), 32768, H=32, d=128)


def test_plan_128k():
    _check_plan(mask_bounds("causal_document_window", 1, 131072, device="cuda", window=8192),
                131072, H=8, d=128)


@pytest.mark.parametrize("S", [1, 100, 129, 300, 1000])
def test_plan_ragged(S):
    names = ["causal", "causal_document", "random_eviction", "qk_sparse", "global_sliding"]
    bl = [gen.make_mask(n, S, seed=i, window=max(1, S // 5), n_global=min(5, S)) for i, n in enumerate(names)]
    _check_plan(_bounds_from(bl), S, H=3)


def test_plan_per_head_masks():
    S, H = 700, 3
    per_b = [[gen.make_mask(n, S, seed=i) for i, n in enumerate(["causal", "share_question", "qk_sparse"])]]
    bounds = bounds_tensor(per_b, device="cuda")
    _check_plan(bounds, S, H=H)


def test_plan_cross_lengths():
    """Sq != Skv: random intervals inside [0, Sq]."""
    Sq, Skv = 300, 777
    rng = np.random.default_rng(1)
    a = rng.integers(0, Sq + 1, size=(4, Skv))
    lts, lte = np.minimum(a[0], a[1]), np.maximum(a[0], a[1])
    uts, ute = np.minimum(a[2], a[3]), np.maximum(a[2], a[3])
    bounds = bounds_tensor([[(lts, lte, uts, ute)]], device="cuda")
    _check_plan(bounds, Sq)


def test_bounds_out_of_range_reported():
    S = 256
    b = [x.copy() for x in gen.causal(S)]
    b[1][17] = S + 1
    bounds = _bounds_from([tuple(b)])
    q = torch.empty(1, S, 1, 64, dtype=torch.bfloat16, device="cuda")
    ws, _ = fm.plan(q, q, bounds)
    assert fm.device_status(ws) == 2  # FM_ERR_BOUNDS
    b[1][17] = -1
    ws, _ = fm.plan(q, q, _bounds_from([tuple(b)]))
    assert fm.device_status(ws) == 2
    ws, _ = fm.plan(q, q, _bounds_from([gen.causal(S)]))
    assert fm.device_status(ws) == 0


# ---------------------------------------------------------------- localisation

def test_localize_config_64k():
    S = 65536
    bounds = mask_bounds("causal_document", 1, S, device="cuda")
    ref_in = bounds.cpu().numpy()
    for chunks in dual_chunk_map(S, 4):
        got = fm.localize(bounds, chunks).cpu().numpy()
        assert np.array_equal(got, om.localize_bounds(ref_in, chunks))


@pytest.mark.parametrize("name", ["causal", "qk_sparse", "share_question", "random_eviction", "global_sliding"])
def test_localize_random_chunks(name):
    S = 3000
    rng = np.random.default_rng(4)
    bounds = bounds_tensor([[gen.make_mask(name, S, seed=1)] * 2] * 2, device="cuda")  # B=2, Hm=2
    ref_in = bounds.cpu().numpy()
    for _ in range(5):
        cuts = np.sort(rng.choice(np.arange(1, S), size=2 * int(rng.integers(1, 9)), replace=False))
        chunks = [(int(a), int(e - a)) for a, e in cuts.reshape(-1, 2)]
        got = fm.localize(bounds, chunks).cpu().numpy()
        assert np.array_equal(got, om.localize_bounds(ref_in, chunks))


def test_localize_rejects_bad_chunk_maps():
    bounds = _bounds_from([gen.causal(256)])
    for chunks in ([(128, 64), (0, 64)], [(0, 64), (32, 64)], [(0, 0)], [], [(-1, 4)]):
        with pytest.raises(fm.FMError) as e:
            fm.localize(bounds, chunks)
        assert e.value.code == 1

"""Grouped-query attention (K/V heads shared by groups of query heads) through
the C ABI against the oracle (GPU).

Query head h reads K/V head h // G (G = H / Hkv); a shared head's dK and dV
sum over its G query heads (oracle.attention).  Tolerances as in parity.py.
"""
import numpy as np
import pytest
import torch

import masked_attention_bound_gb300 as fm
from fm_inputs import masks as gen
from fm_inputs.configs import LONG_128K
from fm_inputs.tensors import bounds_tensor, mask_bounds, randn_bf16
from oracle import masks as om
from parity import compare_bwd, compare_fwd

pytestmark = pytest.mark.gpu


def _inputs(B, Sq, Skv, H, Hkv, d, seed):
    q = randn_bf16(B, Sq, H, d, seed=seed, device="cuda")
    k = randn_bf16(B, Skv, Hkv, d, seed=seed + 1, device="cuda")
    v = randn_bf16(B, Skv, Hkv, d, seed=seed + 2, device="cuda")
    do = randn_bf16(B, Sq, H, d, seed=seed + 3, device="cuda")
    return q, k, v, do


def _run(q, k, v, do, bounds, scale):
    o, lse = fm.forward(q, k, v, bounds, scale)
    dq, dk, dv = fm.backward(q, k, v, o, lse, do, bounds, scale)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [77, 1000])
@pytest.mark.parametrize("H,Hkv", [(4, 1), (4, 2), (6, 3)])
@pytest.mark.parametrize("name", ["causal_document", "share_question"])
def test_gqa_small_shapes(name, H, Hkv, S, d):
    q, k, v, do = _inputs(1, S, S, H, Hkv, d, seed=21)
    bounds = mask_bounds(name, 1, S, device="cuda")
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, d ** -0.5)
    compare_fwd(q, k, v, bounds, d ** -0.5, o, lse)
    compare_bwd(q, k, v, do, bounds, d ** -0.5, dq, dk, dv)


def test_gqa_per_head_masks_strides_and_cross_lengths():
    """Per-query-head masks (so the query heads of one K/V head see different
    keys), strided views, Sq != Skv, two batches."""
    B, Sq, Skv, H, Hkv, d = 2, 384, 640, 4, 2, 128
    base_q = randn_bf16(B, Sq, H, 2 * d, seed=31, device="cuda")
    base_kv = randn_bf16(B, Skv, Hkv, 2 * d, seed=32, device="cuda")
    q, do = base_q[..., :d], base_q[..., d:]
    k, v = base_kv[..., :d], base_kv[..., d:]
    rng = np.random.default_rng(5)
    per_b = []
    for _ in range(B):
        heads = []
        for _ in range(H):
            a = rng.integers(0, Sq + 1, size=(4, Skv))
            heads.append((np.minimum(a[0], a[1]), np.maximum(a[0], a[1]),
                          np.minimum(a[2], a[3]), np.maximum(a[2], a[3])))
        per_b.append(heads)
    bounds = bounds_tensor(per_b, device="cuda")
    o = torch.empty(B, Sq, H, 2 * d, device="cuda", dtype=torch.bfloat16)[..., :d]
    o, lse = fm.forward(q, k, v, bounds, 0.1, o=o)
    dq = torch.empty(B, Sq, H, 2 * d, device="cuda", dtype=torch.bfloat16)[..., d:]
    dk = torch.empty(B, Skv, Hkv, 2 * d, device="cuda", dtype=torch.bfloat16)[..., :d]
    dv = torch.empty(B, Skv, Hkv, 2 * d, device="cuda", dtype=torch.bfloat16)[..., d:]
    do_o = torch.empty(B, Sq, H, 2 * d, device="cuda", dtype=torch.bfloat16)[..., d:]
    do_o.copy_(do)  # dO must have O's strides
    fm.backward(q, k, v, o, lse, do_o, bounds, 0.1, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    compare_fwd(q, k, v, bounds, 0.1, o, lse)
    compare_bwd(q, k, v, do, bounds, 0.1, dq, dk, dv)


def test_gqa_equals_mha_on_repeated_kv():
    """On the GPU alone: O, LSE and dQ of grouped-query attention equal, bit
    for bit, multi-head attention on K/V repeated per query head (the same
    tiles meet the same operands); dK and dV equal the group sums of the
    multi-head gradients up to their bf16 rounding."""
    S, H, Hkv, d = 2 * 1024 + 77, 6, 2, 128
    G = H // Hkv
    q, k, v, do = _inputs(1, S, S, H, Hkv, d, seed=41)
    bounds = mask_bounds("causal_document", 1, S, device="cuda")
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, d ** -0.5)
    kr = k.repeat_interleave(G, dim=2).contiguous()
    vr = v.repeat_interleave(G, dim=2).contiguous()
    o2, lse2, dq2, dk2, dv2 = _run(q, kr, vr, do, bounds, d ** -0.5)
    assert torch.equal(o, o2) and torch.equal(lse, lse2) and torch.equal(dq, dq2)
    for g, m in ((dk, dk2), (dv, dv2)):
        ref = m.float().view(1, S, Hkv, G, d).sum(dim=3)
        err = (g.float() - ref).abs().max().item()
        assert err <= 2e-2 * ref.abs().max().item()


def test_gqa_long_128k_sampled_group():
    """The 128K workload with its 8 query heads over 4 K/V heads: query head 3
    and K/V head 1 (query heads 2 and 3) against the oracle."""
    W = LONG_128K
    Hkv = 4
    q, k, v, do = _inputs(W.B, W.S, W.S, W.H, Hkv, W.d, seed=51)
    bounds = mask_bounds("causal_document_window", W.B, W.S, device="cuda", window=8192)
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, W.scale)
    compare_fwd(q, k, v, bounds, W.scale, o, lse, heads=[(0, 3)], rows=64)
    compare_bwd(q, k, v, do, bounds, W.scale, dq, dk, dv, heads=[(0, 3)])


def test_gqa_plan_orders():
    """The backward's K/V-head units are ordered by the sum of their query
    heads' column counts (per-head masks), the dQ and forward units by query
    head, bit for bit against the oracle."""
    B, S, H, Hkv, d = 2, 1536, 4, 2, 128
    G = H // Hkv
    names = ["causal", "causal_document", "sliding_window", "prefix_lm"]
    per_b = [[gen.make_mask(names[(b + h) % 4], S, b) for h in range(H)] for b in range(B)]
    bounds = bounds_tensor(per_b, device="cuda")
    q = torch.empty(B, S, H, d, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(B, S, Hkv, d, dtype=torch.bfloat16, device="cuda")
    nQ = nK = -(-S // 128)
    nP = (nQ + 1) // 2
    table = om.tile_table(bounds.cpu().numpy(), S)
    rc, _ = om.row_lists(table)
    cc, _ = om.col_lists(table)
    _, pcost, _ = om.pair_lists(table, S)
    ws, L = fm.plan(q, k, bounds, for_bwd=fm.WS_STEP)
    torch.cuda.synchronize()
    assert fm.device_status(ws) == 0

    def view(off, n):
        return ws[off:off + 4 * n].view(torch.int32).cpu().numpy()

    assert np.array_equal(view(L.bwd_order, B * Hkv * nK), om.unit_order(cc, H, G))
    assert np.array_equal(view(L.row_order, B * H * nQ), om.unit_order(rc, H))
    assert np.array_equal(view(L.fwd_order, B * H * nP), om.unit_order(pcost, H))

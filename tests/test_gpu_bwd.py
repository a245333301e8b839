"""Backward parity: fm_bwd through the binding against the fp64 oracle (GPU).

Gradients are compared in full for the sampled (batch, head) pairs:
max |G - G_ref| <= 2e-2 * max |G_ref| for G in dQ, dK, dV.
"""
import numpy as np
import pytest
import torch

import masked_attention_bound_gb300 as fm
from fm_inputs import masks as gen
from fm_inputs.configs import (LOCALIZE_64K, LOCALIZE_RANKS, LONG_128K, SUITE_32K, SWEEP_4K, TINY,
                               TINY_DOCS, dual_chunk_map)
from fm_inputs.tensors import bounds_tensor, mask_bounds, qkv_do, randn_bf16
from parity import GRAD_REL, O_TOL, compare_bwd, compare_fwd

pytestmark = pytest.mark.gpu


def _run(q, k, v, do, bounds, scale):
    o, lse = fm.forward(q, k, v, bounds, scale)
    dq, dk, dv = fm.backward(q, k, v, o, lse, do, bounds, scale)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def test_tiny_config():
    q, k, v, do = qkv_do(TINY.B, TINY.S, TINY.S, TINY.H, TINY.d, device="cuda")
    bounds = bounds_tensor([[gen.causal_document(TINY.S, TINY_DOCS)]], device="cuda")
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, TINY.scale)
    compare_fwd(q, k, v, bounds, TINY.scale, o, lse)
    compare_bwd(q, k, v, do, bounds, TINY.scale, dq, dk, dv)


@pytest.mark.parametrize("name", ["causal_document", "share_question", "random_eviction"])
def test_planned_step_equals_separate_calls(name):
    """One mask analysis per step (fm_plan on a step workspace, then
    fm_fwd_planned and fm_bwd_planned) gives bit-identical O, LSE, dQ, dK, dV
    to fm_fwd and fm_bwd with their own analyses, and launches each analysis
    kernel once per step; repeated on the same workspace, it stays identical."""
    B, S, H, d = 1, 2 * 1024 + 77, 4, 128
    scale = d ** -0.5
    q, k, v, do = qkv_do(B, S, S, H, d, seed=5, device="cuda")
    bounds = mask_bounds(name, B, S, device="cuda")
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, scale)
    desc = fm.make_desc(q, k, v, q)
    ws = fm.workspace(desc, fm.WS_STEP)
    got = None
    fm.profile_read()  # clears the counters
    for rep in range(2):
        fm.profile_enable(True)
        fm.plan(q, k, bounds, ws=ws, for_bwd=fm.WS_STEP)
        o2, lse2 = fm.forward(q, k, v, bounds, scale, ws=ws, planned=True)
        dq2, dk2, dv2 = fm.backward(q, k, v, o2, lse2, do, bounds, scale, ws=ws, planned=True)
        torch.cuda.synchronize()
        fm.profile_enable(False)
        prof = fm.profile_read()
        assert fm.device_status(ws) == 0
        # one launch each per step (order_kernel builds the forward pairs', the
        # dK/dV columns' and the dQ rows' orders in one launch)
        for kname in ("summary_kernel", "classify_kernel", "tile_mask_kernel", "order_kernel",
                      "fwd_kernel", "bwd_pre_kernel", "bwd_kv_kernel", "bwd_dq_kernel"):
            assert prof[kname][1] == 1, (kname, prof[kname])
        for a, b_ in ((o, o2), (lse, lse2), (dq, dq2), (dk, dk2), (dv, dv2)):
            assert torch.equal(a, b_)
        if got is not None:
            assert all(torch.equal(a, b_) for a, b_ in zip(got, (o2, lse2, dq2, dk2, dv2)))
        got = (o2, lse2, dq2, dk2, dv2)


@pytest.mark.parametrize("d", [64, 128])
def test_step_captured_as_cuda_graph(d):
    """A training step (analysis on a step workspace, planned forward and
    backward) captured once as a CUDA graph replays to bit-identical outputs,
    with new inputs copied into the captured buffers between replays."""
    B, S, H = 2, 1000, 4
    scale = d ** -0.5
    q, k, v, do = qkv_do(B, S, S, H, d, seed=21, device="cuda")
    bounds = mask_bounds("causal_document", B, S, device="cuda")
    desc = fm.make_desc(q, k, v, q)
    ws = fm.workspace(desc, fm.WS_STEP)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step(st):
        fm.plan(q, k, bounds, ws=ws, for_bwd=fm.WS_STEP, stream=st)
        fm.forward(q, k, v, bounds, scale, o=o, lse=lse, ws=ws, stream=st, planned=True)
        fm.backward(q, k, v, o, lse, do, bounds, scale, dq=dq, dk=dk, dv=dv, ws=ws, stream=st,
                    planned=True)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)                      # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(side)
    for seed in (22, 23):
        q2, k2, v2, do2 = qkv_do(B, S, S, H, d, seed=seed, device="cuda")
        for dst, src in ((q, q2), (k, k2), (v, v2), (do, do2)):
            dst.copy_(src)
        for t in (o, dq, dk, dv):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert fm.device_status(ws) == 0
        ref = _run(q, k, v, do, bounds, scale)
        for a, b_ in zip(ref, (o, lse, dq, dk, dv)):
            assert torch.equal(a, b_)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [1, 77, 128, 300, 1000])
@pytest.mark.parametrize("name", ["full", "causal", "causal_document", "qk_sparse",
                                  "share_question", "random_eviction", "global_sliding"])
def test_small_shapes(name, S, d):
    B, H = 2, 2
    q, k, v, do = qkv_do(B, S, S, H, d, seed=S + 1, device="cuda")
    bl = [gen.make_mask(name, S, seed=b, window=max(1, S // 5), n_global=min(7, S)) for b in range(B)]
    bounds = bounds_tensor([[x] for x in bl], device="cuda")
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, d ** -0.5)
    compare_bwd(q, k, v, do, bounds, d ** -0.5, dq, dk, dv)


def test_fully_masked_rows_and_columns_are_zero():
    S, H, d = 512, 2, 128
    q, k, v, do = qkv_do(1, S, S, H, d, device="cuda")
    bounds = bounds_tensor([[gen.qk_sparse(S)]], device="cuda")
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, d ** -0.5)
    qs, qe, ks, ke = gen.qk_sparse_ranges(S)
    assert torch.all(dq[:, qs:qe] == 0)
    assert torch.all(dk[:, ks:ke] == 0) and torch.all(dv[:, ks:ke] == 0)
    assert torch.all(torch.isneginf(lse[:, :, qs:qe]))
    compare_bwd(q, k, v, do, bounds, d ** -0.5, dq, dk, dv)


def test_per_head_masks_strides_and_cross_lengths():
    B, Sq, Skv, H, d = 2, 384, 640, 3, 128
    base_q = randn_bf16(B, Sq, H, 2 * d, seed=11, device="cuda")
    base_kv = randn_bf16(B, Skv, H, 2 * d, seed=12, device="cuda")
    q = base_q[..., :d]
    do = base_q[..., d:]
    k, v = base_kv[..., :d], base_kv[..., d:]
    rng = np.random.default_rng(3)
    per_b = []
    for b in range(B):
        heads = []
        for h in range(H):
            a = rng.integers(0, Sq + 1, size=(4, Skv))
            heads.append((np.minimum(a[0], a[1]), np.maximum(a[0], a[1]),
                          np.minimum(a[2], a[3]), np.maximum(a[2], a[3])))
        per_b.append(heads)
    bounds = bounds_tensor(per_b, device="cuda")
    o = torch.empty(B, Sq, H, 2 * d, device="cuda", dtype=torch.bfloat16)[..., :d]
    o, lse = fm.forward(q, k, v, bounds, 0.1, o=o)
    dq = torch.empty(B, Sq, H, 2 * d, device="cuda", dtype=torch.bfloat16)[..., d:]
    dk = torch.empty(B, Skv, H, 2 * d, device="cuda", dtype=torch.bfloat16)[..., :d]
    dv = torch.empty(B, Skv, H, 2 * d, device="cuda", dtype=torch.bfloat16)[..., d:]
    do_o = torch.empty(B, Sq, H, 2 * d, device="cuda", dtype=torch.bfloat16)[..., d:]
    do_o.copy_(do)  # dO must have O's strides
    fm.backward(q, k, v, o, lse, do_o, bounds, 0.1, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    compare_fwd(q, k, v, bounds, 0.1, o, lse)
    compare_bwd(q, k, v, do, bounds, 0.1, dq, dk, dv)


@pytest.mark.parametrize("d", [64, 128])
def test_outputs_in_16_byte_aligned_rows(d):
    """Rows that start on 16-byte but not 32-byte boundaries (head stride
    d + 8, for every tensor) take the kernels' 16-byte store paths for O, dQ,
    dK and dV; the results equal, bit for bit, those of the contiguous
    layout, which takes the 32-byte paths, and match the oracle."""
    B, S, H = 1, 700, 2
    q, k, v, do = qkv_do(B, S, S, H, d, seed=21, device="cuda")
    bounds = mask_bounds("causal_document", B, S, device="cuda")
    ref = _run(q, k, v, do, bounds, d ** -0.5)

    def padded(t):
        big = torch.zeros(B, S, H, d + 8, device="cuda", dtype=torch.bfloat16)
        view = big[..., 8:]
        view.copy_(t)
        return view

    qp, kp, vp, dop = padded(q), padded(k), padded(v), padded(do)
    o = padded(torch.zeros_like(q))
    o, lse = fm.forward(qp, kp, vp, bounds, d ** -0.5, o=o)
    dq, dk, dv = (padded(torch.zeros_like(t)) for t in (q, k, v))
    dq, dk, dv = fm.backward(qp, kp, vp, o, lse, dop, bounds, d ** -0.5, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for t in (o, dq, dk, dv):
        assert t.data_ptr() % 32 == 16 and t.stride(2) % 16 == 8
    for got, want in zip((o, lse, dq, dk, dv), ref):
        assert torch.equal(got, want)
    compare_fwd(q, k, v, bounds, d ** -0.5, o, lse)
    compare_bwd(q, k, v, do, bounds, d ** -0.5, dq, dk, dv)


@pytest.mark.parametrize("name", SWEEP_4K.masks)
def test_sweep_4k_sampled_heads(name):
    W = SWEEP_4K
    q, k, v, do = qkv_do(W.B, W.S, W.S, W.H, W.d, device="cuda")
    bounds = mask_bounds(name, W.B, W.S, device="cuda")
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, W.scale)
    compare_bwd(q, k, v, do, bounds, W.scale, dq, dk, dv, heads=[(0, 0), (3, 15)])


@pytest.mark.parametrize("name", ["causal_document", "share_question", "qk_sparse", "global_sliding"])
def test_suite_32k_sampled_head(name):
    W = SUITE_32K
    q, k, v, do = qkv_do(W.B, W.S, W.S, W.H, W.d, device="cuda")
    bounds = mask_bounds(name, W.B, W.S, device="cuda")
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, W.scale)
    compare_bwd(q, k, v, do, bounds, W.scale, dq, dk, dv, heads=[(0, 5)])


def test_long_128k_sampled_head():
    W = LONG_128K
    q, k, v, do = qkv_do(W.B, W.S, W.S, W.H, W.d, device="cuda")
    bounds = mask_bounds("causal_document_window", W.B, W.S, device="cuda", window=8192)
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, W.scale)
    compare_fwd(q, k, v, bounds, W.scale, o, lse, heads=[(0, 3)], rows=64)
    compare_bwd(q, k, v, do, bounds, W.scale, dq, dk, dv, heads=[(0, 3)])


def test_localized_ranks_match_global_run():
    """Localisation end to end: per simulated rank, localise the bounds and run
    local-Q x full-KV forward and backward; the concatenated O, LSE, dQ and the
    rank sums of dK, dV match the global run (and the global run matches the
    oracle on a sampled head)."""
    W = LOCALIZE_64K
    q, k, v, do = qkv_do(W.B, W.S, W.S, W.H, W.d, device="cuda")
    bounds = mask_bounds("causal_document", W.B, W.S, device="cuda")
    o, lse, dq, dk, dv = _run(q, k, v, do, bounds, W.scale)
    o_l = torch.zeros_like(o)
    lse_l = torch.zeros_like(lse)
    dq_l = torch.zeros_like(dq)
    dk_sum = torch.zeros(dk.shape, dtype=torch.float32, device="cuda")
    dv_sum = torch.zeros(dv.shape, dtype=torch.float32, device="cuda")
    for chunks in dual_chunk_map(W.S, LOCALIZE_RANKS):
        rows = torch.cat([torch.arange(g, g + c, device="cuda") for g, c in chunks])
        lb = fm.localize(bounds, chunks)
        ql, dol = q[:, rows].contiguous(), do[:, rows].contiguous()
        ol, lsel = fm.forward(ql, k, v, lb, W.scale)
        dql, dkl, dvl = fm.backward(ql, k, v, ol, lsel, dol, lb, W.scale)
        o_l[:, rows] = ol
        lse_l[:, :, rows] = lsel
        dq_l[:, rows] = dql
        dk_sum += dkl.float()
        dv_sum += dvl.float()
    torch.cuda.synchronize()
    assert (o_l.float() - o.float()).abs().max().item() <= O_TOL
    fin = torch.isfinite(lse)
    assert torch.equal(fin, torch.isfinite(lse_l))
    assert (lse_l[fin] - lse[fin]).abs().max().item() <= 1e-3
    for got, ref in ((dq_l.float(), dq.float()), (dk_sum, dk.float()), (dv_sum, dv.float())):
        assert (got - ref).abs().max().item() <= GRAD_REL * ref.abs().max().item()
    compare_fwd(q, k, v, bounds, W.scale, o, lse, heads=[(0, 9)], rows=64)
    compare_bwd(q, k, v, do, bounds, W.scale, dq, dk, dv, heads=[(0, 9)])

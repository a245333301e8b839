"""FP8 (e4m3) forward on the GPU against oracle.fp8.

Quantisation: codes and scales bit for bit (both sides divide in fp32 and
round to nearest even).  Forward: O and LSE against the oracle's FP8
attention on the oracle's own quantisation of the same bf16 inputs, with the
bars of parity.py (the e4m3 rounding of Q, K, V and P is in the reference,
so what remains is accumulation order).
"""
import numpy as np
import pytest
import torch

import masked_attention_bound_gb300 as fm
from fm_inputs.configs import SUITE_32K
from fm_inputs.tensors import bounds_tensor, mask_bounds, randn_bf16
from oracle import fp8 as of
from parity import LSE_TOL, O_TOL, mask_vec, o_excess, sample_rows

pytestmark = pytest.mark.gpu


def _codes(t):
    return t.view(torch.float8_e4m3fn).float().cpu().numpy().astype(np.float64)


def _inputs(B, Sq, Skv, H, Hkv, seed, zero_tile=False):
    q = randn_bf16(B, Sq, H, 128, seed=seed, device="cuda")
    k = randn_bf16(B, Skv, Hkv, 128, seed=seed + 1, device="cuda")
    v = randn_bf16(B, Skv, Hkv, 128, seed=seed + 2, device="cuda")
    # V tiles of different magnitudes (the per-tile scales differ)
    mag = torch.tensor([1.0, 8.0, 0.25, 2.0], device="cuda")
    idx = (torch.arange(Skv, device="cuda") // 128) % 4
    v = (v.float() * mag[idx][None, :, None, None]).to(torch.bfloat16)
    if zero_tile and Skv > 256:
        k[:, 128:256] = 0
    return q, k, v


@pytest.mark.parametrize("Sq,Skv,H,Hkv", [(300, 300, 2, 2), (1000, 1000, 4, 2), (384, 640, 2, 1)])
def test_quantize_bit_exact(Sq, Skv, H, Hkv):
    q, k, v = _inputs(2, Sq, Skv, H, Hkv, seed=70, zero_tile=True)
    f = fm.quantize_fp8(q, k, v)
    torch.cuda.synchronize()
    nK = -(-Skv // 128)
    for b in range(2):
        for h in range(H):
            c, s = of.quantize_tiles(q[b, :, h].float().cpu().numpy())
            assert np.array_equal(_codes(f.q8[b, :, h]), c)
            assert np.array_equal(f.q_scale[b, h].cpu().numpy(), s)
        for h in range(Hkv):
            c, s = of.quantize_tiles(k[b, :, h].float().cpu().numpy())
            assert np.array_equal(_codes(f.k8[b, :, h]), c)
            assert np.array_equal(f.k_scale[b, h].cpu().numpy(), s)
            c, s = of.quantize_tiles(v[b, :, h].float().cpu().numpy())
            vt = _codes(f.v8t[b, h])                   # [128][nK*128]
            assert np.array_equal(vt[:, :Skv].T, c) and not vt[:, Skv:].any()
            assert np.array_equal(f.v_scale[b, h].cpu().numpy(), s)
            assert f.v_head_scale[b, h].item() == s.max()
    assert f.v8t.shape[-1] == nK * 128


def _check(q, k, v, bounds, scale, o, lse, heads, rows=None):
    H, Hkv = q.shape[2], k.shape[2]
    for n, (b, h) in enumerate(heads):
        hk = h // (H // Hkv)
        q8, sq = of.quantize_tiles(q[b, :, h].float().cpu().numpy())
        k8, sk = of.quantize_tiles(k[b, :, hk].float().cpu().numpy())
        v8, sv = of.quantize_tiles(v[b, :, hk].float().cpu().numpy())
        r = sample_rows(q.shape[1], rows, n)
        ro, rl = of.forward_head_fp8(q8, sq, k8, sk, v8, sv, mask_vec(bounds, b, h), scale, rows=r)
        go = o[b, r, h].float().cpu().numpy()
        gl = lse[b, h, r].cpu().numpy().astype(np.float64)
        dead = np.isneginf(rl)
        assert np.array_equal(np.isneginf(gl), dead)
        assert float(o_excess(go, ro).max()) <= O_TOL, (b, h)
        if (~dead).any():
            assert float(np.abs(gl[~dead] - rl[~dead]).max()) <= LSE_TOL, (b, h)


@pytest.mark.parametrize("S", [77, 300, 1000])
@pytest.mark.parametrize("name", ["causal_document", "share_question", "full", "causal"])
def test_fp8_forward_small(name, S):
    q, k, v = _inputs(1, S, S, 2, 2, seed=80)
    bounds = mask_bounds(name, 1, S, device="cuda")
    f = fm.quantize_fp8(q, k, v)
    o, lse = fm.forward_fp8(f, bounds, 128 ** -0.5)
    torch.cuda.synchronize()
    _check(q, k, v, bounds, 128 ** -0.5, o, lse, [(0, 0), (0, 1)])


def test_fp8_forward_per_head_masks_gqa_cross_lengths():
    B, Sq, Skv, H, Hkv = 2, 384, 640, 4, 2
    q, k, v = _inputs(B, Sq, Skv, H, Hkv, seed=90)
    rng = np.random.default_rng(9)
    per_b = []
    for _ in range(B):
        heads = []
        for _ in range(H):
            a = rng.integers(0, Sq + 1, size=(4, Skv))
            heads.append((np.minimum(a[0], a[1]), np.maximum(a[0], a[1]),
                          np.minimum(a[2], a[3]), np.maximum(a[2], a[3])))
        per_b.append(heads)
    bounds = bounds_tensor(per_b, device="cuda")
    f = fm.quantize_fp8(q, k, v)
    o, lse = fm.forward_fp8(f, bounds, 0.1)
    torch.cuda.synchronize()
    _check(q, k, v, bounds, 0.1, o, lse, [(b, h) for b in range(B) for h in range(H)])


def test_fp8_forward_32k_sampled_head():
    W = SUITE_32K
    q, k, v = _inputs(W.B, W.S, W.S, W.H, W.H, seed=100)
    bounds = mask_bounds("causal_document", W.B, W.S, device="cuda")
    f = fm.quantize_fp8(q, k, v)
    o, lse = fm.forward_fp8(f, bounds, W.scale)
    torch.cuda.synchronize()
    _check(q, k, v, bounds, W.scale, o, lse, [(0, 7)], rows=512)


def test_forward_into_16_byte_aligned_rows():
    """An O whose rows start on 16-byte but not 32-byte boundaries takes the
    FP8 forward's 16-byte store instance; O and LSE equal, bit for bit, those
    written into a contiguous O (the 32-byte instance)."""
    B, S, H = 1, 700, 2
    q, k, v = _inputs(B, S, S, H, H, seed=91)
    bounds = mask_bounds("causal_document", B, S, device="cuda")
    f = fm.quantize_fp8(q, k, v)
    o_ref, lse_ref = fm.forward_fp8(f, bounds, 128 ** -0.5)
    big = torch.zeros(B, S, H, 128 + 8, device="cuda", dtype=torch.bfloat16)
    o = big[..., 8:]
    o, lse = fm.forward_fp8(f, bounds, 128 ** -0.5, o=o)
    torch.cuda.synchronize()
    assert o.data_ptr() % 32 == 16 and o.stride(2) % 16 == 8
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert torch.all(big[..., :8] == 0)

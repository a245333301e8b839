"""Pins for the FP8 (e4m3) oracle (no GPU).

e4m3 rounding is checked against torch's float8_e4m3fn conversion (a library
routine: nearest, ties to even) over every finite magnitude and random
values, with saturation at 448 from the format's definition; the per-tile
quantisation by its defining properties; the FP8 attention against exact
float64 attention (within the quantisation error, on data whose V tiles
differ in magnitude), by a power-of-two scale invariance, and by a planted
mistake (the V tile's scale ratio left out of P) that must fail the first.
"""
import numpy as np
import pytest
import torch

from fm_inputs import masks as gen
from oracle import attention as oa
from oracle import fp8


def test_e4m3_matches_torch_inside_the_finite_range():
    # every e4m3 value, the midpoints between neighbours, and random values
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    vals = np.unique(codes[np.isfinite(codes)])
    mids = (vals[1:] + vals[:-1]) / 2
    rng = np.random.default_rng(0)
    rand = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 20000)])
    x = np.concatenate([vals, mids, rand]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(fp8.e4m3(x), want.astype(np.float64))


def test_e4m3_saturates_and_keeps_sign():
    x = np.array([448.0, 463.9, 464.0, 500.0, 1e6, -1e6, -449.0])
    assert fp8.e4m3(x).tolist() == [448, 448, 448, 448, 448, -448, -448]
    assert fp8.e4m3(np.array([0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -11])).tolist() == [
        0, 0, 0, 2.0 ** -9]


def test_quantize_tiles_properties():
    rng = np.random.default_rng(1)
    x = rng.normal(0, 3, (300, 64)).astype(np.float32)
    x[128:256] = 0  # an all-zero tile
    codes, s = fp8.quantize_tiles(x)
    assert s.dtype == np.float32 and s[1] == 1 and not codes[128:256].any()
    for t, (lo, hi) in enumerate(((0, 128), (256, 300))):
        ti = 0 if t == 0 else 2
        blk = x[lo:hi]
        assert s[ti] == np.float32(np.abs(blk).max() / np.float32(448))
        # the tile's largest magnitude maps to 448 up to the float32 division
        assert abs(np.abs(codes[lo:hi]).max() - 448) <= 448 * 2 ** -3
        # every code is x * (448 / amax) rounded: within half a step of e4m3
        # at its size of x / s
        err = np.abs(codes[lo:hi] - blk / s[ti])
        assert np.all(err <= np.maximum(np.abs(blk / s[ti]) * 2 ** -4, 2 ** -10))


def _fp8_inputs(S, d, seed, vmag):
    rng = np.random.default_rng(seed)
    q = rng.normal(0, 1, (S, d)).astype(np.float32)
    k = rng.normal(0, 1, (S, d)).astype(np.float32)
    v = rng.normal(0, 1, (S, d)).astype(np.float32)
    for t in range(-(-S // 128)):  # V tiles of very different magnitudes
        v[t * 128:(t + 1) * 128] *= vmag[t % len(vmag)]
    return q, k, v


@pytest.mark.parametrize("name", ["causal", "causal_document", "full"])
def test_fp8_attention_close_to_exact(name):
    S, d, scale = 640, 64, 64 ** -0.5
    q, k, v = _fp8_inputs(S, d, 3, [1.0, 8.0, 0.125, 2.0, 0.5])
    mvec = gen.make_mask(name, S) if name != "causal_document" else gen.causal_document(S, [200, 300, 140])
    q8, sq = fp8.quantize_tiles(q)
    k8, sk = fp8.quantize_tiles(k)
    v8, sv = fp8.quantize_tiles(v)
    o, lse = fp8.forward_head_fp8(q8, sq, k8, sk, v8, sv, mvec, scale)
    ro, rl = oa.forward_head(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                             mvec, scale)
    vmax = np.abs(v).max(axis=0).max()
    err = np.abs(o - ro)
    assert err.max() <= 0.08 * vmax and err.mean() <= 0.01 * vmax
    live = np.isfinite(rl)
    # S from e4m3 Q and K: up to about 2^-4 relative per factor
    assert np.array_equal(np.isfinite(lse), live) and np.abs(lse[live] - rl[live]).max() < 0.25


def test_fp8_attention_power_of_two_invariance():
    S, d, scale = 384, 64, 0.125
    q, k, v = _fp8_inputs(S, d, 4, [1.0, 4.0, 0.25])
    mvec = gen.make_mask("causal", S)
    q8, sq = fp8.quantize_tiles(q)
    k8, sk = fp8.quantize_tiles(k)
    v8, sv = fp8.quantize_tiles(v)
    o, lse = fp8.forward_head_fp8(q8, sq, k8, sk, v8, sv, mvec, scale)
    v8b, svb = fp8.quantize_tiles(v * np.float32(16))
    o2, lse2 = fp8.forward_head_fp8(q8, sq, k8, sk, v8b, svb, mvec, scale)
    assert np.array_equal(v8b, v8) and np.array_equal(o2, 16 * o) and np.array_equal(lse2, lse)


def test_planted_missing_v_ratio_is_caught():
    """P rounded without the V tile's scale ratio (one scale per head assumed)
    is far from exact attention when V tiles differ in magnitude."""
    S, d, scale = 640, 64, 64 ** -0.5
    q, k, v = _fp8_inputs(S, d, 3, [1.0, 8.0, 0.125, 2.0, 0.5])
    mvec = gen.make_mask("full", S)
    q8, sq = fp8.quantize_tiles(q)
    k8, sk = fp8.quantize_tiles(k)
    v8, sv = fp8.quantize_tiles(v)
    o, _ = fp8.forward_head_fp8(q8, sq, k8, sk, v8, np.full_like(sv, sv.max()), mvec, scale)
    ro, _ = oa.forward_head(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                            mvec, scale)
    assert np.abs(o - ro).max() > 0.08 * np.abs(v).max()

"""Packed variable-length batches (fm_varlen_bounds) on the GPU.

Bounds bit for bit against oracle.masks.varlen_bounds; attention over a
packed batch against the oracle run on each sequence alone (an independent
route: no cross-sequence mask is involved there).  Tolerances as in parity.py.
"""
import numpy as np
import pytest
import torch

import masked_attention_bound_gb300 as fm
from fm_inputs.tensors import randn_bf16
from oracle import attention as oa
from oracle import masks as om
from parity import GRAD_FLOOR, GRAD_REL, LSE_TOL, O_TOL, o_excess

pytestmark = pytest.mark.gpu


def _cu(lengths):
    return [0] + np.cumsum(lengths).tolist()


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_bounds_bit_exact(causal):
    rng = np.random.default_rng(7)
    lengths = rng.integers(0, 700, size=40).tolist()
    lengths[3] = 0
    cu = _cu(lengths)
    got = fm.varlen_bounds(torch.tensor(cu, dtype=torch.int32, device="cuda"), causal=causal)
    torch.cuda.synchronize()
    assert np.array_equal(got[:, 0, 0].cpu().numpy(), om.varlen_bounds(cu, causal))


@pytest.mark.parametrize("cu", [[0, 5, 3, 10], [1, 5, 10], [0, 5, 12]])
def test_varlen_bounds_rejects_non_partitions(cu):
    with pytest.raises(ValueError):
        fm.varlen_bounds(torch.tensor(cu, dtype=torch.int32, device="cuda"), total=10)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_packed_batch_equals_each_sequence_alone(causal, d):
    lengths = [300, 0, 700, 77, 129, 423, 1]
    cu = _cu(lengths)
    T, H = cu[-1], 2
    scale = d ** -0.5
    q, k, v, do = (randn_bf16(1, T, H, d, seed=60 + i, device="cuda") for i in range(4))
    bounds = fm.varlen_bounds(torch.tensor(cu, dtype=torch.int32, device="cuda"), causal=causal)
    o, lse = fm.forward(q, k, v, bounds, scale)
    dq, dk, dv = fm.backward(q, k, v, o, lse, do, bounds, scale)
    torch.cuda.synchronize()
    for a, b in zip(cu[:-1], cu[1:]):
        if b == a:
            continue
        mvec = tuple(om.varlen_bounds([0, b - a], causal))
        for h in range(H):
            sl = lambda t: oa.to64(t[0, a:b, h])  # noqa: E731
            rq, rk, rv, ro, rl, _ = oa.backward_head(sl(q), sl(k), sl(v), sl(do), mvec, scale)
            assert float(o_excess(o[0, a:b, h].float().cpu().numpy(), ro).max()) <= O_TOL
            assert float(np.abs(lse[0, h, a:b].cpu().numpy() - rl).max()) <= LSE_TOL
            for g, ref in ((dq, rq), (dk, rk), (dv, rv)):
                err = float(np.abs(g[0, a:b, h].float().cpu().numpy() - ref).max())
                assert err <= GRAD_REL * max(float(np.abs(ref).max()), GRAD_FLOOR), (a, b, h)

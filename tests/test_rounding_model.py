"""The forward's rounding model against the fp64 oracle (no GPU).

Seed 267 of the per-head forward test (B=2, S=640, H=3, d=128, scale 0.1;
head (b=0, h=1), a causal mask) is a case where the rounding that the design
implies -- probabilities rounded to bf16 before the P V product and the output
rounded to bf16 -- alone puts an element more than 1e-2 from the exact result:
row 1 sees two keys, |O_ref| is about 2.27, where bf16 numbers are 2^-6 apart.
The model's O before its final rounding is well within 1e-2, and the parity
bar (1e-2 beyond half a bf16 ulp of O_ref) holds.  Over other seeds the model
stays within the plain 1e-2 as well.
"""
import numpy as np
import pytest

from fm_inputs import masks as gen
from fm_inputs.tensors import randn_bf16
from oracle import attention as oa
from oracle import masks as om
from parity import O_TOL, o_excess
from rounding_model import forward_head

B, S, H, d = 2, 640, 3, 128
NAMES = ("causal", "share_question", "prefix_document")


def _head(seed, b, h):
    base = randn_bf16(B, S, H, 3 * d, seed=seed).float().numpy().astype(np.float64)
    mvec = gen.make_mask(NAMES[h], S, seed=b)
    q, k, v = base[b, :, h, :d], base[b, :, h, d:2 * d], base[b, :, h, 2 * d:]
    ref, _ = oa.forward_head(q, k, v, mvec, 0.1)
    return q, k, v, om.dense_mask(*mvec, S), ref


def test_seed_267_exceeds_1e2_by_rounding_alone():
    q, k, v, M, ref = _head(267, 0, 1)
    o_bf16, o32 = forward_head(q, k, v, M, 0.1)
    err = np.abs(o_bf16 - ref)
    i, c = np.unravel_index(err.argmax(), err.shape)
    assert err.max() > 1e-2
    assert i == 1 and (~M[1]).sum() == 2
    assert abs(ref[i, c]) > 2.0
    assert np.abs(o32 - ref).max() < 0.006
    assert o_excess(o_bf16, ref).max() <= O_TOL


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_model_within_the_plain_bar_on_other_seeds(seed):
    for b in range(B):
        for h in range(H):
            q, k, v, M, ref = _head(seed, b, h)
            o_bf16, _ = forward_head(q, k, v, M, 0.1)
            assert np.abs(o_bf16 - ref).max() <= 1e-2

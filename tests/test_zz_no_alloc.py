"""fm_fwd_static: the forward pass for callers that cannot allocate device
memory (a plugin under a framework that owns every byte of device memory, or
a latency-critical path that must not call cudaMalloc/cudaFree).  Its scratch
is a fixed array inside the library, shared by all calls on a GPU.

Checked through the C ABI against fm_fwd (the entry point with a caller
workspace) on two calls in a row with different masks, so stale scratch from
the first call would show in the second; and the size limit is enforced on
the host.  This file sorts last so that a run stopping at its first failure
has run every other test already.
"""
import ctypes

import pytest
import torch

import masked_attention_bound_gb300 as fm
from masked_attention_bound_gb300 import _abi
from fm_inputs.tensors import mask_bounds, qkv_do
from parity import LSE_TOL, O_TOL

pytestmark = pytest.mark.gpu


def _static_fwd(q, k, v, bounds, scale):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], q.shape[2], q.shape[1], dtype=torch.float32, device=q.device)
    desc = fm.make_desc(q, k, v, o, Hm=bounds.shape[2])
    p = [ctypes.c_void_p(bounds[t].data_ptr()) for t in range(4)]
    rc = fm.lib().fm_fwd_static(ctypes.byref(desc), ctypes.c_void_p(q.data_ptr()),
                                ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()), *p,
                                ctypes.c_float(scale), ctypes.c_void_p(o.data_ptr()),
                                ctypes.c_void_p(lse.data_ptr()),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, o, lse


def test_static_scratch_forward_matches_workspace_forward():
    B, S, H, d = 2, 2048, 4, 128
    q, k, v, _ = qkv_do(B, S, S, H, d, seed=7, device="cuda")
    for n, name in enumerate(("causal_document", "share_question")):
        bounds = mask_bounds(name, B, S, seed=n, device="cuda")
        rc, o_s, lse_s = _static_fwd(q, k, v, bounds, d ** -0.5)
        assert rc == _abi.FM_OK
        o_w, lse_w = fm.forward(q, k, v, bounds, d ** -0.5)
        torch.cuda.synchronize()
        assert (o_s.float() - o_w.float()).abs().max().item() <= O_TOL
        fin = torch.isfinite(lse_w)
        assert torch.equal(fin, torch.isfinite(lse_s))
        assert (lse_s[fin] - lse_w[fin]).abs().max().item() <= LSE_TOL


def test_static_scratch_without_room_for_every_tile_mask():
    """At 32K random eviction the fixed scratch holds the bit masks of only a
    few thousand of the ~33K partial tiles; the forward kernel builds the rest
    from the bounds.  Same bits, same schedule: O and LSE equal fm_fwd's."""
    B, S, H, d = 1, 32768, 2, 64
    q, k, v, _ = qkv_do(B, S, S, H, d, seed=9, device="cuda")
    bounds = mask_bounds("random_eviction", B, S, device="cuda")
    rc, o_s, lse_s = _static_fwd(q, k, v, bounds, d ** -0.5)
    assert rc == _abi.FM_OK
    o_w, lse_w = fm.forward(q, k, v, bounds, d ** -0.5)
    torch.cuda.synchronize()
    assert torch.equal(o_s, o_w)
    assert torch.equal(lse_s, lse_w)


def test_static_scratch_rejects_problems_beyond_its_size():
    B, S, H, d = 1, 1 << 17, 1, 64
    q = torch.empty(B, S, H, d, dtype=torch.bfloat16, device="cuda")
    desc = fm.make_desc(q, q)
    assert fm.lib().fm_workspace_size(ctypes.byref(desc), 0) > (8 << 20)
    bounds = torch.zeros(4, B, 1, S, dtype=torch.int32, device="cuda")
    rc, _, _ = _static_fwd(q, q, q, bounds, 0.1)
    assert rc == _abi.FM_ERR_WORKSPACE

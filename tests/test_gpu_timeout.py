"""The bounded-wait unwind path on the GPU.

Every mbarrier wait in the attention kernels is bounded; on expiry the launch
records FM_ERR_TIMEOUT, drains what it issued, frees its tensor memory and
returns.  Here a test hook shortens the limit to 20 ms and withholds one
consumer release ("P ready", which the MMA thread waits for before the PV or
dV product, or "dS ready", before the dQ product), so the wait runs out on
purpose: no fault, no trap, no endless
loop.  The status word must say FM_ERR_TIMEOUT, and the next ordinary call on
the same GPU must be clean and match the oracle.
"""
import ctypes
import time

import pytest
import torch

import masked_attention_bound_gb300 as fm
from masked_attention_bound_gb300 import _abi
from fm_inputs.tensors import mask_bounds, qkv_do
from parity import compare_bwd, compare_fwd

pytestmark = pytest.mark.gpu

B, S, H, d = 1, 1024, 2, 128
SCALE = d ** -0.5


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _raw_fwd(q, k, v, bounds, o, lse, ws):
    desc = fm.make_desc(q, k, v, o)
    return fm.lib().fm_fwd(ctypes.byref(desc), _p(q), _p(k), _p(v), *[_p(bounds[t]) for t in range(4)],
                           ctypes.c_float(SCALE), _p(o), _p(lse), _p(ws), ws.numel(),
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _raw_bwd(q, k, v, o, lse, do, bounds, dq, dk, dv, ws):
    desc = fm.make_desc(q, k, v, o)
    return fm.lib().fm_bwd(ctypes.byref(desc), _p(q), _p(k), _p(v), _p(o), _p(lse), _p(do),
                           *[_p(bounds[t]) for t in range(4)], ctypes.c_float(SCALE), _p(dq), _p(dk),
                           _p(dv), _p(ws), ws.numel(),
                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _inputs():
    q, k, v, do = qkv_do(B, S, S, H, d, seed=21, device="cuda")
    bounds = mask_bounds("causal_document", B, S, device="cuda")
    return q, k, v, do, bounds


def test_forward_wait_timeout_is_reported_then_next_call_is_clean():
    q, k, v, _, bounds = _inputs()
    desc = fm.make_desc(q, k, v, q)
    ws = fm.workspace(desc, False)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, S, device="cuda")
    assert fm.lib().fm_test_hooks(20_000_000, 1) == _abi.FM_OK
    try:
        t0 = time.time()
        assert _raw_fwd(q, k, v, bounds, o, lse, ws) == _abi.FM_OK
        code = fm.device_status(ws)
        elapsed = time.time() - t0
    finally:
        assert fm.lib().fm_test_hooks(0, 0) == _abi.FM_OK
    assert code == _abi.FM_ERR_TIMEOUT, _abi.status_string(code)
    assert elapsed < 10.0
    # the same GPU, the same workspace: an ordinary call is clean and correct
    o2, lse2 = fm.forward(q, k, v, bounds, SCALE, ws=ws)
    torch.cuda.synchronize()
    assert fm.device_status(ws) == _abi.FM_OK
    compare_fwd(q, k, v, bounds, SCALE, o2, lse2)


# 2: the dK/dV pass's "P ready" (its MMA thread waits before dV); 3: the dQ
# pass's "dS ready" (its dQ MMA thread waits before the dQ product)
@pytest.mark.parametrize("withhold", [2, 3])
def test_backward_wait_timeout_is_reported_then_next_call_is_clean(withhold):
    q, k, v, do, bounds = _inputs()
    o, lse = fm.forward(q, k, v, bounds, SCALE)
    desc = fm.make_desc(q, k, v, o)
    ws = fm.workspace(desc, True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    assert fm.lib().fm_test_hooks(20_000_000, withhold) == _abi.FM_OK
    try:
        t0 = time.time()
        assert _raw_bwd(q, k, v, o, lse, do, bounds, dq, dk, dv, ws) == _abi.FM_OK
        code = fm.device_status(ws)
        elapsed = time.time() - t0
    finally:
        assert fm.lib().fm_test_hooks(0, 0) == _abi.FM_OK
    assert code == _abi.FM_ERR_TIMEOUT, _abi.status_string(code)
    assert elapsed < 10.0
    dq2, dk2, dv2 = fm.backward(q, k, v, o, lse, do, bounds, SCALE, ws=ws)
    torch.cuda.synchronize()
    assert fm.device_status(ws) == _abi.FM_OK
    compare_bwd(q, k, v, do, bounds, SCALE, dq2, dk2, dv2)


def test_hook_values_are_checked():
    assert fm.lib().fm_test_hooks(0, 4) == _abi.FM_ERR_INVALID
    assert fm.lib().fm_test_hooks(0, -1) == _abi.FM_ERR_INVALID
    assert fm.lib().fm_test_hooks(0, 0) == _abi.FM_OK

"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest
import torch

from masked_attention_bound_gb300 import _abi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return _abi.lib()


def _declared_symbols():
    hdr = open(os.path.join(ROOT, "include", "fm.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(fm_[a-z_]+)\s*\(", hdr)))


def test_exports_every_declared_symbol(L):
    syms = _declared_symbols()
    assert len(syms) >= 8
    for s in syms:
        assert hasattr(L, s), s
    assert set(syms) <= set(_abi.SIGNATURES), "binding lacks a signature"


def _desc(B=1, H=2, Hm=1, Sq=256, Skv=256, d=64):
    q = torch.empty(B, Sq, H, d)
    k = torch.empty(B, Skv, H, d)
    D = _abi.FmDesc()
    D.B, D.H, D.Hm, D.Sq, D.Skv, D.d = B, H, Hm, Sq, Skv, d
    D.q_stride[:] = q.stride()[:3]
    D.k_stride[:] = k.stride()[:3]
    D.v_stride[:] = k.stride()[:3]
    D.o_stride[:] = q.stride()[:3]
    return D


def test_workspace_size_and_layout(L):
    D = _desc()
    n0 = L.fm_workspace_size(ctypes.byref(D), 0)
    n1 = L.fm_workspace_size(ctypes.byref(D), 1)
    assert 0 < n0 < n1
    lay = _abi.FmWsLayout()
    assert L.fm_workspace_layout(ctypes.byref(D), 1, ctypes.byref(lay)) == 0
    offs = [getattr(lay, f) for f, _ in _abi.FmWsLayout._fields_]
    assert all(o % 256 == 0 for o in offs)
    assert lay.total == n1
    # the dQ pass's unit order holds B*H*nQ entries before the bit-mask region
    assert lay.masks - lay.row_order >= 1 * 2 * 2 * 4


def test_step_workspace_holds_both_passes(L):
    """A step workspace (mode 2) has every region of the forward's and of the
    backward's layout; mode 3 is rejected."""
    D = _desc()
    n0, n1, n2 = (L.fm_workspace_size(ctypes.byref(D), m) for m in (0, 1, 2))
    assert n2 >= max(n0, n1)
    lays = []
    for m in (0, 1, 2):
        lay = _abi.FmWsLayout()
        assert L.fm_workspace_layout(ctypes.byref(D), m, ctypes.byref(lay)) == 0
        lays.append(lay)
    f, b, st = lays
    assert f.pair_info and f.pair_list and not f.delta and not f.row_order
    assert b.delta and b.lse_log2 and b.row_order and not b.pair_info
    assert st.pair_info and st.pair_list and st.delta and st.lse_log2 and st.row_order
    assert st.total == n2
    # regions in order, none overlapping the next
    offs = sorted(getattr(st, fld) for fld, _ in _abi.FmWsLayout._fields_ if fld != "total")
    assert len(set(offs)) == len(offs)
    assert L.fm_workspace_size(ctypes.byref(D), 3) == 0
    assert L.fm_workspace_layout(ctypes.byref(D), -1, ctypes.byref(_abi.FmWsLayout())) == 1


@pytest.mark.parametrize("field,value,code", [
    ("d", 96, 3), ("d", 0, 1), ("Hm", 3, 1), ("B", 0, 1), ("Sq", 0, 1), ("Skv", -1, 1)])
def test_bad_descriptions(L, field, value, code):
    D = _desc(H=2)
    setattr(D, field, value)
    assert L.fm_workspace_size(ctypes.byref(D), 0) == 0
    lay = _abi.FmWsLayout()
    assert L.fm_workspace_layout(ctypes.byref(D), 0, ctypes.byref(lay)) == code


def test_bad_strides(L):
    D = _desc()
    D.q_stride[1] = 12  # not a multiple of 8 elements
    assert L.fm_workspace_size(ctypes.byref(D), 0) == 0


def test_null_pointers_rejected_on_host(L):
    D = _desc()
    nul = ctypes.c_void_p(0)
    r = L.fm_fwd(ctypes.byref(D), nul, nul, nul, nul, nul, nul, nul, ctypes.c_float(1.0),
                 nul, nul, nul, 0, nul)
    assert r == _abi.FM_ERR_INVALID
    r = L.fm_bwd(ctypes.byref(D), nul, nul, nul, nul, nul, nul, nul, nul, nul, nul,
                 ctypes.c_float(1.0), nul, nul, nul, nul, 0, nul)
    assert r == _abi.FM_ERR_INVALID
    assert L.fm_device_status(nul, nul) == _abi.FM_ERR_INVALID


def test_localize_rejects_on_host(L):
    nul = ctypes.c_void_p(0)
    starts = (ctypes.c_int32 * 2)(64, 0)
    lens = (ctypes.c_int32 * 2)(32, 32)
    fake_in, fake_out = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 30)
    # descending chunks
    assert L.fm_localize(fake_in, 1, 1, 128, starts, lens, 2, fake_out, nul) == _abi.FM_ERR_INVALID
    # overlapping chunks
    starts = (ctypes.c_int32 * 2)(0, 16)
    assert L.fm_localize(fake_in, 1, 1, 128, starts, lens, 2, fake_out, nul) == _abi.FM_ERR_INVALID
    # too many chunks
    many = (ctypes.c_int32 * 200)(*range(0, 200))
    ones = (ctypes.c_int32 * 200)(*([1] * 200))
    assert L.fm_localize(fake_in, 1, 1, 128, many, ones, 200, fake_out, nul) == _abi.FM_ERR_INVALID
    # overlapping in/out buffers
    starts = (ctypes.c_int32 * 2)(0, 64)
    assert L.fm_localize(fake_in, 1, 1, 128, starts, lens, 2, fake_in, nul) == _abi.FM_ERR_INVALID


def test_status_strings(L):
    for c in range(7):
        assert len(L.fm_status_string(c)) > 0
    assert L.fm_version() >= 100

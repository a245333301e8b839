"""Masked attention in FlashMask's column-wise sparse mask form, for GB300.

Thin Python binding over the C ABI of ``include/fm.h`` (``libfm.so``, built
from ``csrc/`` for sm_103a).  PyTorch provides device memory and streams; every
step of the computation runs in the library's CUDA kernels.  If the library is
missing, every call raises: there is no CPU or PyTorch fallback.

Tensors: q/k/v/o/dO/dq/dk/dv are bf16 CUDA tensors in BSHD layout
([batch][seq][head][head_dim], head_dim contiguous, other strides multiples of
8 elements; outputs whose strides are multiples of 16 elements, on 32-byte
aligned storage such as torch's own allocations, take the kernels' faster
32-byte stores).  ``bounds`` is an int32 CUDA tensor [4][B][Hm][Skv] holding
LTS, LTE, UTS, UTE; key j is hidden from query row i iff LTS[j] <= i < LTE[j]
or UTS[j] <= i < UTE[j].
"""
from __future__ import annotations

import ctypes
from typing import NamedTuple

import torch

from ._abi import FMError, FmDesc, FmWsLayout, check, lib  # noqa: F401

__all__ = ["FMError", "make_desc", "workspace_size", "workspace_layout", "workspace", "plan",
           "forward", "backward", "localize", "device_status", "lib", "profile_enable",
           "profile_read"]


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _strides(t):
    s = t.stride()
    if s[3] != 1:
        raise ValueError("head_dim must be the contiguous dimension")
    return (s[0], s[1], s[2])


def make_desc(q, k, v=None, o=None, Hm: int = 1) -> FmDesc:
    """Problem description from BSHD tensors (v defaults to k's strides, o to q's).
    k and v may have fewer heads than q (grouped-query attention)."""
    B, Sq, H, d = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    D = FmDesc()
    D.B, D.H, D.Hm, D.Sq, D.Skv, D.d, D.Hkv = B, H, Hm, Sq, Skv, d, Hkv
    D.q_stride[:] = _strides(q)
    D.k_stride[:] = _strides(k)
    D.v_stride[:] = _strides(v if v is not None else k)
    D.o_stride[:] = _strides(o if o is not None else q)
    return D


# workspace kinds: the forward's, the backward's, and a step workspace with
# both passes' regions (one mask analysis per training step)
WS_FWD, WS_BWD, WS_STEP = 0, 1, 2


def workspace_size(desc: FmDesc, for_bwd) -> int:
    """Bytes of workspace; ``for_bwd`` is False/True or one of WS_FWD, WS_BWD, WS_STEP."""
    n = lib().fm_workspace_size(ctypes.byref(desc), int(for_bwd))
    if n == 0:
        raise FMError(1, "fm_workspace_size")
    return n


def workspace_layout(desc: FmDesc, for_bwd) -> FmWsLayout:
    out = FmWsLayout()
    check(lib().fm_workspace_layout(ctypes.byref(desc), int(for_bwd), ctypes.byref(out)),
          "fm_workspace_layout")
    return out


def workspace(desc: FmDesc, for_bwd, device="cuda") -> torch.Tensor:
    """A byte tensor large enough (and 256-byte aligned) for the call."""
    return torch.empty(workspace_size(desc, for_bwd), dtype=torch.uint8, device=device)


def _bounds_ptrs(bounds):
    if bounds.dtype != torch.int32 or not bounds.is_contiguous() or bounds.dim() != 4 \
            or bounds.shape[0] != 4:
        raise ValueError("bounds must be a contiguous int32 tensor [4][B][Hm][Skv]")
    return [ctypes.c_void_p(bounds[t].data_ptr()) for t in range(4)]


def plan(q, k, bounds, ws=None, for_bwd=False, stream=None):
    """Run the mask analysis only; returns (workspace tensor, layout).  With
    ``for_bwd=WS_STEP`` it prepares a step workspace for
    ``forward(..., planned=True)`` and ``backward(..., planned=True)``."""
    desc = make_desc(q, k, Hm=bounds.shape[2])
    if ws is None:
        ws = workspace(desc, for_bwd, q.device)
    check(lib().fm_plan(ctypes.byref(desc), *_bounds_ptrs(bounds), _p(ws), ws.numel(),
                        int(for_bwd), _stream_ptr(stream)), "fm_plan")
    return ws, workspace_layout(desc, for_bwd)


def forward(q, k, v, bounds, scale, o=None, lse=None, ws=None, stream=None, planned=False):
    """O [B][Sq][H][d] bf16 and LSE [B][H][Sq] fp32 (natural log).  ``planned``:
    ``ws`` is a step workspace that ``plan(..., for_bwd=WS_STEP)`` prepared for
    these bounds; the mask analysis is then not run again."""
    B, Sq, H, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=q.device)
    desc = make_desc(q, k, v, o, Hm=bounds.shape[2])
    if ws is None:
        if planned:
            raise ValueError("planned=True needs the step workspace plan() prepared")
        ws = workspace(desc, False, q.device)
    name = "fm_fwd_planned" if planned else "fm_fwd"
    check(getattr(lib(), name)(ctypes.byref(desc), _p(q), _p(k), _p(v), *_bounds_ptrs(bounds),
                               ctypes.c_float(scale), _p(o), _p(lse), _p(ws), ws.numel(),
                               _stream_ptr(stream)), name)
    return o, lse


def backward(q, k, v, o, lse, do, bounds, scale, dq=None, dk=None, dv=None, ws=None,
             stream=None, planned=False):
    """dQ, dK, dV (bf16) for the loss whose gradient with respect to O is dO.
    ``planned`` as for ``forward``."""
    if do.stride() != o.stride():
        do = do.contiguous() if o.is_contiguous() else do
        if do.stride() != o.stride():
            raise ValueError("dO must have O's strides")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for a, b_ in ((dq, q), (dk, k), (dv, v)):
        if a.stride() != b_.stride():
            raise ValueError("gradient tensors must have the strides of their inputs")
    desc = make_desc(q, k, v, o, Hm=bounds.shape[2])
    if ws is None:
        if planned:
            raise ValueError("planned=True needs the step workspace plan() prepared")
        ws = workspace(desc, True, q.device)
    name = "fm_bwd_planned" if planned else "fm_bwd"
    check(getattr(lib(), name)(ctypes.byref(desc), _p(q), _p(k), _p(v), _p(o), _p(lse), _p(do),
                               *_bounds_ptrs(bounds), ctypes.c_float(scale), _p(dq), _p(dk),
                               _p(dv), _p(ws), ws.numel(), _stream_ptr(stream)), name)
    return dq, dk, dv


class Fp8Inputs(NamedTuple):
    """e4m3 codes and per-tile scales of Q, K, V (fm_quantize_fp8)."""
    q8: torch.Tensor           # uint8 [B][Sq][H][128]
    k8: torch.Tensor           # uint8 [B][Skv][Hkv][128]
    v8t: torch.Tensor          # uint8 [B][Hkv][128][nK*128], V transposed per head
    q_scale: torch.Tensor      # fp32 [B][H][nQ]
    k_scale: torch.Tensor      # fp32 [B][Hkv][nK]
    v_scale: torch.Tensor      # fp32 [B][Hkv][nK]
    v_head_scale: torch.Tensor  # fp32 [B][Hkv]


def quantize_fp8(q, k, v, stream=None) -> Fp8Inputs:
    """Per-tile e4m3 quantisation of bf16 Q, K, V (head_dim 128)."""
    B, Sq, H, d = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    nQ, nK = -(-Sq // 128), -(-Skv // 128)
    dev = q.device
    out = Fp8Inputs(
        torch.empty(B, Sq, H, d, dtype=torch.uint8, device=dev),
        torch.empty(B, Skv, Hkv, d, dtype=torch.uint8, device=dev),
        torch.empty(B, Hkv, d, nK * 128, dtype=torch.uint8, device=dev),
        torch.empty(B, H, nQ, dtype=torch.float32, device=dev),
        torch.empty(B, Hkv, nK, dtype=torch.float32, device=dev),
        torch.empty(B, Hkv, nK, dtype=torch.float32, device=dev),
        torch.empty(B, Hkv, dtype=torch.float32, device=dev))
    desc = make_desc(q, k, v)
    check(lib().fm_quantize_fp8(ctypes.byref(desc), _p(q), _p(k), _p(v), *(_p(t) for t in out),
                                _stream_ptr(stream)), "fm_quantize_fp8")
    return out


def forward_fp8(f: Fp8Inputs, bounds, scale, o=None, lse=None, ws=None, stream=None):
    """FP8 forward (fm_fwd_fp8) on quantised inputs: O bf16 [B][Sq][H][128], LSE."""
    B, Sq, H, d = f.q8.shape
    if o is None:
        o = torch.empty(B, Sq, H, d, dtype=torch.bfloat16, device=f.q8.device)
    if lse is None:
        lse = torch.empty(B, H, Sq, dtype=torch.float32, device=f.q8.device)
    desc = make_desc(f.q8, f.k8, f.k8, o, Hm=bounds.shape[2])
    if ws is None:
        ws = workspace(desc, WS_FWD, f.q8.device)
    check(lib().fm_fwd_fp8(ctypes.byref(desc), _p(f.q8), _p(f.k8), _p(f.v8t), _p(f.q_scale),
                           _p(f.k_scale), _p(f.v_scale), _p(f.v_head_scale), *_bounds_ptrs(bounds),
                           ctypes.c_float(scale), _p(o), _p(lse), _p(ws), ws.numel(),
                           _stream_ptr(stream)), "fm_fwd_fp8")
    return o, lse


def varlen_bounds(cu_seqlens, total=None, causal=True, stream=None, validate=True):
    """Bounds [4][1][1][total] of a packed variable-length batch (fm_varlen_bounds):
    sequence s holds tokens [cu_seqlens[s], cu_seqlens[s+1]) and sees only itself
    (causally if ``causal``).  ``cu_seqlens``: int32 device tensor [n + 1].
    ``total`` defaults to cu_seqlens[-1] (a device read).  With ``validate``, a
    cu_seqlens that is not a partition of [0, total) raises ValueError."""
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor with at least two entries")
    cu = cu_seqlens.contiguous()
    if total is None:
        total = int(cu[-1].item())
    out = torch.empty(4, 1, 1, total, dtype=torch.int32, device=cu.device)
    bad = torch.zeros(1, dtype=torch.int32, device=cu.device) if validate else None
    check(lib().fm_varlen_bounds(_p(cu), cu.numel() - 1, int(total), int(bool(causal)), _p(out),
                                 _p(bad) if bad is not None else None, _stream_ptr(stream)),
          "fm_varlen_bounds")
    if bad is not None and int(bad.item()) != 0:
        raise ValueError("cu_seqlens is not a partition of [0, total)")
    return out


def localize(bounds, chunks, out=None, stream=None):
    """Bounds local to a rank holding query chunks ``chunks`` = [(global_start, length), ...]
    (ascending, non-overlapping), for local-Q x full-KV attention."""
    if bounds.dtype != torch.int32 or not bounds.is_contiguous() or bounds.shape[0] != 4:
        raise ValueError("bounds must be a contiguous int32 tensor [4][B][Hm][Skv]")
    _, B, Hm, Skv = bounds.shape
    if out is None:
        out = torch.empty_like(bounds)
    n = len(chunks)
    starts = (ctypes.c_int32 * max(n, 1))(*[int(g) for g, _ in chunks])
    lens = (ctypes.c_int32 * max(n, 1))(*[int(c) for _, c in chunks])
    check(lib().fm_localize(_p(bounds), B, Hm, Skv, starts, lens, n, _p(out),
                            _stream_ptr(stream)), "fm_localize")
    return out


def device_status(ws, stream=None) -> int:
    """Synchronise and return the device status code of a workspace (0 = OK)."""
    return lib().fm_device_status(_p(ws), _stream_ptr(stream))


def profile_enable(on: bool = True):
    """Bracket every library kernel launch with CUDA events (see fm.h)."""
    check(lib().fm_profile_enable(int(bool(on))), "fm_profile_enable")


def profile_read():
    """{kernel name: (total device ms, launches)} since the last read; clears."""
    from ._abi import KERNEL_IDS
    ms = (ctypes.c_double * KERNEL_IDS)()
    n = (ctypes.c_int * KERNEL_IDS)()
    check(lib().fm_profile_read(ms, n, KERNEL_IDS), "fm_profile_read")
    return {lib().fm_kernel_name(i).decode(): (ms[i], n[i]) for i in range(KERNEL_IDS)}


def measure_exp2_rate(stream=None) -> float:
    """exp2 evaluations per second of this GPU (ex2.approx.f32, all SMs)."""
    out = ctypes.c_double(0.0)
    check(lib().fm_measure_exp2_rate(ctypes.byref(out), _stream_ptr(stream)),
          "fm_measure_exp2_rate")
    return out.value

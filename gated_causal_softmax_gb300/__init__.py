"""Python binding of libgcs_attn (GB300 / sm_103a gated causal softmax attention).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  PyTorch provides device memory (outputs and workspace are allocated here with
the caching allocator) and the current stream.  There is no CPU or PyTorch fallback: if
the library cannot be built or loaded, every call raises.

Entry points (same names as the C ABI in include/gcs_attn.h):
    attn_fwd(q, k, v, cu_seqlens, ...)           -> (o, lse)
    attn_bwd(q, k, v, o, lse, dout, cu_seqlens, ...) -> (dq, dk, dv, dlog_gate, dsink)
    attn_decode_paged(q, k_cache, v_cache, ...)  -> out
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

__all__ = [
    "load",
    "lib",
    "attn_fwd",
    "attn_bwd",
    "attn_decode_paged",
    "attn_decode_paged_noalloc",
    "attn_prefill_paged",
    "selftest_bounded_wait",
    "set_device_checks",
    "device_checks",
    "check_prefill_inputs",
    "check_paged_inputs",
    "PrefillArgs",
    "DecodeArgs",
    "GcsError",
    "get_device_status",
    "set_kernel_events",
    "STATUS",
]

STATUS = {
    0: "GCS_OK",
    1: "GCS_ERR_INVALID_ARG",
    2: "GCS_ERR_UNSUPPORTED",
    3: "GCS_ERR_WORKSPACE",
    4: "GCS_ERR_CUDA",
    5: "GCS_ERR_DEVICE_TIMEOUT",
}

_c_int, _c_float, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
_i64 = ctypes.c_int64


class Strides(ctypes.Structure):
    """gcs_strides: element strides (token, head) of a [tokens, heads, dim] tensor; (0, 0) =
    contiguous."""
    _fields_ = [("token", _i64), ("head", _i64)]


class PrefillArgs(ctypes.Structure):
    _fields_ = [
        ("num_seqs", _c_int),
        ("cu_seqlens", _vp),
        ("total_tokens", _c_int),
        ("max_seqlen", _c_int),
        ("hq", _c_int),
        ("hkv", _c_int),
        ("dqk", _c_int),
        ("dv", _c_int),
        ("scale", _c_float),
        ("window", _c_int),
        ("q", _vp),
        ("k", _vp),
        ("v", _vp),
        ("log_gate", _vp),
        ("sink", _vp),
        ("deterministic", _c_int),
        ("q_stride", Strides),
        ("k_stride", Strides),
        ("v_stride", Strides),
        ("o_stride", Strides),
        ("do_stride", Strides),
        ("dq_stride", Strides),
        ("dk_stride", Strides),
        ("dv_stride", Strides),
    ]


class DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("num_reqs", _c_int),
        ("cu_q", _vp),
        ("total_q", _c_int),
        ("max_q_len", _c_int),
        ("seq_lens", _vp),
        ("max_seq_len", _c_int),
        ("block_table", _vp),
        ("max_blocks_per_req", _c_int),
        ("k_cache", _vp),
        ("v_cache", _vp),
        ("k_scale", _vp),
        ("v_scale", _vp),
        ("num_blocks", _c_int),
        ("block_size", _c_int),
        ("hq", _c_int),
        ("hkv", _c_int),
        ("d", _c_int),
        ("scale", _c_float),
        ("segment_len", _c_int),
        ("q", _vp),
        ("kv_format", _c_int),
        ("scale_mode", _c_int),
        ("g_cache", _vp),
        ("sink", _vp),
        ("window", _c_int),
        ("q_stride", Strides),
        ("out_stride", Strides),
        ("kv_stride_block", _i64),
        ("kv_stride_head", _i64),
        ("kv_stride_slot", _i64),
    ]


KV_FP8_E4M3, KV_BF16 = 0, 1
SCALE_PER_TOKEN, SCALE_PER_TENSOR = 0, 1


class GcsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


_LIB: Optional[ctypes.CDLL] = None


def _declare(lib: ctypes.CDLL) -> None:
    P = ctypes.POINTER
    lib.gcs_status_str.argtypes = [_c_int]
    lib.gcs_status_str.restype = ctypes.c_char_p
    lib.gcs_version.argtypes = []
    lib.gcs_version.restype = ctypes.c_char_p
    lib.attn_fwd_workspace.argtypes = [P(PrefillArgs)]
    lib.attn_fwd_workspace.restype = ctypes.c_size_t
    lib.attn_bwd_workspace.argtypes = [P(PrefillArgs)]
    lib.attn_bwd_workspace.restype = ctypes.c_size_t
    lib.attn_decode_workspace.argtypes = [P(DecodeArgs)]
    lib.attn_decode_workspace.restype = ctypes.c_size_t
    lib.attn_fwd.argtypes = [P(PrefillArgs), _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.attn_fwd.restype = _c_int
    lib.attn_bwd.argtypes = [P(PrefillArgs), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.attn_bwd.restype = _c_int
    lib.attn_decode_paged.argtypes = [P(DecodeArgs), _vp, _vp, ctypes.c_size_t, _vp]
    lib.attn_decode_paged.restype = _c_int
    lib.attn_decode_paged_noalloc.argtypes = [P(DecodeArgs), _vp, _vp]
    lib.attn_decode_paged_noalloc.restype = _c_int
    lib.attn_prefill_paged_workspace.argtypes = [P(DecodeArgs)]
    lib.attn_prefill_paged_workspace.restype = ctypes.c_size_t
    lib.attn_prefill_paged.argtypes = [P(DecodeArgs), _vp, _vp, ctypes.c_size_t, _vp]
    lib.attn_prefill_paged.restype = _c_int
    lib.gcs_get_device_status.argtypes = [P(_c_int), _c_int]
    lib.gcs_get_device_status.restype = _c_int
    lib.gcs_selftest_bounded_wait.argtypes = [_vp]
    lib.gcs_selftest_bounded_wait.restype = _c_int
    lib.gcs_set_kernel_events.argtypes = [_vp, _vp]
    lib.gcs_set_kernel_events.restype = _c_int
    lib.gcs_set_device_checks.argtypes = [_c_int]
    lib.gcs_set_device_checks.restype = _c_int
    lib.gcs_get_device_checks.argtypes = []
    lib.gcs_get_device_checks.restype = _c_int
    lib.gcs_check_prefill_inputs.argtypes = [P(PrefillArgs), _vp]
    lib.gcs_check_prefill_inputs.restype = _c_int
    lib.gcs_check_paged_inputs.argtypes = [P(DecodeArgs), _vp]
    lib.gcs_check_paged_inputs.restype = _c_int


def load(build_if_needed: bool = True) -> ctypes.CDLL:
    """Load (building first if the library is missing or stale) libgcs_attn.so."""
    global _LIB
    if _LIB is not None:
        return _LIB
    from . import build as _build

    path = _build.LIB
    if build_if_needed:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libgcs_attn.so not found at {path}; run gated_causal_softmax_gb300.build.build()")
    lib = ctypes.CDLL(path)
    _declare(lib)
    _LIB = lib
    return lib


def lib() -> ctypes.CDLL:
    return load()


def _check(status: int, what: str) -> None:
    if status == 0:
        return
    if status == 2:
        raise NotImplementedError(f"{what}: {STATUS[2]}")
    raise GcsError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _need(t: torch.Tensor, dtype, name: str, strided: bool = False) -> torch.Tensor:
    """Checks device, dtype and layout: contiguous, or (strided=True) any layout whose last
    dimension is contiguous (the library validates the other strides)."""
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if strided:
        if t.stride(-1) != 1:
            raise ValueError(f"{name} must have a contiguous last dimension")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _st(t: Optional[torch.Tensor]) -> Strides:
    """Token and head strides of a [tokens, heads, dim] tensor."""
    if t is None:
        return Strides(0, 0)
    if t.dim() != 3:
        raise ValueError("expected a [tokens, heads, dim] tensor")
    return Strides(t.stride(0), t.stride(1))


def set_kernel_events(before: Optional[torch.cuda.Event], after: Optional[torch.cuda.Event]) -> None:
    """Arm two recorded-once torch CUDA events around the main kernel of the next call."""
    h = lambda e: None if e is None else e.cuda_event
    _check(load().gcs_set_kernel_events(h(before), h(after)), "gcs_set_kernel_events")


def get_device_status(clear: bool = True) -> int:
    """Per-device status word: GCS_ERR_DEVICE_TIMEOUT (5) from a kernel that gave up on a bounded
    wait, GCS_ERR_INVALID_ARG (1) from a failed device-content check, else 0."""
    st = _c_int(0)
    _check(load().gcs_get_device_status(ctypes.byref(st), 1 if clear else 0), "gcs_get_device_status")
    return st.value


def selftest_bounded_wait() -> int:
    """Runs the bounded-wait self-test kernel on the current stream, waits for it and returns
    (and clears) the device status word: GCS_ERR_DEVICE_TIMEOUT (5) when the wait gave up."""
    _check(load().gcs_selftest_bounded_wait(_stream()), "gcs_selftest_bounded_wait")
    torch.cuda.synchronize()
    return get_device_status(clear=True)


def set_device_checks(enable: bool) -> None:
    """Checked mode for every later call of this process: each call first checks its index
    arrays on the device; a failed check records GCS_ERR_INVALID_ARG (1) in the device status
    word and the call's kernels see an empty batch."""
    _check(load().gcs_set_device_checks(1 if enable else 0), "gcs_set_device_checks")


def device_checks() -> bool:
    return bool(load().gcs_get_device_checks())


def check_prefill_inputs(q, k, v, cu_seqlens, max_seqlen=None, scale=None, window=0, log_gate=None,
                         sink=None) -> None:
    """Launches the device-content checks of a prefill call's cu_seqlens on the current stream
    (nothing else); read the result with get_device_status()."""
    a = prefill_args(q, k, v, cu_seqlens, max_seqlen, scale, window, log_gate, sink)
    _check(load().gcs_check_prefill_inputs(ctypes.byref(a), _stream()), "gcs_check_prefill_inputs")


def check_paged_inputs(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, max_q_len, max_seq_len,
                       scale=None, segment_len=0, g_cache=None, sink=None, window=0) -> None:
    """Launches the device-content checks of a paged call's cu_q, seq_lens and page table on
    the current stream (nothing else); read the result with get_device_status()."""
    a = decode_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, max_q_len, max_seq_len,
                    scale, segment_len, g_cache, sink, window)
    _check(load().gcs_check_paged_inputs(ctypes.byref(a), _stream()), "gcs_check_paged_inputs")


def prefill_args(q, k, v, cu_seqlens, max_seqlen, scale, window, log_gate, sink) -> PrefillArgs:
    _need(q, torch.bfloat16, "q", strided=True)
    _need(k, torch.bfloat16, "k", strided=True)
    _need(v, torch.bfloat16, "v", strided=True)
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    if log_gate is not None:
        _need(log_gate, torch.float32, "log_gate")
    if sink is not None:
        _need(sink, torch.float32, "sink")
    tot, hq, dqk = q.shape
    hkv, dv = k.shape[1], v.shape[2]
    if max_seqlen is None:
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max())
    if scale is None:
        scale = 1.0 / math.sqrt(dqk)
    return PrefillArgs(
        num_seqs=cu_seqlens.numel() - 1,
        cu_seqlens=cu_seqlens.data_ptr(),
        total_tokens=tot,
        max_seqlen=int(max_seqlen),
        hq=hq,
        hkv=hkv,
        dqk=dqk,
        dv=dv,
        scale=float(scale),
        window=int(window),
        q=q.data_ptr(),
        k=k.data_ptr(),
        v=v.data_ptr(),
        log_gate=_ptr(log_gate),
        sink=_ptr(sink),
        q_stride=_st(q),
        k_stride=_st(k),
        v_stride=_st(v),
    )


def attn_fwd(q, k, v, cu_seqlens, max_seqlen=None, scale=None, window=0, log_gate=None, sink=None, out=None,
             lse=None, workspace=None):
    """Prefill forward.  q [tot, hq, dqk], k [tot, hkv, dqk], v [tot, hkv, dv] bf16;
    cu_seqlens int32 [num_seqs + 1]; log_gate fp32 [tot, hq] or None; sink fp32 [hq] or None.
    Returns o bf16 [tot, hq, dv] and lse fp32 [hq, tot]."""
    L = load()
    a = prefill_args(q, k, v, cu_seqlens, max_seqlen, scale, window, log_gate, sink)
    tot, hq, _ = q.shape
    if out is None:
        out = torch.empty((tot, hq, v.shape[2]), dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, "out", strided=True)
    a.o_stride = _st(out)
    if lse is None:
        lse = torch.empty((hq, tot), dtype=torch.float32, device=q.device)
    ws_bytes = L.attn_fwd_workspace(ctypes.byref(a))
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = L.attn_fwd(ctypes.byref(a), out.data_ptr(), lse.data_ptr(), _ptr(workspace),
                    workspace.numel() if workspace is not None else 0, _stream())
    _check(st, "attn_fwd")
    return out, lse


def attn_bwd(q, k, v, o, lse, dout, cu_seqlens, max_seqlen=None, scale=None, window=0, log_gate=None, sink=None,
             workspace=None, dq=None, dk=None, dv=None, dlog_gate=None, dsink=None, deterministic=False):
    """Prefill backward of sum(O * dO).  Returns dq, dk, dv (bf16), dlog_gate fp32 [tot, hq]
    (None without gates) and dsink fp32 [hq] (None without sink).  deterministic=True makes
    head dims above 128 take the fixed-order route (dims <= 128 always do)."""
    L = load()
    a = prefill_args(q, k, v, cu_seqlens, max_seqlen, scale, window, log_gate, sink)
    a.deterministic = 1 if deterministic else 0
    _need(o, torch.bfloat16, "o", strided=True)
    _need(dout, torch.bfloat16, "dout", strided=True)
    _need(lse, torch.float32, "lse")
    new = lambda t: torch.empty(t.shape, dtype=t.dtype, device=t.device)
    dq = new(q) if dq is None else _need(dq, torch.bfloat16, "dq", strided=True)
    dk = new(k) if dk is None else _need(dk, torch.bfloat16, "dk", strided=True)
    dv = new(v) if dv is None else _need(dv, torch.bfloat16, "dv", strided=True)
    a.o_stride, a.do_stride = _st(o), _st(dout)
    a.dq_stride, a.dk_stride, a.dv_stride = _st(dq), _st(dk), _st(dv)
    if log_gate is not None and dlog_gate is None:
        dlog_gate = torch.empty_like(log_gate)
    if sink is not None and dsink is None:
        dsink = torch.empty_like(sink)
    ws_bytes = L.attn_bwd_workspace(ctypes.byref(a))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    st = L.attn_bwd(ctypes.byref(a), o.data_ptr(), lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                    dv.data_ptr(), _ptr(dlog_gate), _ptr(dsink), workspace.data_ptr(), workspace.numel(), _stream())
    _check(st, "attn_bwd")
    return dq, dk, dv, dlog_gate, dsink


def decode_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, max_q_len, max_seq_len, scale,
                segment_len, g_cache=None, sink=None, window=0) -> DecodeArgs:
    """Marshals the decode arguments.  The cache format follows the cache dtype (fp8 e4m3 as
    uint8 or float8_e4m3fn, or bf16); fp8 scales are per token when they have the page shape
    [num_blocks, num_kv_heads, block_size] and per tensor when they hold one value; a bf16
    cache takes no scales.  Any other scale shape raises NotImplementedError.

    q may be strided (last dim contiguous).  The caches are [num_blocks, num_kv_heads,
    block_size, d] views with any strides the library accepts, shared by K and V: a
    [num_blocks, block_size, num_kv_heads, d] cache is passed as cache.permute(0, 2, 1, 3)."""
    _need(q, torch.bfloat16, "q", strided=True)
    if k_cache.dtype == torch.float8_e4m3fn:
        k_cache = k_cache.view(torch.uint8)
    if v_cache.dtype == torch.float8_e4m3fn:
        v_cache = v_cache.view(torch.uint8)
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(cu_q, torch.int32, "cu_q")
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache shapes differ")
    if k_cache.stride() != v_cache.stride():
        raise ValueError("k_cache and v_cache must share one layout")
    nb, hkv, bs, d = k_cache.shape
    if k_cache.dtype == torch.bfloat16:
        _need(k_cache, torch.bfloat16, "k_cache", strided=True)
        _need(v_cache, torch.bfloat16, "v_cache", strided=True)
        if k_scale is not None or v_scale is not None:
            raise ValueError("a bf16 KV cache takes no scales")
        kv_format, scale_mode, ks_ptr, vs_ptr = KV_BF16, SCALE_PER_TOKEN, None, None
    else:
        _need(k_cache, torch.uint8, "k_cache", strided=True)
        _need(v_cache, torch.uint8, "v_cache", strided=True)
        _need(k_scale, torch.float32, "k_scale")
        _need(v_scale, torch.float32, "v_scale")
        if tuple(k_scale.shape) == (nb, hkv, bs) and tuple(v_scale.shape) == (nb, hkv, bs):
            scale_mode = SCALE_PER_TOKEN
        elif k_scale.numel() == 1 and v_scale.numel() == 1:
            scale_mode = SCALE_PER_TENSOR
        else:
            raise NotImplementedError("fp8 scales must have the page shape [num_blocks, num_kv_heads, block_size] "
                                      "(per token) or hold one value (per tensor)")
        kv_format, ks_ptr, vs_ptr = KV_FP8_E4M3, k_scale.data_ptr(), v_scale.data_ptr()
    if g_cache is not None:
        _need(g_cache, torch.float32, "g_cache")
        if tuple(g_cache.shape) != (nb, q.shape[1], bs):
            raise ValueError("g_cache must be [num_blocks, num_q_heads, block_size]")
    if sink is not None:
        _need(sink, torch.float32, "sink")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return DecodeArgs(
        num_reqs=seq_lens.numel(),
        cu_q=cu_q.data_ptr(),
        total_q=q.shape[0],
        max_q_len=int(max_q_len),
        seq_lens=seq_lens.data_ptr(),
        max_seq_len=int(max_seq_len),
        block_table=block_table.data_ptr(),
        max_blocks_per_req=block_table.shape[1],
        k_cache=k_cache.data_ptr(),
        v_cache=v_cache.data_ptr(),
        k_scale=ks_ptr,
        v_scale=vs_ptr,
        num_blocks=nb,
        block_size=bs,
        hq=q.shape[1],
        hkv=hkv,
        d=d,
        scale=float(scale),
        segment_len=int(segment_len),
        q=q.data_ptr(),
        kv_format=kv_format,
        scale_mode=scale_mode,
        g_cache=None if g_cache is None else g_cache.data_ptr(),
        sink=None if sink is None else sink.data_ptr(),
        window=int(window),
        q_stride=_st(q),
        kv_stride_block=k_cache.stride(0),
        kv_stride_head=k_cache.stride(1),
        kv_stride_slot=k_cache.stride(2),
    )


def attn_decode_paged(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, max_q_len, max_seq_len,
                      scale=None, segment_len=2048, out=None, workspace=None, g_cache=None, sink=None, window=0):
    """Paged decode.  q bf16 [total_q, hq, d]; caches fp8 e4m3 (uint8 or float8_e4m3fn) or bf16
    [num_blocks, hkv, block_size, d]; fp8 scales fp32 [num_blocks, hkv, block_size] (per token)
    or one value each (per tensor), None for bf16; block_table int32 [R, max_blocks]; seq_lens
    int32 [R]; cu_q int32 [R + 1].  Optional decoding features: g_cache fp32 [num_blocks, hq,
    block_size] cumulative log gates, sink fp32 [hq], window (0 = none)."""
    L = load()
    a = decode_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, max_q_len, max_seq_len,
                    scale, segment_len, g_cache, sink, window)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    a.out_stride = _st(_need(out, torch.bfloat16, "out", strided=True))
    ws_bytes = L.attn_decode_workspace(ctypes.byref(a))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    st = L.attn_decode_paged(ctypes.byref(a), out.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream())
    _check(st, "attn_decode_paged")
    return out


def attn_prefill_paged(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, max_q_len, max_seq_len,
                       scale=None, segment_len=0, out=None, workspace=None, g_cache=None, sink=None, window=0):
    """Paged chunked prefill: like attn_decode_paged, but a request's q_len may be anything
    from 1 to its seq_len (its query rows are the last q_len cached positions).  fp8 e4m3
    cache with per-token or per-tensor scales.  segment_len 0 lets the library choose the
    split of the context (no workspace when it needs none); otherwise a multiple of 128."""
    L = load()
    a = decode_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, max_q_len, max_seq_len,
                    scale, segment_len, g_cache, sink, window)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    a.out_stride = _st(_need(out, torch.bfloat16, "out", strided=True))
    ws_bytes = L.attn_prefill_paged_workspace(ctypes.byref(a))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    st = L.attn_prefill_paged(ctypes.byref(a), out.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream())
    _check(st, "attn_prefill_paged")
    return out


def attn_decode_paged_noalloc(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, max_q_len,
                              max_seq_len, scale=None, segment_len=2048, out=None, g_cache=None, sink=None, window=0):
    """attn_decode_paged without a workspace: the library keeps the split-K partials in
    its own fixed 64 MiB device scratch (for callers that cannot allocate device memory).
    Calls share that scratch, so calls must not overlap on the GPU."""
    L = load()
    a = decode_args(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, cu_q, max_q_len, max_seq_len,
                    scale, segment_len, g_cache, sink, window)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    a.out_stride = _st(_need(out, torch.bfloat16, "out", strided=True))
    _check(L.attn_decode_paged_noalloc(ctypes.byref(a), out.data_ptr(), _stream()), "attn_decode_paged_noalloc")
    return out


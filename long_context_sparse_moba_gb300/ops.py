"""Python binding of ``libmoba_gb300.so`` (argument marshalling only).

Every function below calls the C ABI of ``include/moba.h`` with the tensors'
device pointers and the current CUDA stream; all arithmetic runs in the
library's kernels.  There is no fallback: if the library is missing or a call
fails, a ``RuntimeError`` is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoba_gb300.so")

MOBA_OK = 0
MOBA_ERR_INVALID_ARG = 1
MOBA_ERR_UNSUPPORTED = 2
MOBA_ERR_CUDA = 3
MOBA_ERR_WORKSPACE = 4
MOBA_ERR_TIMEOUT = 5

_lib = None

_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGNATURES = {
    "moba_num_blocks": (_I, [_I, _I]),
    "moba_status_string": (ctypes.c_char_p, [_I]),
    "moba_last_cuda_error": (ctypes.c_char_p, []),
    "moba_kpool": (_I, [_P, _P, _I, _I, _I, _I, _I, _P]),
    "moba_kpool_varlen": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moba_gate_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "moba_gate_topk_varlen": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "moba_attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "moba_attn_fwd_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moba_attn_fwd_ws": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "moba_attn_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "moba_attn_fwd_varlen_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "moba_attn_fwd_varlen_ws": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                     _P, _SZ, _P]),
    "moba_get_status": (_I, [_P]),
    "moba_launch_count": (ctypes.c_ulonglong, []),
    "moba_decode_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "moba_decode_workspace_size": (_SZ, [_I, _I, _I, _I]),
    "moba_decode_fwd_ws": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ,
                                _P]),
    "moba_attn_fwd_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "moba_attn_fwd_noalloc_capacity": (_SZ, []),
    "moba_debug_timeout_info": (None, [_P]),
    "moba_attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "moba_attn_bwd_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moba_attn_bwd_ws": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P,
                              _SZ, _P]),
    "moba_attn_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                  _I, _I, _P]),
    "moba_attn_bwd_varlen_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "moba_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moba_kpool_ex": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moba_kpool_varlen_ex": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moba_gate_topk_ex": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "moba_gate_topk_varlen_ex": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "moba_attn_fwd_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moba_attn_fwd_host": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P]),
    "moba_attn_fwd_host_scratch_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moba_attn_fwd_varlen_ex": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                                     _P, _SZ, _P]),
    "moba_attn_bwd_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P,
                              _P, _SZ, _P]),
    "moba_attn_bwd_varlen_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                     _I, _I, _I, _P, _P, _SZ, _P]),
}

POOL_MEAN = 0
POOL_MAX = 1
GATE_TCGEN05 = 0
GATE_CUDA_CORES = 1
ATTN_TCGEN05 = 0
ATTN_MMA_SYNC = 1
SCHEDULE_ADAPTIVE = 0
SCHEDULE_BLOCK_MAJOR = 1


class Options(ctypes.Structure):
    """``moba_options_t``: per-call options (all zero = the defaults)."""
    _fields_ = [("pooling", ctypes.c_int), ("gate_kernel", ctypes.c_int),
                ("attn_kernel", ctypes.c_int), ("debug_flags", ctypes.c_int),
                ("wait_limit_cycles", ctypes.c_longlong), ("idx_out", ctypes.c_void_p),
                ("phase_events", ctypes.c_void_p), ("schedule", ctypes.c_int),
                ("idx_in", ctypes.c_void_p)]


def _options(pooling=POOL_MEAN, gate_kernel=GATE_TCGEN05, attn_kernel=ATTN_TCGEN05,
             debug_flags=0, wait_limit_cycles=0, idx_out=None, phase_events=None,
             schedule=SCHEDULE_ADAPTIVE, idx_in=None):
    """An Options structure and the objects that must outlive the call."""
    o = Options(int(pooling), int(gate_kernel), int(attn_kernel), int(debug_flags),
                int(wait_limit_cycles), None, None, int(schedule), None)
    keep = []
    if idx_out is not None:
        o.idx_out = idx_out.data_ptr()
    if idx_in is not None:
        if idx_in.dtype != torch.int32 or not idx_in.is_cuda or not idx_in.is_contiguous():
            raise ValueError("idx_in must be a contiguous int32 CUDA tensor")
        o.idx_in = idx_in.data_ptr()
    if phase_events is not None:
        if len(phase_events) != len(PHASES) + 1:
            raise ValueError(f"phase_events needs {len(PHASES) + 1} events")
        arr = (ctypes.c_void_p * len(phase_events))()
        for i, ev in enumerate(phase_events):
            arr[i] = ev.cuda_event
        o.phase_events = ctypes.cast(arr, ctypes.c_void_p)
        keep.append(arr)
    return o, keep

PHASES = ("tables", "kpool", "gate", "regroup", "attn_past", "attn_current")


def phase_events(stream=None):
    """Seven timing events for the forward's ``phase_events`` option, created on
    the stream (torch creates an event's CUDA handle at its first record)."""
    st = stream if stream is not None else torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(PHASES) + 1)]
    for e in evs:
        e.record(st)
    return evs


def phase_ms(events) -> dict:
    """{phase: ms} between the recorded events (synchronises the last one)."""
    events[-1].synchronize()
    return {name: events[i].elapsed_time(events[i + 1]) for i, name in enumerate(PHASES)}


def lib():
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m long_context_sparse_moba_gb300.build` (needs nvcc)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(code: int) -> str:
    return lib().moba_status_string(code).decode()


def _check(code: int, what: str):
    if code != MOBA_OK:
        extra = ""
        if code == MOBA_ERR_CUDA:
            extra = ": " + lib().moba_last_cuda_error().decode()
        raise RuntimeError(f"{what} failed: {status_string(code)} ({code}){extra}")


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, dtype, name):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def _out(t, shape, dtype, like, name):
    """A result buffer: a new tensor on like's device, or the caller's one
    after checking its dtype, layout, shape and device."""
    shape = tuple(int(x) for x in shape)
    if t is None:
        return torch.empty(shape, dtype=dtype, device=like.device)
    _need(t, dtype, name)
    if tuple(t.shape) != shape or t.device != like.device:
        raise ValueError(f"{name} must have shape {shape} on {like.device}")
    return t


def _ws(workspace):
    if workspace is not None:
        _need(workspace, torch.uint8, "workspace")
    return workspace


def num_blocks(length: int, block_size: int) -> int:
    return int(lib().moba_num_blocks(int(length), int(block_size)))


def _nb_total(cu_host, block_size):
    return sum(num_blocks(cu_host[b + 1] - cu_host[b], block_size) for b in range(len(cu_host) - 1))


def kpool(k, block_size: int, stream=None, pooling=POOL_MEAN):
    """Pooled keys of k [B, S, H, D] -> kbar [B * n, H, D] fp32 (mean, or the
    element-wise maximum with ``pooling=POOL_MAX``)."""
    _need(k, torch.bfloat16, "k")
    B, S, H, D = k.shape
    kbar = torch.empty(B * num_blocks(S, block_size), H, D, dtype=torch.float32, device=k.device)
    o, _keep = _options(pooling=pooling)
    _check(lib().moba_kpool_ex(_ptr(k), _ptr(kbar), B, H, S, D, block_size, ctypes.byref(o),
                               _stream(stream)), "moba_kpool")
    return kbar


def kpool_varlen(k, cu_seqlens, block_size: int, stream=None, pooling=POOL_MEAN):
    """Varlen k [total, H, D], cu_seqlens int32 CUDA [num_seqs + 1]."""
    _need(k, torch.bfloat16, "k")
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    total, H, D = k.shape
    nb = _nb_total(cu_seqlens.tolist(), block_size)
    kbar = torch.empty(nb, H, D, dtype=torch.float32, device=k.device)
    o, _keep = _options(pooling=pooling)
    _check(lib().moba_kpool_varlen_ex(_ptr(k), _ptr(kbar), _ptr(cu_seqlens),
                                      cu_seqlens.numel() - 1, total, H, D, block_size,
                                      ctypes.byref(o), _stream(stream)), "moba_kpool_varlen")
    return kbar


def gate_topk(q, kbar, block_size: int, topk: int, stream=None, gate_kernel=GATE_TCGEN05):
    """Selected blocks idx [B, S, H, topk] int32 (ascending, -1 padded)."""
    _need(q, torch.bfloat16, "q")
    _need(kbar, torch.float32, "kbar")
    B, S, H, D = q.shape
    if block_size > 0 and tuple(kbar.shape) != (B * num_blocks(S, block_size), H, D):
        raise ValueError("kbar must be [B * ceil(S / block_size), H, D] (as kpool returns it)")
    idx = torch.empty(B, S, H, topk, dtype=torch.int32, device=q.device)
    o, _keep = _options(gate_kernel=gate_kernel)
    _check(lib().moba_gate_topk_ex(_ptr(q), _ptr(kbar), _ptr(idx), B, H, S, D, block_size, topk,
                                   ctypes.byref(o), _stream(stream)), "moba_gate_topk")
    return idx


def gate_topk_varlen(q, kbar, cu_seqlens, block_size: int, topk: int, stream=None,
                     gate_kernel=GATE_TCGEN05):
    _need(q, torch.bfloat16, "q")
    _need(kbar, torch.float32, "kbar")
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    total, H, D = q.shape
    idx = torch.empty(total, H, topk, dtype=torch.int32, device=q.device)
    o, _keep = _options(gate_kernel=gate_kernel)
    _check(lib().moba_gate_topk_varlen_ex(_ptr(q), _ptr(kbar), _ptr(idx), _ptr(cu_seqlens),
                                          cu_seqlens.numel() - 1, total, H, D, block_size, topk,
                                          ctypes.byref(o), _stream(stream)),
           "moba_gate_topk_varlen")
    return idx


def workspace_size(B, H, S, D, block_size, topk) -> int:
    return int(lib().moba_attn_fwd_workspace_size(B, H, S, D, block_size, topk))


def varlen_workspace_size(num_seqs, total, max_seqlen, H, D, block_size, topk) -> int:
    return int(lib().moba_attn_fwd_varlen_workspace_size(num_seqs, total, max_seqlen, H, D,
                                                         block_size, topk))


def _idx_buffer(idx_out, rows_shape, topk, like):
    if idx_out is None:
        return None
    return _out(idx_out, (*rows_shape, topk), torch.int32, like, "idx_out")


def attn_fwd(q, k, v, block_size: int, topk: int, out=None, lse=None, workspace=None,
             stream=None, idx_out=None, phase_events=None, **options):
    """MoBA forward for q, k, v [B, S, H, D] bf16 -> (out [B, S, H, D] bf16, lse [B, H, S] fp32).

    With ``workspace`` (a uint8 CUDA tensor of at least :func:`workspace_size`
    bytes) the call allocates nothing; otherwise the library allocates its
    scratch stream-ordered.  ``idx_out`` ([B, S, H, topk] int32) receives the
    selection the call used; ``phase_events`` (see :func:`phase_events`) are
    recorded between its phases; further keyword ``options`` (pooling,
    gate_kernel, attn_kernel, debug_flags, wait_limit_cycles) are per call."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    B, S, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape")
    out = _out(out, q.shape, torch.bfloat16, q, "out")
    lse = _out(lse, (B, H, S), torch.float32, q, "lse")
    workspace = _ws(workspace)
    idx_out = _idx_buffer(idx_out, (B, S, H), topk, q)
    o, _keep = _options(idx_out=idx_out, phase_events=phase_events, **options)
    rc = lib().moba_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, S, D,
                                block_size, topk, ctypes.byref(o), _ptr(workspace),
                                workspace.numel() if workspace is not None else 0,
                                _stream(stream))
    _check(rc, "moba_attn_fwd")
    return out, lse


def host_scratch_size(B: int, H: int, S: int, D: int, block_size: int, topk: int) -> int:
    """Bytes of device scratch :func:`attn_fwd_host` needs."""
    return int(lib().moba_attn_fwd_host_scratch_size(B, H, S, D, block_size, topk))


def attn_fwd_host(q, k, v, block_size: int, topk: int, out, lse, scratch, stream=None,
                  **options):
    """The forward on host tensors (page-locked for asynchronous copies): q, k,
    v [B, S, H, D] bf16 in, out [B, S, H, D] bf16 and lse [B, H, S] fp32 filled
    in once ``stream`` has reached the end of the call's work.  ``scratch`` is a
    uint8 CUDA tensor of at least :func:`host_scratch_size` bytes; the library
    copies the inputs in and the results out itself."""
    for t, n, dt in ((q, "q", torch.bfloat16), (k, "k", torch.bfloat16),
                     (v, "v", torch.bfloat16), (out, "out", torch.bfloat16),
                     (lse, "lse", torch.float32)):
        if t.dtype != dt or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host {dt} tensor")
    B, S, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or out.shape != q.shape or \
            tuple(lse.shape) != (B, H, S):
        raise ValueError("q, k, v, out must be [B, S, H, D] and lse [B, H, S]")
    _need(scratch, torch.uint8, "scratch")
    o, _keep = _options(**options)
    rc = lib().moba_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, S, D,
                                  block_size, topk, ctypes.byref(o), _ptr(scratch),
                                  scratch.numel(), _stream(stream))
    _check(rc, "moba_attn_fwd_host")
    return out, lse


def decode_workspace_size(B: int, H: int, D: int, topk: int) -> int:
    return int(lib().moba_decode_workspace_size(B, H, D, topk))


def decode_fwd(q, k_cache, v_cache, kbar, cache_lens, block_size: int, topk: int, out=None,
               lse=None, idx=None, workspace=None, stream=None):
    """One decode step: q [B, H, D] bf16 against k_cache, v_cache [B, S_max, H,
    D] bf16 (the new token already at position cache_lens[b] - 1), kbar the
    caches' pooled keys (:func:`kpool` of k_cache), cache_lens int32 [B] on the
    device -> (out [B, H, D] bf16, lse [B, H] fp32, idx [B, H, topk] int32)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, n)
    _need(kbar, torch.float32, "kbar")
    _need(cache_lens, torch.int32, "cache_lens")
    B, H, D = q.shape
    if k_cache.dim() != 4 or k_cache.shape[0] != B or k_cache.shape[2:] != (H, D) or \
            v_cache.shape != k_cache.shape:
        raise ValueError("k_cache, v_cache must be [B, S_max, H, D] matching q")
    S_max = k_cache.shape[1]
    if block_size > 0 and tuple(kbar.shape) != (B * num_blocks(S_max, block_size), H, D):
        raise ValueError("kbar must be [B * ceil(S_max / block_size), H, D] (kpool of k_cache)")
    out = _out(out, q.shape, torch.bfloat16, q, "out")
    lse = _out(lse, (B, H), torch.float32, q, "lse")
    idx = _out(idx, (B, H, topk), torch.int32, q, "idx")
    workspace = _ws(workspace)
    st = _stream(stream)
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kbar), _ptr(cache_lens), _ptr(out),
            _ptr(lse), _ptr(idx), B, H, S_max, D, block_size, topk)
    if workspace is None:
        rc = lib().moba_decode_fwd(*args, st)
    else:
        rc = lib().moba_decode_fwd_ws(*args, _ptr(workspace), workspace.numel(), st)
    _check(rc, "moba_decode_fwd")
    return out, lse, idx


def attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, block_size: int, topk: int, out=None,
                    lse=None, workspace=None, stream=None, idx_out=None, phase_events=None,
                    **options):
    """Varlen MoBA forward: q, k, v [total, H, D] bf16, cu_seqlens int32 CUDA
    [num_seqs + 1] -> (out [total, H, D] bf16, lse [H, total] fp32).  Options
    as for :func:`attn_fwd` (``idx_out`` is [total, H, topk])."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    total, H, D = q.shape
    ns = cu_seqlens.numel() - 1
    for t, n in ((k, "k"), (v, "v")):
        if t.shape != q.shape:
            raise ValueError(f"{n} must have the shape of q")
    out = _out(out, q.shape, torch.bfloat16, q, "out")
    lse = _out(lse, (H, total), torch.float32, q, "lse")
    workspace = _ws(workspace)
    idx_out = _idx_buffer(idx_out, (total, H), topk, q)
    o, _keep = _options(idx_out=idx_out, phase_events=phase_events, **options)
    rc = lib().moba_attn_fwd_varlen_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                       _ptr(cu_seqlens), ns, total, max_seqlen, H, D,
                                       block_size, topk, ctypes.byref(o), _ptr(workspace),
                                       workspace.numel() if workspace is not None else 0,
                                       _stream(stream))
    _check(rc, "moba_attn_fwd_varlen")
    return out, lse


def bwd_workspace_size(B, H, S, D, block_size, topk) -> int:
    return int(lib().moba_attn_bwd_workspace_size(B, H, S, D, block_size, topk))


def attn_bwd(q, k, v, out, lse, dout, block_size: int, topk: int, dq=None, dk=None, dv=None,
             workspace=None, stream=None, **options):
    """MoBA backward for the forward ``attn_fwd(q, k, v, block_size, topk)``:
    q, k, v, out, dout [B, S, H, D] bf16 and lse [B, H, S] fp32 (as the forward
    returned them) -> (dq, dk, dv) [B, S, H, D] bf16.  The gate's selection is
    recomputed (with the same ``options`` as the forward) and held fixed, or,
    with ``idx_in`` ([B, S, H, topk] int32, the forward's ``idx_out``), taken
    as it is."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    B, S, H, D = q.shape
    for t, n in ((k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        if t.shape != q.shape:
            raise ValueError(f"{n} must have the shape of q")
    if tuple(lse.shape) != (B, H, S):
        raise ValueError("lse must be [B, H, S]")
    dq = _out(dq, q.shape, torch.bfloat16, q, "dq")
    dk = _out(dk, q.shape, torch.bfloat16, q, "dk")
    dv = _out(dv, q.shape, torch.bfloat16, q, "dv")
    workspace = _ws(workspace)
    o, _keep = _options(**options)
    rc = lib().moba_attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, H, S, D, block_size, topk,
                                ctypes.byref(o), _ptr(workspace),
                                workspace.numel() if workspace is not None else 0,
                                _stream(stream))
    _check(rc, "moba_attn_bwd")
    return dq, dk, dv


def attn_bwd_varlen(q, k, v, out, lse, dout, cu_seqlens, max_seqlen: int, block_size: int,
                    topk: int, stream=None, **options):
    """Varlen backward: q, k, v, out, dout [total, H, D] bf16, lse [H, total]
    fp32, cu_seqlens int32 CUDA [num_seqs + 1] -> (dq, dk, dv) [total, H, D]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    total, H, D = q.shape
    ns = cu_seqlens.numel() - 1
    for t, n in ((k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        if t.shape != q.shape:
            raise ValueError(f"{n} must have the shape of q")
    if tuple(lse.shape) != (H, total):
        raise ValueError("lse must be [H, total]")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    o, _keep = _options(**options)
    rc = lib().moba_attn_bwd_varlen_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                       _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens),
                                       ns, total, max_seqlen, H, D, block_size, topk,
                                       ctypes.byref(o), None, 0, _stream(stream))
    _check(rc, "moba_attn_bwd_varlen")
    return dq, dk, dv


def get_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(lib().moba_get_status(_stream(stream)))


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().moba_launch_count())


def attn_fwd_noalloc(q, k, v, block_size: int, topk: int, out, lse, stream=None):
    """moba_attn_fwd without any device allocation: the scratch is the
    library's static device array (see include/moba.h); `out` and `lse` must be
    provided by the caller."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, torch.bfloat16, n)
    _need(lse, torch.float32, "lse")
    B, S, H, D = q.shape
    for t, n in ((k, "k"), (v, "v"), (out, "out")):
        if t.shape != q.shape:
            raise ValueError(f"{n} must have the shape of q")
    if tuple(lse.shape) != (B, H, S):
        raise ValueError("lse must be [B, H, S]")
    _check(lib().moba_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, S,
                                       D, block_size, topk, _stream(stream)),
           "moba_attn_fwd_noalloc")
    return out, lse


def noalloc_capacity() -> int:
    return int(lib().moba_attn_fwd_noalloc_capacity())


def debug_timeout_info():
    """(barrier address, parity, block, thread) of the last reported timeout."""
    buf = (ctypes.c_int * 4)()
    lib().moba_debug_timeout_info(ctypes.cast(buf, ctypes.c_void_p))
    return tuple(buf)

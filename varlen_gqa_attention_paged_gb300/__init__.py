"""Unified paged varlen GQA attention for GB300 (sm_103a).

Python binding of the C ABI in ``include/ua.h``: it only turns torch tensors into
device pointers, the current CUDA stream and host-side sizes, and calls
``ua_unified_attention`` in ``libua.so``.  Every step of the computation runs in the
library's CUDA kernels; without the built library this module raises.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib
from ._lib import (UA_BACKEND_2D, UA_BACKEND_AUTO, UA_BACKEND_SPLIT, UA_DT_BF16, UA_DT_F8E4M3,
                   UA_DT_F16, UA_DT_F32, UA_PATH_2D, UA_PATH_SPLIT)

__all__ = ["unified_attention", "prepare", "PreparedAttention", "plan", "device_status",
           "device_status_reset", "UaError", "BACKENDS", "library_path"]

BACKENDS = {"auto": UA_BACKEND_AUTO, "2d": UA_BACKEND_2D, "split": UA_BACKEND_SPLIT}
_DTYPES = {torch.float16: UA_DT_F16, torch.bfloat16: UA_DT_BF16,
           torch.float8_e4m3fn: UA_DT_F8E4M3, torch.float32: UA_DT_F32}


class UaError(RuntimeError):
    def __init__(self, code: int, what: str):
        lib = _lib.load()
        super().__init__(f"{what}: {lib.ua_status_string(code).decode()} (status {code})")
        self.code = code


def library_path() -> str:
    return _lib.LIB_PATH


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _shape(q, k_cache, block_table, cu_seqlens_q, max_seqlen_q, max_seqlen_k, qq_bias,
           out_dtype_code, num_splits, workspace, events, k_scale_tok=None, v_scale_tok=None):
    sh = _lib.UaShape()
    sh.num_seqs = cu_seqlens_q.numel() - 1
    sh.total_q = q.shape[0]
    sh.max_seqlen_q = int(max_seqlen_q)
    sh.max_seqlen_k = int(max_seqlen_k)
    sh.max_blocks_per_seq = block_table.shape[-1]
    sh.num_blocks = k_cache.shape[0]
    sh.qq_bias_stride = qq_bias.shape[-1] if qq_bias is not None else 0
    sh.q_dtype = _dtype_code(q)
    sh.out_dtype = out_dtype_code
    sh.num_splits = int(num_splits)
    if workspace is not None:
        sh.workspace = workspace.data_ptr()
        sh.workspace_bytes = workspace.numel() * workspace.element_size()
    if events is not None:
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event lazily, on its first record
                e.record()
        arr = (ctypes.c_void_p * 3)(*[e.cuda_event for e in events])
        sh.events = ctypes.cast(arr, ctypes.c_void_p)
        sh._events_keepalive = arr  # noqa: SLF001 -- keep the array alive for the call
    if (k_scale_tok is None) != (v_scale_tok is None):
        raise ValueError("per-token scales: give both k_scale_tok and v_scale_tok, or neither")
    if k_scale_tok is not None:
        for t, ptr, strides in ((k_scale_tok, "k_scale_tok", "k_scale_stride"),
                                (v_scale_tok, "v_scale_tok", "v_scale_stride")):
            if t.dtype != torch.float32 or not t.is_cuda or t.dim() != 3:
                raise ValueError("per-token scales are float32 CUDA tensors [blocks, slots, H_kv]")
            if tuple(t.shape) != tuple(k_cache.shape[:3]):
                raise ValueError("per-token scales must be [num_blocks, block_size, H_kv]")
            setattr(sh, ptr, t.data_ptr())
            setattr(sh, strides, (ctypes.c_int64 * 3)(*t.stride()))
    return sh


def unified_attention(q, k_cache, v_cache, cu_seqlens_q, seq_lens_k, block_table, *,
                      max_seqlen_q: int, max_seqlen_k: int, scale: float | None = None,
                      softcap: float = 0.0, window_left: int = -1, alibi_slopes=None,
                      qq_bias=None, sinks=None, kv_scale=None, k_scale_tok=None,
                      v_scale_tok=None, out=None, out_dtype=None,
                      backend: str = "auto", num_splits: int = 0, workspace=None, stream=None,
                      events=None):
    """Paged varlen GQA attention on the GPU; returns ``out`` [total_q, H_q, D].

    q [total_q, H_q, D] f16/bf16; k_cache, v_cache [num_blocks, block_size, H_kv, D]
    f16/bf16/float8_e4m3fn; cu_seqlens_q [S+1], seq_lens_k [S], block_table [S, max_blocks]
    int32; alibi_slopes / sinks [H_q] and qq_bias [rows, stride] float32; kv_scale float32[2]
    (k_scale, v_scale) for the fp8 cache, or k_scale_tok / v_scale_tok float32 [num_blocks,
    block_size, H_kv] (any strides) for per-token fp8 scales.  max_seqlen_q / max_seqlen_k
    are host ints.
    """
    lib = _lib.load()
    total_q, hq, d = q.shape
    num_blocks, block_size, hkv, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape:
        raise ValueError("q, k_cache and v_cache disagree on shape")
    if qq_bias is not None and qq_bias.shape[0] < max_seqlen_q:
        raise ValueError("qq_bias needs at least max_seqlen_q rows")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("seq_lens_k", seq_lens_k),
                    ("block_table", block_table)):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 tensor")
    if not (q.is_cuda and k_cache.is_cuda and v_cache.is_cuda):
        raise ValueError("q, k_cache and v_cache must be CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=out_dtype or q.dtype, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sh = _shape(q, k_cache, block_table, cu_seqlens_q, max_seqlen_q, max_seqlen_k, qq_bias,
                _dtype_code(out), num_splits, workspace, events, k_scale_tok, v_scale_tok)
    rc = lib.ua_unified_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(cu_seqlens_q), _ptr(seq_lens_k),
        _ptr(block_table), block_size, hq, hkv, d, float(scale), float(softcap or 0.0),
        int(window_left if window_left is not None else -1), _ptr(alibi_slopes), _ptr(qq_bias),
        _ptr(sinks), _dtype_code(k_cache), _ptr(kv_scale), BACKENDS[backend],
        ctypes.c_void_p(stream.cuda_stream), ctypes.byref(sh))
    if rc != 0:
        raise UaError(rc, "ua_unified_attention")
    return out


class PreparedAttention:
    """``unified_attention`` with its sizes and options marshalled once, for a loop that
    calls it again and again with the same shapes (a decode loop, a captured step).

    Built by :func:`prepare`.  Calling it passes new per-step tensors -- ``q``,
    ``cu_seqlens_q``, ``seq_lens_k``, ``block_table``, ``out`` -- each of the prepared one's
    shape, dtype and device (checked); any left out keeps the prepared tensor.  The caches,
    the score features, the scales and the host sizes (``max_seqlen_q``/``max_seqlen_k``)
    stay as prepared.  Returns ``out``.
    """

    _STEP = ("q", "cu_seqlens_q", "seq_lens_k", "block_table", "out")
    _POS = {"q": 0, "out": 3, "cu_seqlens_q": 4, "seq_lens_k": 5, "block_table": 6}

    def __init__(self, lib, args, shape, tensors, stream):
        self._lib = lib
        self._args = args
        self._shape = shape
        self._meta = {n: (tuple(t.shape), t.dtype, t.device) for n, t in tensors.items()}
        self._keep = dict(tensors)
        self._stream = stream
        self.out = tensors["out"]

    def __call__(self, q=None, cu_seqlens_q=None, seq_lens_k=None, block_table=None, out=None,
                 stream=None):
        args = self._args
        for name, t in (("q", q), ("cu_seqlens_q", cu_seqlens_q), ("seq_lens_k", seq_lens_k),
                        ("block_table", block_table), ("out", out)):
            if t is None:
                continue
            if (tuple(t.shape), t.dtype, t.device) != self._meta[name] or not t.is_contiguous():
                raise ValueError(f"{name}: shape, dtype, device or layout differs from the "
                                 "prepared call")
            args[self._POS[name]] = ctypes.c_void_p(t.data_ptr())
            self._keep[name] = t
        if stream is not None:
            args[-2] = ctypes.c_void_p(stream.cuda_stream)
        rc = self._lib.ua_unified_attention(*args)
        if rc != 0:
            raise UaError(rc, "ua_unified_attention")
        return self._keep["out"]


def prepare(q, k_cache, v_cache, cu_seqlens_q, seq_lens_k, block_table, *, max_seqlen_q: int,
            max_seqlen_k: int, scale: float | None = None, softcap: float = 0.0,
            window_left: int = -1, alibi_slopes=None, qq_bias=None, sinks=None, kv_scale=None,
            k_scale_tok=None, v_scale_tok=None, out=None, out_dtype=None, backend: str = "auto",
            num_splits: int = 0, workspace=None, stream=None) -> PreparedAttention:
    """Validate and marshal a ``unified_attention`` call once (same arguments); the
    returned :class:`PreparedAttention` makes the call with new per-step tensors."""
    lib = _lib.load()
    total_q, hq, d = q.shape
    num_blocks, block_size, hkv, dk = k_cache.shape
    if dk != d or v_cache.shape != k_cache.shape:
        raise ValueError("q, k_cache and v_cache disagree on shape")
    if qq_bias is not None and qq_bias.shape[0] < max_seqlen_q:
        raise ValueError("qq_bias needs at least max_seqlen_q rows")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("seq_lens_k", seq_lens_k),
                    ("block_table", block_table)):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 tensor")
    if not (q.is_cuda and k_cache.is_cuda and v_cache.is_cuda):
        raise ValueError("q, k_cache and v_cache must be CUDA tensors")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((total_q, hq, d), dtype=out_dtype or q.dtype, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sh = _shape(q, k_cache, block_table, cu_seqlens_q, max_seqlen_q, max_seqlen_k, qq_bias,
                _dtype_code(out), num_splits, workspace, None, k_scale_tok, v_scale_tok)
    args = [_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(cu_seqlens_q),
            _ptr(seq_lens_k), _ptr(block_table), block_size, hq, hkv, d, float(scale),
            float(softcap or 0.0), int(window_left if window_left is not None else -1),
            _ptr(alibi_slopes), _ptr(qq_bias), _ptr(sinks), _dtype_code(k_cache), _ptr(kv_scale),
            BACKENDS[backend], ctypes.c_void_p(stream.cuda_stream), ctypes.byref(sh)]
    tensors = {"q": q, "cu_seqlens_q": cu_seqlens_q, "seq_lens_k": seq_lens_k,
               "block_table": block_table, "out": out}
    prep = PreparedAttention(lib, args, sh, tensors, stream)
    # the caches, score features and scales the prepared call points at stay alive with it
    prep._static = (k_cache, v_cache, alibi_slopes, qq_bias, sinks, kv_scale, k_scale_tok,
                    v_scale_tok, workspace)
    return prep


def plan(*, num_seqs, total_q, max_seqlen_q, max_seqlen_k, block_size, num_q_heads,
         num_kv_heads, head_dim, window_left=-1, kv_dtype=UA_DT_BF16, q_dtype=None,
         backend="auto", num_splits=0, num_sms=0, max_blocks_per_seq=1, num_blocks=1,
         per_token_scales=False):
    """The dispatcher's decision for these sizes (host only; no GPU needed when num_sms > 0).
    per_token_scales: plan for an fp8 call with per-token K/V scales (the dispatcher only
    tests the scale pointers for null; this passes a placeholder that is never read)."""
    lib = _lib.load()
    sh = _lib.UaShape()
    if per_token_scales:
        sh.k_scale_tok = sh.v_scale_tok = 256
    sh.num_seqs, sh.total_q = num_seqs, total_q
    sh.max_seqlen_q, sh.max_seqlen_k = max_seqlen_q, max_seqlen_k
    sh.max_blocks_per_seq, sh.num_blocks = max_blocks_per_seq, num_blocks
    sh.q_dtype = q_dtype if q_dtype is not None else (UA_DT_BF16 if kv_dtype == UA_DT_F8E4M3
                                                      else kv_dtype)
    sh.out_dtype = sh.q_dtype
    sh.num_splits = num_splits
    pl = _lib.UaPlan()
    rc = lib.ua_plan(ctypes.byref(sh), block_size, num_q_heads, num_kv_heads, head_dim,
                     window_left, kv_dtype, BACKENDS[backend], num_sms, ctypes.byref(pl))
    if rc != 0:
        raise UaError(rc, "ua_plan")
    return {f: getattr(pl, f) for f, _ in pl._fields_}


def device_status(stream=None) -> int:
    """Synchronise the stream and return the kernels' device check status (ua_status_t)."""
    lib = _lib.load()
    stream = stream or torch.cuda.current_stream()
    st = ctypes.c_int(0)
    rc = lib.ua_device_status(ctypes.c_void_p(stream.cuda_stream), ctypes.byref(st))
    if rc != 0:
        raise UaError(rc, "ua_device_status")
    return st.value


def device_status_reset(stream=None) -> None:
    lib = _lib.load()
    stream = stream or torch.cuda.current_stream()
    rc = lib.ua_device_status_reset(ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise UaError(rc, "ua_device_status_reset")

"""Plain fp64 CPU oracle for unified paged varlen GQA attention.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the CPU-baseline
leg of ``bench.py`` are the only callers.  The oracle shares no code with the
CUDA library and never calls it; the product path never calls the oracle.

The arithmetic lives in ``ua_ref.c`` (one output row at a time, by the plain
definition, plus the split-KV form used to pin the partition/merge algorithm);
this module only marshals arrays into it and spreads rows over host threads.
Sources are cited in ``ua_ref.c``.  Parity unpinned: the order in which softcap and
the ALiBi / QQ-bias terms compose (the pages name the terms, not their order); every
term on its own is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ua_ref.c")
_SO = os.path.join(_HERE, "libua_ref.so")
_LOCK = threading.Lock()
_LIB = None

# element-type codes understood by ua_ref.c
F16, BF16, E4M3, F32 = 0, 1, 2, 3

ERRORS = {1: "invalid argument", 3: "block id out of range", 4: "out of memory"}


def build(force: bool = False) -> str:
    """Compile ua_ref.c into libua_ref.so with the host C compiler (no fast-math)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _SO)
    return _SO


class Problem(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("seq_lens_k", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("alibi_slopes", ctypes.c_void_p),
        ("qq_bias", ctypes.c_void_p),
        ("sinks", ctypes.c_void_p),
        ("q_dtype", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("window_left", ctypes.c_int32),
        ("qq_bias_stride", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("softcap", ctypes.c_double),
        ("k_scale", ctypes.c_double),
        ("v_scale", ctypes.c_double),
        ("k_scale_tok", ctypes.c_void_p),
        ("v_scale_tok", ctypes.c_void_p),
        ("k_scale_strides", ctypes.c_int64 * 3),
        ("v_scale_strides", ctypes.c_int64 * 3),
    ]


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            handle = ctypes.CDLL(build())
            handle.ua_ref_attention.argtypes = [ctypes.POINTER(Problem), ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_void_p]
            handle.ua_ref_attention.restype = ctypes.c_int
            handle.ua_ref_attention_rows.argtypes = [ctypes.POINTER(Problem), ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
            handle.ua_ref_attention_rows.restype = ctypes.c_int
            for name, arg in (("ua_ref_decode_f16", ctypes.c_uint16),
                              ("ua_ref_decode_bf16", ctypes.c_uint16),
                              ("ua_ref_decode_e4m3", ctypes.c_uint8)):
                fn = getattr(handle, name)
                fn.argtypes = [arg]
                fn.restype = ctypes.c_double
            _LIB = handle
    return _LIB


def _raw(x, kind):
    """Host array of raw element bits (numpy), plus its type code."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.float16:
            return x.view(torch.int16).numpy().view(np.uint16), F16
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), BF16
        if x.dtype == torch.float8_e4m3fn:
            return x.view(torch.uint8).numpy(), E4M3
        if x.dtype == torch.float32:
            return x.numpy(), F32
        if x.dtype == torch.int32:
            return x.numpy(), None
        raise TypeError(f"unsupported tensor dtype {x.dtype}")
    x = np.ascontiguousarray(x)
    if kind is not None:
        return x, kind
    if x.dtype == np.float16:
        return x.view(np.uint16), F16
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.int32:
        return x, None
    raise TypeError(f"numpy dtype {x.dtype} needs an explicit element-type code")


def _opt_f32(x):
    if x is None:
        return None
    a, _ = _raw(x, F32)
    return np.ascontiguousarray(a, dtype=np.float32)


def _tok_scale(x):
    """A per-token fp8 scale array [num_blocks, block_size, H_kv] (float32 numpy array or
    torch tensor, any strides): the array kept alive, its first element's address and its
    element strides."""
    if x is None:
        return None, None, (0, 0, 0)
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        if x.dtype != torch.float32:
            raise TypeError("per-token scales must be float32")
        a = x.detach().cpu().numpy()
    else:
        a = np.asarray(x)
        if a.dtype != np.float32:
            raise TypeError("per-token scales must be float32")
    if a.ndim != 3 or any(st % 4 for st in a.strides) or any(st < 0 for st in a.strides):
        raise ValueError("per-token scales are [num_blocks, block_size, H_kv] with positive strides")
    return a, a.ctypes.data, tuple(st // 4 for st in a.strides)


def _problem(q, k_cache, v_cache, cu_seqlens_q, seq_lens_k, block_table, *, scale, softcap,
             window_left, alibi_slopes, qq_bias, qq_bias_stride, sinks, k_scale, v_scale,
             q_dtype, kv_dtype, k_scale_tok=None, v_scale_tok=None):
    qa, qk = _raw(q, q_dtype)
    ka, kk = _raw(k_cache, kv_dtype)
    va, vk = _raw(v_cache, kv_dtype)
    cu = np.ascontiguousarray(_raw(cu_seqlens_q, None)[0], dtype=np.int32)
    sl = np.ascontiguousarray(_raw(seq_lens_k, None)[0], dtype=np.int32)
    bt = np.ascontiguousarray(_raw(block_table, None)[0], dtype=np.int32)
    al, qb, sk = _opt_f32(alibi_slopes), _opt_f32(qq_bias), _opt_f32(sinks)
    if kk != vk:
        raise ValueError("k_cache and v_cache must share one element type")
    num_blocks, block_size, hkv, d = ka.shape
    total_q, hq, dq = qa.shape
    if dq != d or bt.ndim != 2:
        raise ValueError("shape mismatch")
    if qb is not None and qq_bias_stride is None:
        qq_bias_stride = qb.shape[-1]
    kt, ktp, kts = _tok_scale(k_scale_tok)
    vt, vtp, vts = _tok_scale(v_scale_tok)
    for t in (kt, vt):
        if t is not None and (t.shape[0] != num_blocks or t.shape[1] != block_size or
                              t.shape[2] != hkv):
            raise ValueError("per-token scales are [num_blocks, block_size, H_kv]")
    keep = [qa, ka, va, cu, sl, bt, al, qb, sk, kt, vt]
    ptr = lambda a: None if a is None else a.ctypes.data  # noqa: E731
    prob = Problem(ptr(qa), ptr(ka), ptr(va), ptr(cu), ptr(sl), ptr(bt), ptr(al), ptr(qb), ptr(sk),
                   qk, kk, len(sl), bt.shape[1], num_blocks, block_size, hq, hkv, d,
                   -1 if window_left is None else int(window_left),
                   int(qq_bias_stride or 0), float(scale), float(softcap or 0.0),
                   float(k_scale), float(v_scale), ktp, vtp,
                   (ctypes.c_int64 * 3)(*kts), (ctypes.c_int64 * 3)(*vts))
    return prob, keep, total_q, hq, d


def attention(q, k_cache, v_cache, cu_seqlens_q, seq_lens_k, block_table, *, scale, softcap=0.0,
              window_left=-1, alibi_slopes=None, qq_bias=None, qq_bias_stride=None, sinks=None,
              k_scale=1.0, v_scale=1.0, q_dtype=None, kv_dtype=None, n_part=0, threads=1,
              token_range=None, head_range=None, k_scale_tok=None, v_scale_tok=None):
    """Attention output [total_q, H_q, D] in float64.

    ``n_part <= 0`` evaluates the plain definition; ``n_part >= 1`` evaluates the
    split-KV partition/merge form.  Rows outside ``token_range``/``head_range`` stay 0.
    ``k_scale_tok`` / ``v_scale_tok``: fp8 per-token scales [num_blocks, block_size, H_kv]
    (any strides) in place of the per-tensor ``k_scale`` / ``v_scale``.
    """
    prob, keep, total_q, hq, d = _problem(
        q, k_cache, v_cache, cu_seqlens_q, seq_lens_k, block_table, scale=scale, softcap=softcap,
        window_left=window_left, alibi_slopes=alibi_slopes, qq_bias=qq_bias,
        qq_bias_stride=qq_bias_stride, sinks=sinks, k_scale=k_scale, v_scale=v_scale,
        q_dtype=q_dtype, kv_dtype=kv_dtype, k_scale_tok=k_scale_tok, v_scale_tok=v_scale_tok)
    out = np.zeros((total_q, hq, d), dtype=np.float64)
    t0, t1 = token_range or (0, total_q)
    h0, h1 = head_range or (0, hq)
    L = lib()
    jobs = [(t0, t1, h, h + 1) for h in range(h0, h1)] if threads > 1 else [(t0, t1, h0, h1)]

    def run(job):
        return L.ua_ref_attention(ctypes.byref(prob), job[0], job[1], job[2], job[3], int(n_part),
                                  out.ctypes.data)

    if threads > 1:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            codes = list(ex.map(run, jobs))
    else:
        codes = [run(j) for j in jobs]
    del keep
    bad = [c for c in codes if c]
    if bad:
        raise ValueError(f"oracle: {ERRORS.get(bad[0], bad[0])}")
    return out


def attention_rows(q, k_cache, v_cache, cu_seqlens_q, seq_lens_k, block_table, tokens, heads, *,
                   scale, softcap=0.0, window_left=-1, alibi_slopes=None, qq_bias=None,
                   qq_bias_stride=None, sinks=None, k_scale=1.0, v_scale=1.0, q_dtype=None,
                   kv_dtype=None, threads=1, k_scale_tok=None, v_scale_tok=None):
    """Selected output rows: result[r] is the row of (tokens[r], heads[r]), float64 [n, D]."""
    prob, keep, total_q, hq, d = _problem(
        q, k_cache, v_cache, cu_seqlens_q, seq_lens_k, block_table, scale=scale, softcap=softcap,
        window_left=window_left, alibi_slopes=alibi_slopes, qq_bias=qq_bias,
        qq_bias_stride=qq_bias_stride, sinks=sinks, k_scale=k_scale, v_scale=v_scale,
        q_dtype=q_dtype, kv_dtype=kv_dtype, k_scale_tok=k_scale_tok, v_scale_tok=v_scale_tok)
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    hd = np.ascontiguousarray(heads, dtype=np.int32)
    out = np.zeros((len(tok), d), dtype=np.float64)
    L = lib()
    chunks = np.array_split(np.arange(len(tok)), max(1, min(threads, len(tok))))

    def run(idx):
        if len(idx) == 0:
            return 0
        a, b = int(idx[0]), int(idx[-1]) + 1
        return L.ua_ref_attention_rows(ctypes.byref(prob), tok[a:b].ctypes.data,
                                       hd[a:b].ctypes.data, b - a, out[a:b].ctypes.data)

    if threads > 1:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            codes = list(ex.map(run, chunks))
    else:
        codes = [run(c) for c in chunks]
    del keep
    bad = [c for c in codes if c]
    if bad:
        raise ValueError(f"oracle: {ERRORS.get(bad[0], bad[0])}")
    return out


def decode(codes, kind):
    """Exact float64 value of each raw element code under element type ``kind``."""
    L = lib()
    fn = {F16: L.ua_ref_decode_f16, BF16: L.ua_ref_decode_bf16, E4M3: L.ua_ref_decode_e4m3}[kind]
    return np.array([fn(int(c)) for c in np.asarray(codes).ravel()], dtype=np.float64)

"""ua_unified_attention_noalloc: the entry point for callers that may not allocate.

Some callers cannot call cudaMalloc at call time -- a serving runtime that has given
all free device memory to its own cache pool, a process held to a fixed memory
budget, a latency-critical loop where an allocation could block the device.  For them
the library keeps the split-KV path's scratch in one fixed device array.  These tests
call that entry point through the C ABI and check it against ua_unified_attention
(which uses its own workspace) on two calls in a row, plus the size limit.

This file is collected last on purpose: it runs after every other test when the suite
stops at the first failure, and it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import varlen_gqa_attention_paged_gb300 as ua
import workloads as W
from tests._gpu import TOL, to_dev
from varlen_gqa_attention_paged_gb300 import _lib

pytestmark = pytest.mark.gpu


def _c_call(fn, inp, d, out, backend, shape_overrides=None):
    sh = ua._shape(d["q"], d["k_cache"], d["block_table"], d["cu_seqlens_q"], inp.max_seqlen_q,
                   inp.max_seqlen_k, d["qq_bias"], ua._DTYPES[out.dtype], 0, None, None)
    for k, v in (shape_overrides or {}).items():
        setattr(sh, k, v)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    spec = inp.spec
    stream = torch.cuda.current_stream()
    return fn(p(d["q"]), p(d["k_cache"]), p(d["v_cache"]), p(out), p(d["cu_seqlens_q"]),
              p(d["seq_lens_k"]), p(d["block_table"]), spec.block_size, spec.num_q_heads,
              spec.num_kv_heads, spec.head_dim, float(inp.scale), float(inp.softcap),
              int(inp.window_left), p(d["alibi_slopes"]), p(d["qq_bias"]), p(d["sinks"]),
              ua._DTYPES[spec.kv_dtype], p(d["kv_scale"]), ua.BACKENDS[backend],
              ctypes.c_void_p(stream.cuda_stream), ctypes.byref(sh))


def test_noalloc_matches_the_default_entry_point_on_two_calls_in_a_row():
    lib = _lib.load()
    # two different split-path problems back to back: the second call reuses the array
    # the first one left behind
    for spec in (W.SWDECODE_BF16, W.DECODE):
        inp = W.make(spec, poison=True)
        d = to_dev(inp)
        shape = (inp.total_q, spec.num_q_heads, spec.head_dim)
        ref = torch.empty(shape, dtype=torch.float32, device="cuda")
        got = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        assert _c_call(lib.ua_unified_attention, inp, d, ref, "split") == 0
        assert _c_call(lib.ua_unified_attention_noalloc, inp, d, got, "split") == 0
        torch.cuda.synchronize()
        diff = (got.double() - ref.double()).abs().max().item()
        assert np.isfinite(diff) and diff <= TOL[spec.kv_dtype], f"{spec.name}: {diff:.3e}"


def test_noalloc_rejects_calls_beyond_its_scratch():
    lib = _lib.load()
    inp = W.make(W.TINY)
    d = to_dev(inp)
    out = torch.empty((inp.total_q, 4, 64), dtype=torch.float32, device="cuda")
    # 2 tokens x 4 heads x 128 partitions needs little scratch; pretend the batch has
    # 100000 query tokens so the plan needs more than the fixed array holds
    need = ua.plan(num_seqs=2, total_q=100000, max_seqlen_q=1, max_seqlen_k=37, block_size=16,
                   num_q_heads=4, num_kv_heads=2, head_dim=64, kv_dtype=ua.UA_DT_F16,
                   backend="split", num_splits=128)["workspace_bytes"]
    assert need > _lib.UA_NOALLOC_SCRATCH_BYTES
    rc = _c_call(lib.ua_unified_attention_noalloc, inp, d, out, "split",
                 dict(total_q=100000, max_seqlen_q=1, num_splits=128))
    assert rc == _lib.UA_ERR_SCRATCH_LIMIT
    assert b"scratch" in lib.ua_status_string(rc)

"""ua_unified_attention_noalloc: the entry point for callers that may not allocate.

Some callers cannot call cudaMalloc at call time -- a serving runtime that has given
all free device memory to its own cache pool, a process held to a fixed memory
budget, a latency-critical loop where an allocation could block the device.  For them
the library keeps the split-KV path's scratch in one fixed device array.  These tests
call that entry point through the C ABI on problems whose plan needs that scratch
(partitions merged by the separate merge kernel), check the output against the oracle
and against ua_unified_attention on two rounds of calls in a row (each call follows a
different problem's, so contents left in the array by the call before would show),
check that the call allocates no device memory, and check the size limit.

This file is collected last on purpose: it runs after every other test when the suite
stops at the first failure, and it also passes alone in a fresh process.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
import varlen_gqa_attention_paged_gb300 as ua
import workloads as W
from tests._gpu import TOL, max_err, to_dev
from varlen_gqa_attention_paged_gb300 import _lib

pytestmark = pytest.mark.gpu
THREADS = min(16, os.cpu_count() or 1)

# Problems whose split path merges through the scratch: the sliding-window decode forced
# to 20 partitions (more than one thread-block cluster holds, so the merge kernel runs),
# and the mixed prefill + decode batch (the tensor-memory kernel's split, merged by the
# merge kernel).
CASES = [(W.SWDECODE_BF16, "split", 20), (W.MIXED, "auto", 0)]


def _c_call(fn, inp, d, out, backend, num_splits=0, shape_overrides=None, stream=None):
    sh = ua._shape(d["q"], d["k_cache"], d["block_table"], d["cu_seqlens_q"], inp.max_seqlen_q,
                   inp.max_seqlen_k, d["qq_bias"], ua._DTYPES[out.dtype], num_splits, None, None)
    for k, v in (shape_overrides or {}).items():
        setattr(sh, k, v)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    spec = inp.spec
    stream = stream or torch.cuda.current_stream()
    return fn(p(d["q"]), p(d["k_cache"]), p(d["v_cache"]), p(out), p(d["cu_seqlens_q"]),
              p(d["seq_lens_k"]), p(d["block_table"]), spec.block_size, spec.num_q_heads,
              spec.num_kv_heads, spec.head_dim, float(inp.scale), float(inp.softcap),
              int(inp.window_left), p(d["alibi_slopes"]), p(d["qq_bias"]), p(d["sinks"]),
              ua._DTYPES[spec.kv_dtype], p(d["kv_scale"]), ua.BACKENDS[backend],
              ctypes.c_void_p(stream.cuda_stream), ctypes.byref(sh))


def _plan(inp, backend, num_splits):
    spec = inp.spec
    return ua.plan(num_seqs=inp.num_seqs, total_q=inp.total_q, max_seqlen_q=inp.max_seqlen_q,
                   max_seqlen_k=inp.max_seqlen_k, block_size=spec.block_size,
                   num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                   head_dim=spec.head_dim, window_left=inp.window_left,
                   kv_dtype=ua._DTYPES[spec.kv_dtype], q_dtype=ua._DTYPES[spec.q_dtype],
                   backend=backend, num_splits=num_splits,
                   max_blocks_per_seq=inp.block_table.shape[-1],
                   num_blocks=inp.k_cache.shape[0])


_PREPARED = {}


def _prepared(spec):
    if spec.name not in _PREPARED:
        inp = W.make(spec, poison=True)
        _PREPARED[spec.name] = (inp, to_dev(inp),
                                oracle.attention(threads=THREADS, **inp.oracle_kwargs()))
    return _PREPARED[spec.name]


def test_noalloc_uses_its_scratch_and_matches_the_oracle_on_two_calls_in_a_row():
    lib = _lib.load()
    for spec, backend, nsplit in CASES:
        inp, _, _ = _prepared(spec)
        pl = _plan(inp, backend, nsplit)
        # the merge kernel over the scratch, not the in-cluster merge
        assert pl["path"] == ua.UA_PATH_SPLIT and pl["cluster_z"] == 1, (spec.name, pl)
        assert 0 < pl["workspace_bytes"] <= _lib.UA_NOALLOC_SCRATCH_BYTES, (spec.name, pl)
    for _ in range(2):
        for spec, backend, nsplit in CASES:
            inp, d, want = _prepared(spec)
            shape = (inp.total_q, spec.num_q_heads, spec.head_dim)
            got = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            ref = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
            assert _c_call(lib.ua_unified_attention_noalloc, inp, d, got, backend, nsplit) == 0
            torch.cuda.synchronize()
            err = max_err(got, want)
            assert err <= TOL[spec.kv_dtype], f"{spec.name}: {err:.3e} against the oracle"
            assert _c_call(lib.ua_unified_attention, inp, d, ref, backend, nsplit) == 0
            torch.cuda.synchronize()
            diff = (got.double() - ref.double()).abs().max().item()
            assert np.isfinite(diff) and diff <= TOL[spec.kv_dtype], f"{spec.name}: {diff:.3e}"
    assert ua.device_status() == 0


def test_noalloc_allocates_no_device_memory():
    lib = _lib.load()
    spec, backend, nsplit = CASES[0]
    inp, d, want = _prepared(spec)
    out = torch.empty((inp.total_q, spec.num_q_heads, spec.head_dim), dtype=torch.float32,
                      device="cuda")
    # the first call on the device loads the kernels and looks up the array's address
    assert _c_call(lib.ua_unified_attention_noalloc, inp, d, out, backend, nsplit) == 0
    torch.cuda.synchronize()
    # a stream the library has never seen: ua_unified_attention would allocate its
    # workspace for it (at least 1 MiB; this plan needs 2.6 MB)
    for fn, allocates in ((lib.ua_unified_attention_noalloc, False),
                          (lib.ua_unified_attention, True)):
        stream = torch.cuda.Stream()
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        assert _c_call(fn, inp, d, out, backend, nsplit, stream=stream) == 0
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        if allocates:  # the check sees an allocation when there is one
            assert free1 <= free0 - (1 << 20), (free0, free1)
        else:
            assert free1 >= free0, (free0, free1)
        assert max_err(out, want) <= TOL[spec.kv_dtype]


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
                 shape_overrides=dict(total_q=100000, max_seqlen_q=1, num_splits=128))
    assert rc == _lib.UA_ERR_SCRATCH_LIMIT
    assert b"scratch" in lib.ua_status_string(rc)

"""The C ABI on the host: the library loads, exports what include/ua.h declares, rejects
bad arguments before touching the GPU, and the dispatcher plans as designed."""
import ctypes
import os
import re
import subprocess

import pytest

import varlen_gqa_attention_paged_gb300 as ua
from varlen_gqa_attention_paged_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "ua.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(ua_\w+)\s*\(", text,
                                 flags=re.M)))


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    assert lib.ua_version() == 100
    assert lib.ua_status_string(0) == b"ok"
    assert b"workspace" in lib.ua_status_string(4)


def test_binding_structs_match_the_header_layout(tmp_path):
    """Every field of ua_shape_t and ua_plan_t sits at the same offset, with the same size,
    in the C compiler's layout of include/ua.h and in the ctypes mirrors of the binding."""
    structs = {"ua_shape_t": _lib.UaShape, "ua_plan_t": _lib.UaPlan}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "ua.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu %zu\\n", offsetof({cname}, {f}), '
                         f"sizeof((({cname}*)0)->{f}));")
    lines += ["return 0;", "}"]
    src, exe = tmp_path / "layout.c", tmp_path / "layout"
    src.write_text("\n".join(lines) + "\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(root, "include"), "-o", str(exe),
                    str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {}
    for ln in out.splitlines():
        parts = ln.split()
        got[(parts[0], parts[1])] = tuple(int(x) for x in parts[2:])
    for cname, py in structs.items():
        assert got[(cname, "sizeof")] == (ctypes.sizeof(py),), cname
        for f, _ in py._fields_:
            desc = getattr(py, f)
            assert got[(cname, f)] == (desc.offset, desc.size), (cname, f)


FAKE = 0x7f0000001000  # aligned, never dereferenced: every case fails validation first


def call(**over):
    sh = _lib.UaShape()
    sh.num_seqs, sh.total_q, sh.max_seqlen_q, sh.max_seqlen_k = 2, 6, 5, 37
    sh.max_blocks_per_seq, sh.num_blocks, sh.q_dtype, sh.out_dtype = 3, 8, 0, 0
    for k in list(over):
        if hasattr(sh, k) and k not in ("head_dim",):
            setattr(sh, k, over.pop(k))
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, cu=FAKE, sl=FAKE, bt=FAKE, block_size=16, hq=4,
             hkv=2, d=64, scale=0.125, softcap=0.0, wl=-1, alibi=None, qq=None, sinks=None,
             kv_dtype=0, kv_scale=None, backend=0)
    a.update(over)
    v = lambda x: None if x is None else ctypes.c_void_p(x)  # noqa: E731
    return _lib.load().ua_unified_attention(
        v(a["q"]), v(a["k"]), v(a["v"]), v(a["out"]), v(a["cu"]), v(a["sl"]), v(a["bt"]),
        a["block_size"], a["hq"], a["hkv"], a["d"], a["scale"], a["softcap"], a["wl"],
        v(a["alibi"]), v(a["qq"]), v(a["sinks"]), a["kv_dtype"], v(a["kv_scale"]), a["backend"],
        None, ctypes.byref(sh))


@pytest.mark.parametrize("over,code", [
    (dict(d=96), _lib.UA_ERR_INVALID_ARG),
    (dict(hq=6, hkv=4), _lib.UA_ERR_INVALID_ARG),
    (dict(hkv=0), _lib.UA_ERR_INVALID_ARG),
    (dict(block_size=0), _lib.UA_ERR_INVALID_ARG),
    (dict(q=None), _lib.UA_ERR_INVALID_ARG),
    (dict(bt=None), _lib.UA_ERR_INVALID_ARG),
    (dict(k=FAKE + 8), _lib.UA_ERR_INVALID_ARG),
    (dict(kv_dtype=7), _lib.UA_ERR_INVALID_ARG),
    (dict(backend=9), _lib.UA_ERR_INVALID_ARG),
    (dict(kv_dtype=1), _lib.UA_ERR_UNSUPPORTED),            # f16 q with a bf16 cache
    (dict(kv_dtype=2), _lib.UA_ERR_INVALID_ARG),            # fp8 cache without kv_scale
    (dict(qq=FAKE, qq_bias_stride=4), _lib.UA_ERR_INVALID_ARG),   # stride < max_seqlen_q
    (dict(out_dtype=2), _lib.UA_ERR_INVALID_ARG),
    (dict(num_blocks=-1), _lib.UA_ERR_INVALID_ARG),
])
def test_host_validation_rejects_before_any_launch(over, code):
    assert call(**over) == code


def test_empty_batch_is_a_no_op():
    assert call(total_q=0) == _lib.UA_OK
    assert call(num_seqs=0, total_q=0) == _lib.UA_OK


def _plan(**kw):
    base = dict(num_seqs=8, total_q=8, max_seqlen_q=1, max_seqlen_k=6700, block_size=16,
                num_q_heads=32, num_kv_heads=8, head_dim=128, window_left=4095,
                kv_dtype=_lib.UA_DT_BF16, num_sms=152, max_blocks_per_seq=419, num_blocks=4190)
    base.update(kw)
    return ua.plan(**base)


def test_dispatcher_splits_long_underfilled_decode():
    p = _plan()
    assert p["path"] == _lib.UA_PATH_SPLIT and p["n_part"] >= 2
    # the key-major decode tile: 8 rows of a kv-head per CTA, three CTAs per SM
    assert p["kernel"] == 2 and p["block_m"] == 8
    assert p["grid_y"] == 8 and p["grid_z"] == p["n_part"]
    assert p["grid_x"] == 8 and p["slot_per_seq"] == 1
    # the partitions of a slot form one cluster with some of its kv-heads (8 CTAs at most)
    # and merge through distributed shared memory: no workspace
    assert p["cluster_z"] == p["n_part"] and p["cluster_y"] * p["cluster_z"] <= 8
    assert 8 % p["cluster_y"] == 0 and p["workspace_bytes"] == 0
    # 9 to 16 partitions: a cluster of the partitions alone
    p = _plan(backend="split", num_splits=12)
    assert p["cluster_z"] == 12 and p["cluster_y"] == 1 and p["workspace_bytes"] == 0
    # more than 16 partitions: the merge kernel and its scratch
    p = _plan(backend="split", num_splits=20)
    assert p["cluster_z"] == 1 and p["cluster_y"] == 8
    assert p["workspace_bytes"] >= 8 * 32 * 20 * (128 + 2) * 4


def test_dispatcher_keeps_short_or_full_grids_on_2d():
    # short walk (below two minimum partitions of 256 keys): no split
    assert _plan(max_seqlen_k=200, window_left=-1)["path"] == _lib.UA_PATH_2D
    # long prefill: the 2D grid already fills the device
    p = _plan(num_seqs=5, total_q=18432, max_seqlen_q=4096, max_seqlen_k=18432, window_left=-1)
    assert p["path"] == _lib.UA_PATH_2D and p["block_m"] >= 64 and p["workspace_bytes"] == 0


def test_dispatcher_forced_backends_and_split_count():
    assert _plan(backend="2d")["n_part"] == 1
    assert _plan(backend="split", max_seqlen_k=40, window_left=-1)["n_part"] >= 2
    assert _plan(backend="split", num_splits=5)["n_part"] == 5
    one = _plan(backend="split", num_splits=20)["workspace_bytes"]
    assert one > 0
    assert ua._lib.load().ua_workspace_bytes is not None


def test_dispatcher_walk_uses_the_window():
    # a short window bounds the walk: no split even though kv_len is long
    assert _plan(window_left=127)["path"] == _lib.UA_PATH_2D


def test_dispatcher_split_fits_one_wave():
    for hkv, seqs, kv in ((8, 8, 1), (2, 4, 0), (8, 2, 2), (1, 1, 1)):
        p = _plan(num_seqs=seqs, total_q=seqs, num_kv_heads=hkv, num_q_heads=4 * hkv, kv_dtype=kv,
                  window_left=-1, max_seqlen_k=100000)
        active = seqs * p["grid_y"]                     # CTAs of one partition
        per_sm = 3 if p["kernel"] == 2 else 2  # decode tile: three an SM (two-head tile: two)
        assert p["path"] == _lib.UA_PATH_SPLIT
        assert active * p["n_part"] <= per_sm * 152
        # the largest count that fits: one more partition would start a second wave (of
        # the slots, or of the clusters, which host-only plans give 90 % of the slots)
        assert active * (p["n_part"] + 1) > 0.9 * per_sm * 152 or p["n_part"] == 128


def test_dispatcher_decode_kernels():
    # at most 8 rows per kv-head, head_dim <= 128, page boxes: the key-major decode tile
    assert _plan()["kernel"] == 2
    # fp8 with at most 4 rows per kv-head and an even kv-head count: two kv-heads a CTA
    p = _plan(head_dim=64, kv_dtype=2)
    assert p["kernel"] == 64 and p["grid_y"] == 4 and p["block_m"] == 8
    assert _plan(kv_dtype=2, max_seqlen_q=2)["kernel"] == 2          # 8 rows a kv-head
    assert _plan(kv_dtype=2, num_kv_heads=1, num_q_heads=4)["kernel"] in (2, 32)  # one kv-head
    assert _plan(kv_dtype=2, num_kv_heads=4, num_q_heads=4, max_seqlen_q=4)["kernel"] == 64
    assert _plan(kv_dtype=2, per_token_scales=True)["kernel"] == 2  # scales: one head a CTA
    # more rows (up to 16), head_dim 256, pages not a multiple of 16: the 16-row tile
    assert _plan(max_seqlen_q=3)["kernel"] == 1
    assert _plan(head_dim=256)["kernel"] == 1
    assert _plan(block_size=13)["kernel"] == 1
    # a decode grid of at most one CTA per SM: the decode tile with eight consumer warps
    p = _plan(num_seqs=4, total_q=4, max_seqlen_k=4096, num_q_heads=16, num_kv_heads=2,
              window_left=-1, kv_dtype=_lib.UA_DT_F16)
    assert p["kernel"] == 32 and p["grid_x"] * p["grid_y"] * p["grid_z"] <= 152
    assert p["cluster_z"] == p["n_part"] and p["workspace_bytes"] == 0


def test_dispatcher_prefill_kernels():
    prefill = dict(num_seqs=5, total_q=18432, max_seqlen_q=4096, max_seqlen_k=18432,
                   window_left=-1, max_blocks_per_seq=1152, num_blocks=6000)
    # 16-bit caches, and fp8 at head_dim 64 and 128: the tensor-memory kernel, two q tiles
    # a CTA when the grid still fills the device
    for kv in (_lib.UA_DT_BF16, _lib.UA_DT_F16, _lib.UA_DT_F8E4M3):
        for d in (64, 128):
            p = _plan(kv_dtype=kv, head_dim=d, **prefill)
            assert p["kernel"] == 16 and p["block_m"] == 2 * 128, (kv, d)
    # head_dim 256 (16-bit or fp8 caches): the tensor-memory kernel, one q tile a CTA
    assert _plan(kv_dtype=_lib.UA_DT_F8E4M3, head_dim=256, **prefill)["kernel"] == 8
    assert _plan(kv_dtype=_lib.UA_DT_BF16, head_dim=256, **prefill)["kernel"] == 8
    # pages not a multiple of 16: the 64-row tile kernel
    assert _plan(kv_dtype=_lib.UA_DT_F8E4M3, block_size=13, **prefill)["kernel"] == 4


def test_dispatcher_mixed_batch_splits_underfilled_long_walks():
    p = _plan(num_seqs=5, total_q=327, max_seqlen_q=129, max_seqlen_k=1328, num_q_heads=16,
              num_kv_heads=2, window_left=-1)
    assert p["path"] == _lib.UA_PATH_SPLIT and p["n_part"] >= 2 and p["slot_per_seq"] == 0

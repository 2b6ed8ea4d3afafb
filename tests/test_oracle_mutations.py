"""Plant plausible mistakes in copies of the oracle (CPU only) and check the pins see them.

Each mutant is the oracle source with one textual change (a dropped term, a wrong
sign or offset, a transposed index), compiled into a temporary library.  A pin
that cannot tell the mutant from the original would not protect the GPU parity
tests, so every mutant must disagree with the dense brute force or the library
reference on at least one of the probe problems.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests._dense import dense_attention

SRC = os.path.join(os.path.dirname(oracle.__file__), "ua_ref.c")

MUTANTS = {
    "alibi_sign": ("(double)(j - ctx);", "(double)(ctx - j);"),
    "alibi_offset_from_row": ("(double)(j - ctx);", "(double)(j - ctx - i);"),
    "qq_bias_transposed": ("qq_bias[(size_t)i * P->qq_bias_stride + (j - ctx)]",
                           "qq_bias[(size_t)(j - ctx) * P->qq_bias_stride + i]"),
    "softcap_before_scale": ("double v = P->scale * dot;\n  if (P->softcap > 0.0) v = P->softcap * tanh(v / P->softcap);",
                             "double v = dot;\n  if (P->softcap > 0.0) v = P->softcap * tanh(v / P->softcap);\n  v *= P->scale;"),
    "window_off_by_one": ("*lo = p - P->window_left;", "*lo = p - P->window_left + 1;"),
    "sink_dropped_from_den": ("double den = P->sinks ? exp((double)P->sinks[h] - m) : 0.0;",
                              "double den = 0.0;"),
    "group_interleaved": ("add_value_row(P, b, j, h / G, w, acc)", "add_value_row(P, b, j, h % P->num_kv_heads, w, acc)"),
    "v_scale_dropped": ("double vscale = kv_scale_of(P, 1, b, j, g);", "double vscale = 1.0;"),
    "k_token_scale_for_v": ("double vscale = kv_scale_of(P, 1, b, j, g);",
                            "double vscale = kv_scale_of(P, 0, b, j, g);"),
    "token_scale_slot_stride": ("(int64_t)(j % P->block_size) * st[1]",
                                "(int64_t)(j % P->block_size) * st[2]"),
    "token_scale_head_dropped": ("+ (int64_t)g * st[2]", "+ 0 * st[2]"),
    "slot_from_wrong_block": ("(size_t)(j % P->block_size)", "(size_t)((j + 1) % P->block_size)"),
    "causal_excludes_self": ("*hi = p + 1 < kv_len ? p + 1 : kv_len;", "*hi = p < kv_len ? p : kv_len;"),
    "qq_bias_skips_first_key": ("if (P->qq_bias && j >= ctx)", "if (P->qq_bias && j >= ctx + 1)"),
    "e4m3_exponent_bias": ("else v = ldexp(1.0 + m / 8.0, e - 7);", "else v = ldexp(1.0 + m / 8.0, e - 8);"),
    "e4m3_subnormal_scale": ("if (e == 0) v = ldexp((double)m, -9);", "if (e == 0) v = ldexp((double)m, -10);"),
}

PROBES = [
    dict(alibi=True, window=7, sinks=True),
    dict(qq_bias=True, qq_bias_shape=(8, 64), qq_bias_std=0.5, softcap=0.8),
    dict(kv_dtype=torch.float8_e4m3fn, q_dtype=torch.bfloat16, window=5),
    dict(kv_dtype=torch.float8_e4m3fn, q_dtype=torch.bfloat16, per_token_scales=True, sinks=True),
]


def _compile(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(path), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    lib.ua_ref_attention.argtypes = [ctypes.POINTER(oracle.Problem), ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.ua_ref_attention.restype = ctypes.c_int
    return lib


def _run(lib, inp):
    prob, keep, total_q, hq, d = oracle._problem(**inp.oracle_kwargs(), q_dtype=None,
                                                 kv_dtype=None)
    out = np.zeros((total_q, hq, d))
    rc = lib.ua_ref_attention(ctypes.byref(prob), 0, total_q, 0, hq, 0, out.ctypes.data)
    del keep
    assert rc == 0
    return out


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(tmp_path, name):
    lib = _compile(tmp_path, name, *MUTANTS[name])
    worst = 0.0
    for i, feat in enumerate(PROBES):
        spec = W.Spec(name="m", seqs=[(1, 37), (5, 18), (7, 7), (3, 40)], num_q_heads=8,
                      num_kv_heads=2, head_dim=16, block_size=16, seed=40 + i, **feat)
        inp = W.make(spec)
        diff = np.abs(_run(lib, inp) - dense_attention(**inp.oracle_kwargs()))
        # a mutant that reads out of range can return NaN, which max() would skip
        worst = max(worst, float("inf") if np.isnan(diff).any() else float(diff.max()))
    assert worst > 1e-6, f"mutant {name} survived the pins"

"""Helpers that run the CUDA path on an input set (tests only)."""
import numpy as np
import torch

import varlen_gqa_attention_paged_gb300 as ua

# the stated parity bars: max abs error vs the fp64 oracle, by cache type
TOL = {torch.float16: 2e-3, torch.bfloat16: 2e-3, torch.float8_e4m3fn: 2e-2}


def to_dev(inp, dev="cuda"):
    d = {}
    for name in ("q", "k_cache", "v_cache", "cu_seqlens_q", "seq_lens_k", "block_table",
                 "alibi_slopes", "qq_bias", "sinks"):
        t = getattr(inp, name)
        d[name] = None if t is None else t.to(dev).contiguous()
    d["kv_scale"] = None
    if inp.spec.kv_dtype == torch.float8_e4m3fn:
        d["kv_scale"] = torch.tensor([inp.k_scale, inp.v_scale], dtype=torch.float32, device=dev)
    # per-token scales keep their strides (V's differ from K's)
    for name in ("k_scale_tok", "v_scale_tok"):
        t = getattr(inp, name)
        d[name] = None if t is None else t.to(dev)
    return d


def run(inp, backend="auto", out_dtype=torch.float32, dev_inputs=None, replica=0, **kw):
    d = dev_inputs or to_dev(inp)
    bt = d["block_table"] if d["block_table"].dim() == 2 else d["block_table"][replica]
    out = ua.unified_attention(d["q"], d["k_cache"], d["v_cache"], d["cu_seqlens_q"],
                               d["seq_lens_k"], bt, max_seqlen_q=inp.max_seqlen_q,
                               max_seqlen_k=inp.max_seqlen_k, scale=inp.scale,
                               softcap=inp.softcap, window_left=inp.window_left,
                               alibi_slopes=d["alibi_slopes"], qq_bias=d["qq_bias"],
                               sinks=d["sinks"], kv_scale=d["kv_scale"],
                               k_scale_tok=d["k_scale_tok"], v_scale_tok=d["v_scale_tok"],
                               out_dtype=out_dtype,
                               backend=backend, **kw)
    torch.cuda.synchronize()
    return out


def max_err(out, want):
    got = out.detach().cpu().to(torch.float64).numpy()
    return float(np.abs(got - want).max()) if got.size else 0.0


def ulp16(x, dtype):
    """Spacing of the 16-bit type at |x| (normal range), elementwise."""
    mant = 7 if dtype == torch.bfloat16 else 10
    tiny = 2.0 ** -133 if dtype == torch.bfloat16 else 2.0 ** -24
    ax = np.maximum(np.abs(x), 1e-30)
    return np.maximum(2.0 ** (np.floor(np.log2(ax)) - mant), tiny)

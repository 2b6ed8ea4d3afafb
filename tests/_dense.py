"""Independent dense brute-force attention, used only to pin the oracle.

It is written separately from the oracle and shares nothing with it: torch's own
dtype conversions decode the cache, the cache is gathered densely through the block
table, and each (sequence, head) is one masked softmax over a full score matrix
with an extra zero-valued column for the sink.
"""
import math

import numpy as np
import torch


def dense_attention(q, k_cache, v_cache, cu_seqlens_q, seq_lens_k, block_table, *, scale,
                    softcap=0.0, window_left=-1, alibi_slopes=None, qq_bias=None,
                    qq_bias_stride=None, sinks=None, k_scale=1.0, v_scale=1.0, k_scale_tok=None,
                    v_scale_tok=None, **_):
    qd = q.to(torch.float64).numpy()
    kd = k_cache.to(torch.float64).numpy()
    vd = v_cache.to(torch.float64).numpy()
    if k_cache.dtype == torch.float8_e4m3fn:
        # per-token scales [num_blocks, block_size, H_kv] broadcast over the head dim
        kd = kd * (k_scale if k_scale_tok is None else
                   k_scale_tok.to(torch.float64).numpy()[..., None])
        vd = vd * (v_scale if v_scale_tok is None else
                   v_scale_tok.to(torch.float64).numpy()[..., None])
    cu = cu_seqlens_q.numpy()
    sl = seq_lens_k.numpy()
    bt = block_table.numpy()
    nb, bs, hkv, d = kd.shape
    total_q, hq, _ = qd.shape
    grp = hq // hkv
    qq = None if qq_bias is None else qq_bias.to(torch.float64).numpy().ravel()
    out = np.zeros((total_q, hq, d))
    for b in range(len(sl)):
        t0, t1, kl = int(cu[b]), int(cu[b + 1]), int(sl[b])
        ql = t1 - t0
        if ql == 0 or kl == 0:
            continue
        ctx = kl - ql
        blocks = bt[b, : math.ceil(kl / bs)]
        K = kd[blocks].reshape(-1, hkv, d)[:kl]
        V = vd[blocks].reshape(-1, hkv, d)[:kl]
        jj = np.arange(kl)[None, :]
        pos = (ctx + np.arange(ql))[:, None]
        allowed = jj <= pos
        if window_left is not None and window_left >= 0:
            allowed &= (pos - jj) <= window_left
        for h in range(hq):
            g = h // grp
            S = scale * (qd[t0:t1, h, :] @ K[:, g, :].T)
            if softcap and softcap > 0:
                S = softcap * np.tanh(S / softcap)
            if alibi_slopes is not None:
                S = S + float(alibi_slopes[h]) * (jj - ctx)
            if qq is not None:
                rel = jj - ctx
                idx = np.arange(ql)[:, None] * qq_bias_stride + np.clip(rel, 0, None)
                S = S + np.where(rel >= 0, qq[np.minimum(idx, qq.size - 1)], 0.0)
            S = np.where(allowed, S, -np.inf)
            Vh = V[:, g, :]
            if sinks is not None:
                S = np.concatenate([S, np.full((ql, 1), float(sinks[h]))], axis=1)
                Vh = np.concatenate([Vh, np.zeros((1, d))], axis=0)
            m = S.max(axis=1, keepdims=True)
            live = np.isfinite(m[:, 0])
            P = np.zeros_like(S)
            P[live] = np.exp(S[live] - m[live])
            P[live] /= P[live].sum(axis=1, keepdims=True)
            out[t0:t1, h, :] = P @ Vh
    return out

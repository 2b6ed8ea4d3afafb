"""Pins of the CPU oracle against things other than itself (no GPU needed).

* brute force: an independently written dense masked-softmax reference (_dense.py)
* a library routine: torch's float64 scaled_dot_product_attention with an additive
  mask (ALiBi, QQ-bias, causal and window masks) and an extra key for the sink
* decoders: every f16 / bf16 / e4m3 code against torch's own conversions
* invariants: rows sum to 1, block-table permutation, split == one pass, a window
  at least kv_len long is plain causal, per-row shifts, MHA replication
* closed forms: a single key, equal keys, no keys, sinks over equal scores, a
  saturated softcap
"""
import math
from dataclasses import replace

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as W
from tests._dense import dense_attention

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def small_spec(seed=0, **kw):
    base = dict(name="t", seqs=[(1, 37), (5, 18), (7, 7), (3, 40), (0, 9)], num_q_heads=8,
                num_kv_heads=2, head_dim=16, block_size=16, seed=seed)
    base.update(kw)
    return W.Spec(**base)


def run_both(inp, **extra):
    kw = inp.oracle_kwargs()
    kw.update(extra)
    got = oracle.attention(**kw)
    want = dense_attention(**kw)
    return got, want


# ----------------------------------------------------------------------------- decoders

def test_f16_and_bf16_decoders_match_torch_on_all_codes():
    codes = np.arange(1 << 16, dtype=np.uint16)
    f16 = torch.from_numpy(codes.view(np.int16).copy()).view(torch.float16).to(torch.float64)
    bf16 = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    for kind, ref in ((oracle.F16, f16.numpy()), (oracle.BF16, bf16.numpy())):
        got = oracle.decode(codes, kind)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decoder_matches_torch_and_the_spec():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode(codes, oracle.E4M3)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # values fixed by the OCP e4m3fn definition
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6 and got[0x38] == 1.0
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and nan.sum() == 2


# ----------------------------------------------------------------------------- brute force

FEATURES = [
    dict(),
    dict(window=5),
    dict(softcap=0.7),
    dict(alibi=True),
    dict(qq_bias=True, qq_bias_shape=(8, 64), qq_bias_std=0.5),
    dict(sinks=True),
    dict(window=9, sinks=True, alibi=True),
    dict(softcap=1.5, alibi=True, qq_bias=True, qq_bias_shape=(8, 64), qq_bias_std=0.3),
    dict(window=1, softcap=2.0, qq_bias=True, qq_bias_shape=(8, 64), sinks=True),
]


@pytest.mark.parametrize("feat", range(len(FEATURES)))
@pytest.mark.parametrize("dtypes", [(torch.float16, torch.float16), (torch.bfloat16, torch.bfloat16),
                                    (torch.bfloat16, torch.float8_e4m3fn)])
def test_oracle_equals_dense_brute_force(feat, dtypes):
    spec = small_spec(seed=10 + feat, q_dtype=dtypes[0], kv_dtype=dtypes[1], **FEATURES[feat])
    got, want = run_both(W.make(spec))
    assert np.abs(got - want).max() <= 1e-12


@pytest.mark.parametrize("feat", [dict(), dict(window=5, sinks=True), dict(softcap=0.9, alibi=True)])
@pytest.mark.parametrize("bs", [13, 16])
def test_oracle_per_token_scales_equal_dense_brute_force(feat, bs):
    """fp8 with one K and one V scale per cached token (V's scales with other strides)."""
    spec = small_spec(seed=60 + bs, q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn,
                      block_size=bs, per_token_scales=True, **feat)
    inp = W.make(spec)
    assert inp.k_scale_tok.stride() != inp.v_scale_tok.stride()
    got, want = run_both(inp)
    assert np.abs(got - want).max() <= 1e-12


def test_uniform_per_token_scales_equal_the_per_tensor_scale():
    inp = W.make(small_spec(seed=61, q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn,
                            sinks=True, window=9))
    kw = inp.oracle_kwargs()
    ks, vs = float(np.float32(inp.k_scale)), float(np.float32(inp.v_scale))  # float32 values
    kw.update(k_scale=ks, v_scale=vs)
    base = oracle.attention(**kw)
    shape = inp.k_cache.shape[:3]
    kw.update(k_scale_tok=torch.full(shape, ks, dtype=torch.float32),
              v_scale_tok=torch.full(shape[::-1], vs, dtype=torch.float32).permute(2, 1, 0),
              k_scale=7.0, v_scale=9.0)  # ignored when per-token scales are given
    assert np.array_equal(oracle.attention(**kw), base)


@pytest.mark.parametrize("bs", [1, 13, 16, 32, 784])
@pytest.mark.parametrize("heads", [(4, 4), (8, 2), (7, 1), (6, 3)])
def test_oracle_block_sizes_and_groups(bs, heads):
    spec = small_spec(seed=bs + heads[0], num_q_heads=heads[0], num_kv_heads=heads[1],
                      block_size=bs, window=17, sinks=True)
    got, want = run_both(W.make(spec))
    assert np.abs(got - want).max() <= 1e-12


def test_oracle_rows_entry_matches_full_output():
    inp = W.make(small_spec(seed=3, sinks=True, alibi=True, window=6))
    full = oracle.attention(**inp.oracle_kwargs())
    tok = np.array([0, 3, 5, 6, 12, 15], dtype=np.int32)
    hd = np.array([7, 0, 3, 1, 5, 2], dtype=np.int32)
    rows = oracle.attention_rows(tokens=tok, heads=hd, **inp.oracle_kwargs())
    assert np.array_equal(rows, full[tok, hd])


# ----------------------------------------------------------------------------- library routine

def _sdpa_reference(inp):
    """torch SDPA (float64) per sequence with an additive mask and an extra sink key."""
    kw = inp.oracle_kwargs()
    q = inp.q.to(torch.float64)
    kd, vd = inp.k_cache.to(torch.float64), inp.v_cache.to(torch.float64)
    bs, hkv, d = kd.shape[1], kd.shape[2], kd.shape[3]
    H = q.shape[1]
    out = torch.zeros_like(q)
    cu, sl, bt = inp.cu_seqlens_q.tolist(), inp.seq_lens_k.tolist(), inp.block_table
    for b in range(len(sl)):
        t0, t1, kl = cu[b], cu[b + 1], sl[b]
        ql = t1 - t0
        if ql == 0 or kl == 0:
            continue
        ctx = kl - ql
        blocks = bt[b, : math.ceil(kl / bs)].long()
        K = kd[blocks].reshape(-1, hkv, d)[:kl].repeat_interleave(H // hkv, dim=1)
        V = vd[blocks].reshape(-1, hkv, d)[:kl].repeat_interleave(H // hkv, dim=1)
        j = torch.arange(kl, dtype=torch.float64)[None, :]
        i = torch.arange(ql, dtype=torch.float64)[:, None]
        ok = (j <= ctx + i)
        if inp.window_left >= 0:
            ok &= (ctx + i - j) <= inp.window_left
        bias = torch.zeros((H, ql, kl), dtype=torch.float64)
        if inp.alibi_slopes is not None:
            bias += inp.alibi_slopes.to(torch.float64)[:, None, None] * (j - ctx)[None]
        if inp.qq_bias is not None:
            qq = inp.qq_bias.to(torch.float64)
            for ii in range(ql):
                for jj in range(max(ctx, 0), kl):
                    bias[:, ii, jj] += qq[ii, jj - ctx]
        bias = bias.masked_fill(~ok[None], float("-inf"))
        Qh = q[t0:t1].transpose(0, 1)           # [H, ql, d]
        Kh, Vh = K.transpose(0, 1), V.transpose(0, 1)
        if inp.sinks is not None:               # an extra key: zero value, logit = sink
            Kh = torch.cat([Kh, torch.zeros((H, 1, d), dtype=torch.float64)], dim=1)
            Vh = torch.cat([Vh, torch.zeros((H, 1, d), dtype=torch.float64)], dim=1)
            bias = torch.cat([bias, inp.sinks.to(torch.float64)[:, None, None].expand(H, ql, 1)],
                             dim=2)
        o = F.scaled_dot_product_attention(Qh, Kh, Vh, attn_mask=bias, scale=kw["scale"])
        out[t0:t1] = o.transpose(0, 1)
    return out.numpy()


@pytest.mark.parametrize("feat", [dict(), dict(alibi=True), dict(window=4), dict(sinks=True),
                                  dict(qq_bias=True, qq_bias_shape=(8, 64), qq_bias_std=0.4),
                                  dict(alibi=True, sinks=True, window=11)])
def test_oracle_equals_torch_sdpa(feat):
    inp = W.make(small_spec(seed=5, q_dtype=torch.float16, kv_dtype=torch.float16,
                            seqs=[(1, 37), (5, 18), (7, 7), (3, 40)], **feat))
    got = oracle.attention(**inp.oracle_kwargs())
    want = _sdpa_reference(inp)
    assert np.abs(got - want).max() <= 1e-12


# ----------------------------------------------------------------------------- invariants

def test_rows_sum_to_one():
    inp = W.make(small_spec(seed=6, window=8, alibi=True, softcap=3.0))
    inp.v_cache = torch.ones_like(inp.v_cache)
    got = oracle.attention(**inp.oracle_kwargs())
    live = got[: inp.total_q]
    assert np.abs(live - 1.0).max() <= 1e-14
    # with sinks: every component equals 1 - (sink share) < 1
    inp2 = W.make(small_spec(seed=6, sinks=True))
    inp2.v_cache = torch.ones_like(inp2.v_cache)
    got2 = oracle.attention(**inp2.oracle_kwargs())
    assert np.all(got2 < 1.0) and np.all(got2 > 0.0)
    assert np.abs(got2 - got2[..., :1]).max() <= 1e-15


@pytest.mark.parametrize("kv_dtype,per_token", [(torch.float16, False),
                                                (torch.float8_e4m3fn, False),
                                                (torch.float8_e4m3fn, True)])
def test_block_table_permutation_is_bit_exact(kv_dtype, per_token):
    inp = W.make(small_spec(seed=7, kv_dtype=kv_dtype, q_dtype=torch.float16, sinks=True,
                            window=10, num_blocks=24, per_token_scales=per_token))
    base = oracle.attention(**inp.oracle_kwargs())
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(inp.k_cache.shape[0], generator=g)   # new position of block b
    k2 = torch.empty_like(inp.k_cache)
    v2 = torch.empty_like(inp.v_cache)
    k2.view(torch.uint8)[perm] = inp.k_cache.view(torch.uint8)
    v2.view(torch.uint8)[perm] = inp.v_cache.view(torch.uint8)
    bt2 = perm[inp.block_table.long()].to(torch.int32)
    kw = inp.oracle_kwargs()
    kw.update(k_cache=k2, v_cache=v2, block_table=bt2)
    if per_token:  # the scales move with their blocks
        ks2, vs2 = torch.empty_like(inp.k_scale_tok), torch.empty_like(inp.v_scale_tok)
        ks2[perm] = inp.k_scale_tok
        vs2[perm] = inp.v_scale_tok
        kw.update(k_scale_tok=ks2, v_scale_tok=vs2)
    assert np.array_equal(oracle.attention(**kw), base)


@pytest.mark.parametrize("n_part", [1, 2, 3, 7, 16, 64])
@pytest.mark.parametrize("sinks", [False, True])
def test_split_merge_equals_one_pass(n_part, sinks):
    inp = W.make(small_spec(seed=8, sinks=sinks, window=23, alibi=True))
    one = oracle.attention(**inp.oracle_kwargs())
    split = oracle.attention(n_part=n_part, **inp.oracle_kwargs())
    assert np.abs(one - split).max() <= 1e-12


def test_window_at_least_kv_len_is_plain_causal():
    spec = small_spec(seed=9, sinks=True)
    inp = W.make(spec)
    causal = oracle.attention(**inp.oracle_kwargs())
    for wl in (40, 41, 1000):
        kw = inp.oracle_kwargs()
        kw["window_left"] = wl
        assert np.array_equal(oracle.attention(**kw), causal)
    kw = inp.oracle_kwargs()
    kw["window_left"] = 5
    assert not np.array_equal(oracle.attention(**kw), causal)


def test_per_row_shift_invariance_without_sinks():
    # q_len == kv_len (no prefix): a per-row constant in the QQ-bias shifts every allowed
    # score of the row alike, so the softmax (without a sink) must not move.
    spec = small_spec(seed=11, seqs=[(6, 6), (9, 9)], qq_bias=True, qq_bias_shape=(16, 16),
                      qq_bias_std=0.0)
    inp = W.make(spec)
    base = oracle.attention(**inp.oracle_kwargs())
    inp.qq_bias = (torch.arange(16, dtype=torch.float32) * 0.37 - 1.0)[:, None].expand(16, 16)
    inp.qq_bias = inp.qq_bias.contiguous()
    shifted = oracle.attention(**inp.oracle_kwargs())
    assert np.abs(shifted - base).max() <= 1e-13
    # with a sink the shift changes the sink's share, so the output must move
    inp_s = W.make(replace(spec, sinks=True))
    a = oracle.attention(**inp_s.oracle_kwargs())
    inp_s.qq_bias = inp.qq_bias
    b = oracle.attention(**inp_s.oracle_kwargs())
    assert np.abs(a - b).max() > 1e-3


def test_huge_softcap_is_no_softcap_and_minus_inf_sink_is_no_sink():
    inp = W.make(small_spec(seed=12, alibi=True))
    base = oracle.attention(**inp.oracle_kwargs())
    kw = inp.oracle_kwargs()
    kw["softcap"] = 1e30
    assert np.abs(oracle.attention(**kw) - base).max() <= 1e-9
    kw = inp.oracle_kwargs()
    kw["sinks"] = torch.full((inp.spec.num_q_heads,), -1e30)
    assert np.array_equal(oracle.attention(**kw), base)


def test_mha_replication_equals_gqa():
    inp = W.make(small_spec(seed=13, num_q_heads=6, num_kv_heads=2, window=12, sinks=True))
    gqa = oracle.attention(**inp.oracle_kwargs())
    kw = inp.oracle_kwargs()
    kw["k_cache"] = inp.k_cache.repeat_interleave(3, dim=2).contiguous()
    kw["v_cache"] = inp.v_cache.repeat_interleave(3, dim=2).contiguous()
    assert np.array_equal(oracle.attention(**kw), gqa)


# ----------------------------------------------------------------------------- closed forms

def test_single_allowed_key_returns_that_value_row():
    inp = W.make(small_spec(seed=14, sinks=False))
    kw = inp.oracle_kwargs()
    kw["window_left"] = 0          # each row sees only its own position
    got = oracle.attention(**kw)
    vd = inp.v_cache.to(torch.float64)
    bs, G = inp.spec.block_size, inp.spec.num_q_heads // inp.spec.num_kv_heads
    cu, sl = inp.cu_seqlens_q.tolist(), inp.seq_lens_k.tolist()
    for b in range(inp.num_seqs):
        ctx = sl[b] - (cu[b + 1] - cu[b])
        for t in range(cu[b], cu[b + 1]):
            p = ctx + t - cu[b]
            blk = int(inp.block_table[b, p // bs])
            for h in range(inp.spec.num_q_heads):
                assert np.array_equal(got[t, h], vd[blk, p % bs, h // G].numpy())


def test_equal_keys_give_the_mean_value_and_sink_closed_form():
    spec = small_spec(seed=15, seqs=[(3, 12), (1, 20)], window=6)
    inp = W.make(spec)
    inp.k_cache = torch.full_like(inp.k_cache, 0.25)   # every score of a row is equal
    got = oracle.attention(**inp.oracle_kwargs())
    vd = inp.v_cache.to(torch.float64)
    bs, G, D = spec.block_size, spec.num_q_heads // spec.num_kv_heads, spec.head_dim
    cu, sl = inp.cu_seqlens_q.tolist(), inp.seq_lens_k.tolist()
    sinks = torch.linspace(-1.0, 2.0, spec.num_q_heads)
    kw = inp.oracle_kwargs()
    kw["sinks"] = sinks
    got_s = oracle.attention(**kw)
    qd = inp.q.to(torch.float64)
    for b in range(inp.num_seqs):
        ctx = sl[b] - (cu[b + 1] - cu[b])
        for t in range(cu[b], cu[b + 1]):
            p = ctx + t - cu[b]
            keys = list(range(max(0, p - inp.window_left), p + 1))
            for h in range(spec.num_q_heads):
                rows = [vd[int(inp.block_table[b, j // bs]), j % bs, h // G] for j in keys]
                vbar = torch.stack(rows).mean(0).numpy()
                assert np.abs(got[t, h] - vbar).max() <= 1e-14
                s = inp.scale * 0.25 * float(qd[t, h].sum())
                n = len(keys)
                expect = n * math.exp(s) * vbar / (math.exp(float(sinks[h])) + n * math.exp(s))
                assert np.abs(got_s[t, h] - expect).max() <= 1e-13
    assert D == 16


def test_rows_without_keys_are_zero():
    # kv_len 0 (an empty decode slot) and kv_len < q_len: rows before the first key are 0
    spec = small_spec(seed=16, seqs=[(1, 0), (4, 2), (2, 5)], sinks=True)
    inp = W.make(spec)
    got = oracle.attention(**inp.oracle_kwargs())
    assert np.array_equal(got[0], np.zeros_like(got[0]))
    assert np.array_equal(got[1:3], np.zeros_like(got[1:3]))     # positions -2, -1
    assert np.abs(got[3:5]).max() > 0                            # positions 0, 1
    want = dense_attention(**inp.oracle_kwargs())
    assert np.abs(got - want).max() <= 1e-12


def test_saturated_softcap_closed_form():
    # one sequence, q_len 1, kv_len 2: raw scaled scores [+big, 0] -> capped to [c, 0]
    spec = small_spec(seed=17, seqs=[(1, 2)], num_q_heads=1, num_kv_heads=1, head_dim=16,
                      q_dtype=torch.float32, kv_dtype=torch.float16, scale=0.5)
    inp = W.make(spec)
    inp.q = torch.zeros((1, 1, 16), dtype=torch.float32)
    inp.q[0, 0, 0] = 1000.0
    k = torch.zeros_like(inp.k_cache)
    blk = int(inp.block_table[0, 0])
    k[blk, 0, 0, 0] = 1.0              # key 0: raw dot 1000, scaled 500
    inp.k_cache = k
    c = 1.75
    kw = inp.oracle_kwargs()
    kw["softcap"] = c
    got = oracle.attention(**kw)[0, 0]
    vd = inp.v_cache.to(torch.float64)[blk, :2, 0].numpy()
    expect = (math.exp(c) * vd[0] + vd[1]) / (math.exp(c) + 1.0)
    assert np.abs(got - expect).max() <= 1e-14


def test_block_id_out_of_range_is_reported():
    inp = W.make(small_spec(seed=18))
    kw = inp.oracle_kwargs()
    bt = inp.block_table.clone()
    bt[0, 0] = 10_000
    kw["block_table"] = bt
    with pytest.raises(ValueError, match="block id"):
        oracle.attention(**kw)

"""GPU parity: the CUDA path, called through the C ABI, against the fp64 CPU oracle.

Every call runs with unused cache slots and blocks poisoned with NaN (e4m3 code
0x7F), so a read outside the attended keys shows up in the output.  The bar is the
stated one: max abs error 2e-3 for fp16/bf16 caches and 2e-2 for the fp8 cache, on
the fp32-output mode; 16-bit outputs may add one unit in the last place of their type.
"""
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import varlen_gqa_attention_paged_gb300 as ua
import workloads as W
from tests._gpu import TOL, max_err, run, to_dev, ulp16

pytestmark = pytest.mark.gpu
THREADS = min(16, os.cpu_count() or 1)

_ORACLE_CACHE = {}


def oracle_out(inp, key):
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = oracle.attention(threads=THREADS, **inp.oracle_kwargs())
    return _ORACLE_CACHE[key]


_INPUT_CACHE = {}


def inputs(spec):
    if spec.name not in _INPUT_CACHE:
        _INPUT_CACHE[spec.name] = W.make(spec, poison=True)
    return _INPUT_CACHE[spec.name]


FULL = [W.TINY, W.DECODE, W.MIXED, W.SWDECODE_BF16, W.SWDECODE_FP8, W.SWDECODE_FP8_TOK]


@pytest.mark.parametrize("backend", ["auto", "2d", "split"])
@pytest.mark.parametrize("spec", FULL, ids=lambda s: s.name)
def test_workload_parity_fp32_out(spec, backend):
    inp = inputs(spec)
    want = oracle_out(inp, spec.name)
    out = run(inp, backend=backend)
    err = max_err(out, want)
    assert np.isfinite(out.cpu().numpy()).all()
    assert err <= TOL[spec.kv_dtype], f"{spec.name}/{backend}: max abs err {err:.3e}"


@pytest.mark.parametrize("spec", FULL, ids=lambda s: s.name)
def test_workload_parity_16bit_out(spec):
    inp = inputs(spec)
    want = oracle_out(inp, spec.name)
    out = run(inp, backend="auto", out_dtype=spec.q_dtype)
    got = out.cpu().to(torch.float64).numpy()
    bound = TOL[spec.kv_dtype] + ulp16(want, spec.q_dtype)
    assert (np.abs(got - want) <= bound).all()


def _plan(inp, backend="auto", num_splits=0):
    """The dispatcher's decision for an input set on this device."""
    spec = inp.spec
    bt = inp.block_table if inp.block_table.dim() == 2 else inp.block_table[0]
    return ua.plan(num_seqs=inp.num_seqs, total_q=inp.total_q, max_seqlen_q=inp.max_seqlen_q,
                   max_seqlen_k=inp.max_seqlen_k, block_size=spec.block_size,
                   num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                   head_dim=spec.head_dim, window_left=inp.window_left,
                   kv_dtype=ua._DTYPES[spec.kv_dtype], q_dtype=ua._DTYPES[spec.q_dtype],
                   backend=backend, num_splits=num_splits, max_blocks_per_seq=bt.shape[-1],
                   num_blocks=inp.k_cache.shape[0],
                   per_token_scales=inp.k_scale_tok is not None)


def _tile_rows(inp, tokens_per_tile, tiles_per_seq=64):
    """(token, head) rows of every head for the first and last token of `tiles_per_seq`
    q tiles of each sequence, spread from the first tile to the last (both parities of
    the tile index, so both tiles of a two-tile CTA)."""
    cu = inp.cu_seqlens_q.tolist()
    tok = []
    for b in range(inp.num_seqs):
        a, e = cu[b], cu[b + 1]
        n = (e - a + tokens_per_tile - 1) // tokens_per_tile
        for t in sorted(set(np.linspace(0, n - 1, min(n, tiles_per_seq)).round().astype(int))):
            first = a + t * tokens_per_tile
            tok += [first, min(e, first + tokens_per_tile) - 1]
    hq = inp.spec.num_q_heads
    tok = np.repeat(np.array(tok, dtype=np.int32), hq)
    heads = np.tile(np.arange(hq, dtype=np.int32), len(tok) // hq)
    # shuffled, so the oracle's threads get rows of every sequence (and cost) alike
    perm = np.random.default_rng(0).permutation(len(tok))
    return tok[perm], heads[perm]


@pytest.mark.parametrize("spec,kernel", [(W.PREFILL_D128, 16), (W.PREFILL_D128_FP8, 16),
                                         (W.PREFILL_D256, 8), (W.PREFILL_D256_FP8, 8)],
                         ids=["prefill_d128", "prefill_d128_fp8", "prefill_d256",
                              "prefill_d256_fp8"])
def test_long_prefill_sampled_rows(spec, kernel):
    """Full-size prefill in the bench's launch configuration: every head of the first and
    last token of 64 q tiles per sequence (over 15,000 rows) against the oracle, for the
    fp32 output and for the 16-bit output (the oracle's row rounded, plus the bar)."""
    inp = W.make(spec)
    assert _plan(inp)["kernel"] == kernel
    out = run(inp, backend="auto").cpu()
    out16 = run(inp, backend="auto", out_dtype=spec.q_dtype).cpu()
    assert torch.isfinite(out).all() and torch.isfinite(out16.float()).all()
    tq = 128 // (spec.num_q_heads // spec.num_kv_heads)
    tok, heads = _tile_rows(inp, tq)
    assert len(tok) >= 4000
    want = oracle.attention_rows(tokens=tok, heads=heads, threads=THREADS, **inp.oracle_kwargs())
    ti, hi = torch.from_numpy(tok).long(), torch.from_numpy(heads).long()
    got = out[ti, hi].double().numpy()
    err = float(np.abs(got - want).max())
    assert err <= TOL[spec.kv_dtype], f"max abs err {err:.3e}"
    got16 = out16[ti, hi].double().numpy()
    bound = TOL[spec.kv_dtype] + ulp16(want, spec.q_dtype)
    assert (np.abs(got16 - want) <= bound).all()


# Two 128-row q tiles a CTA with a 16-bit cache (plan kernel code 16, the kernel the long
# prefill bench times): enough tokens that the halved grid still fills the device, with
# the window and sinks, every score feature at G = 16, head_dim 64, ragged sequence ends.
TWO_TILE = {
    "pf2_bf16_window_sinks": dict(seqs=[(1500, 1500), (1000, 1600), (300, 300)],
                                  num_q_heads=32, num_kv_heads=8, q_dtype=torch.bfloat16,
                                  kv_dtype=torch.bfloat16, window=256, sinks=True),
    "pf2_f16_g16_feat": dict(seqs=[(1500, 1700), (1300, 1300)], num_q_heads=16,
                             num_kv_heads=1, softcap=30.0, alibi=True, qq_bias=True,
                             qq_bias_shape=(1500, 1500), sinks=True),
    "pf2_bf16_d64_g8_bs32": dict(seqs=[(1000, 1200), (700, 700), (65, 65)], num_q_heads=32,
                                 num_kv_heads=4, head_dim=64, block_size=32,
                                 q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16),
    "pf2_f16_chunk_behind_prefix": dict(seqs=[(1200, 5000), (1100, 1100), (7, 7)],
                                        num_q_heads=32, num_kv_heads=8, window=700),
}


def _two_tile_inputs(case):
    key = "two_tile/" + case
    if key not in _INPUT_CACHE:
        kw = dict(head_dim=128, seed=200 + sorted(TWO_TILE).index(case))
        kw.update(TWO_TILE[case])
        spec = W.Spec(name=case, **kw)
        _INPUT_CACHE[key] = W.make(spec, poison=True)
    return _INPUT_CACHE[key]


@pytest.mark.parametrize("backend", ["auto", "2d", "split"])
@pytest.mark.parametrize("case", sorted(TWO_TILE))
def test_two_tile_prefill_16bit_cache(case, backend):
    inp = _two_tile_inputs(case)
    assert _plan(inp, backend)["kernel"] == 16, "the case must reach the two-tile kernel"
    want = oracle_out(inp, "two_tile/" + case)
    out = run(inp, backend=backend)
    err = max_err(out, want)
    assert err <= TOL[inp.spec.kv_dtype], f"{case}/{backend}: {err:.3e}"
    if backend == "auto":
        out16 = run(inp, backend=backend, out_dtype=inp.spec.q_dtype)
        got = out16.cpu().to(torch.float64).numpy()
        bound = TOL[inp.spec.kv_dtype] + ulp16(want, inp.spec.q_dtype)
        assert (np.abs(got - want) <= bound).all()


def _small(seed, **kw):
    base = dict(name=f"s{seed}", seqs=[(1, 37), (5, 18), (17, 80), (0, 9), (1, 1), (3, 300)],
                num_q_heads=8, num_kv_heads=2, head_dim=128, seed=seed)
    base.update(kw)
    return W.Spec(**base)


SMALL = {
    "d64_g4_bs13": dict(head_dim=64, block_size=13, num_q_heads=8, num_kv_heads=2),
    "d256_g6_window": dict(head_dim=256, num_q_heads=12, num_kv_heads=2, window=33),
    "mha_bs32": dict(num_q_heads=4, num_kv_heads=4, block_size=32),
    "g7_bs64_sinks": dict(num_q_heads=7, num_kv_heads=1, block_size=64, sinks=True),
    "bf16_all_features": dict(q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, softcap=20.0,
                              alibi=True, qq_bias=True, qq_bias_shape=(32, 64), sinks=True,
                              window=50),
    "fp8_f16q_window": dict(kv_dtype=torch.float8_e4m3fn, window=40, sinks=True),
    "fp8_bf16q_d64": dict(kv_dtype=torch.float8_e4m3fn, q_dtype=torch.bfloat16, head_dim=64),
    "bs1_g16": dict(block_size=1, num_q_heads=16, num_kv_heads=1),
    "window1": dict(window=1, sinks=True),
    "kv_shorter_than_q": dict(seqs=[(4, 2), (1, 0), (6, 6), (2, 40)], sinks=True),
    "g32_decode": dict(seqs=[(1, 700), (1, 33)], num_q_heads=32, num_kv_heads=1),
    # prefill-shaped blocks on the tensor-memory kernel: several key tiles, the window and
    # sinks, partial last pages, rows past the last token of a sequence
    "pf_bf16_window_sinks": dict(seqs=[(200, 500), (129, 129), (1, 300), (37, 45)],
                                 num_q_heads=32, num_kv_heads=8, q_dtype=torch.bfloat16,
                                 kv_dtype=torch.bfloat16, window=150, sinks=True),
    "pf_f16_mha_d64_bs32": dict(seqs=[(150, 333), (20, 20)], num_q_heads=4, num_kv_heads=4,
                                head_dim=64, block_size=32),
    "pf_bf16_g16_d256_feat": dict(seqs=[(40, 500), (9, 9)], num_q_heads=16, num_kv_heads=1,
                                  head_dim=256, block_size=64, q_dtype=torch.bfloat16,
                                  kv_dtype=torch.bfloat16, softcap=30.0, alibi=True,
                                  qq_bias=True, qq_bias_shape=(64, 64), sinks=True),
    "pf_f16_g6_chunk": dict(seqs=[(70, 600), (1, 17)], num_q_heads=12, num_kv_heads=2,
                            window=300),
    # fp8 caches on the tensor-memory kernel (head_dim 64 and 128): codes dequantised to f16
    # tiles in shared memory, a bf16 q converted to f16; one and two q tiles a CTA
    "pf_fp8_bf16q_window_sinks": dict(seqs=[(200, 500), (129, 129), (1, 300), (37, 45)],
                                      num_q_heads=32, num_kv_heads=8, q_dtype=torch.bfloat16,
                                      kv_dtype=torch.float8_e4m3fn, window=150, sinks=True),
    "pf_fp8_f16q_g16_feat": dict(seqs=[(150, 600), (9, 9)], num_q_heads=16, num_kv_heads=1,
                                 kv_dtype=torch.float8_e4m3fn, softcap=30.0, alibi=True,
                                 qq_bias=True, qq_bias_shape=(160, 160), sinks=True),
    "pf_fp8_d64_g8_feat": dict(seqs=[(300, 700), (1, 65), (130, 130)], num_q_heads=16,
                               num_kv_heads=2, head_dim=64, block_size=32,
                               kv_dtype=torch.float8_e4m3fn, softcap=25.0, alibi=True,
                               sinks=True, window=200),
    "pf_fp8_d64_bf16q_mha": dict(seqs=[(200, 333), (64, 64)], num_q_heads=4, num_kv_heads=4,
                                 head_dim=64, q_dtype=torch.bfloat16,
                                 kv_dtype=torch.float8_e4m3fn),
    "pf_fp8_bf16q_two_tiles": dict(seqs=[(1500, 1500), (1000, 1600), (300, 300)],
                                   num_q_heads=32, num_kv_heads=8, block_size=32,
                                   q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn,
                                   window=256),
    # fp8 caches at head_dim 256 on the tensor-memory kernel: half tiles of codes staged and
    # dequantised to f16 slots; odd and even tile counts, every score feature at G = 16
    "pf_fp8_d256_window_sinks": dict(seqs=[(130, 390), (1, 129), (64, 64), (257, 900)],
                                     num_q_heads=8, num_kv_heads=2, head_dim=256,
                                     kv_dtype=torch.float8_e4m3fn, window=200, sinks=True),
    "pf_fp8_d256_bf16q_g16_feat": dict(seqs=[(40, 500), (9, 9), (100, 300)], num_q_heads=16,
                                       num_kv_heads=1, head_dim=256, block_size=64,
                                       q_dtype=torch.bfloat16, kv_dtype=torch.float8_e4m3fn,
                                       softcap=30.0, alibi=True, qq_bias=True,
                                       qq_bias_shape=(100, 112), sinks=True),
    # per-token fp8 scales (V's with other strides) on the tensor-memory kernels: each key's
    # row is dequantised times its own scale
    "pf_fp8_tok_d128_window": dict(seqs=[(200, 500), (129, 129), (1, 300), (37, 45)],
                                   num_q_heads=32, num_kv_heads=8, q_dtype=torch.bfloat16,
                                   kv_dtype=torch.float8_e4m3fn, per_token_scales=True,
                                   window=150, sinks=True),
    "pf_fp8_tok_d64_feat": dict(seqs=[(300, 700), (1, 65), (130, 130)], num_q_heads=16,
                                num_kv_heads=2, head_dim=64, block_size=32,
                                kv_dtype=torch.float8_e4m3fn, per_token_scales=True,
                                softcap=25.0, alibi=True, sinks=True),
    "pf_fp8_tok_d256": dict(seqs=[(130, 390), (64, 64), (257, 600)], num_q_heads=8,
                            num_kv_heads=2, head_dim=256, q_dtype=torch.bfloat16,
                            kv_dtype=torch.float8_e4m3fn, per_token_scales=True, window=300),
    # head_dim 256: K and V stream as half tiles through one ring; odd and even tile counts
    "pf_f16_d256_ragged": dict(seqs=[(130, 390), (1, 129), (64, 64), (257, 900)],
                               num_q_heads=8, num_kv_heads=2, head_dim=256),
    "pf_bf16_d256_mha_window_sinks": dict(seqs=[(300, 700), (17, 17)], num_q_heads=4,
                                          num_kv_heads=4, head_dim=256, q_dtype=torch.bfloat16,
                                          kv_dtype=torch.bfloat16, window=200, sinks=True),
    # decode-shaped q-blocks (at most 8 rows per kv-head) with every score feature, a row
    # with no key, partial pages; 128-byte cache rows (fp8 at d128, 16-bit at d64)
    "dec_fp8_feat": dict(seqs=[(1, 700), (2, 129), (1, 1), (1, 17), (1, 0), (4, 333)],
                          num_q_heads=8, num_kv_heads=4, kv_dtype=torch.float8_e4m3fn,
                          q_dtype=torch.bfloat16, softcap=25.0, alibi=True, qq_bias=True,
                          qq_bias_shape=(8, 16), sinks=True, window=260),
    "dec_bf16_d64_window": dict(seqs=[(1, 900), (4, 300), (1, 65)], num_q_heads=8,
                                 num_kv_heads=4, head_dim=64, q_dtype=torch.bfloat16,
                                 kv_dtype=torch.bfloat16, window=200, sinks=True),
    "dec_f16_d64_g8": dict(seqs=[(1, 500), (1, 31), (1, 16)], num_q_heads=16, num_kv_heads=2,
                            head_dim=64, block_size=32),
    # fp8 with per-token K and V scales (V's with other strides), on the decode tile
    "dec_fp8_tok_feat": dict(seqs=[(1, 700), (2, 129), (1, 1), (1, 17), (1, 0), (4, 333)],
                             num_q_heads=8, num_kv_heads=4, kv_dtype=torch.float8_e4m3fn,
                             q_dtype=torch.bfloat16, per_token_scales=True, softcap=25.0,
                             alibi=True, sinks=True, window=260),
    "dec_fp8_tok_d64_bs32": dict(seqs=[(1, 900), (1, 65), (1, 31)], num_q_heads=16,
                                 num_kv_heads=2, head_dim=64, block_size=32,
                                 kv_dtype=torch.float8_e4m3fn, per_token_scales=True),
    # fp8 decode with at most 4 rows per kv-head: two kv-heads a CTA (one page box carries
    # both heads' rows; their q-blocks share the tile's 8 columns).  Every score feature,
    # empty and one-key rows (G 2, q_len 2); columns left empty in each head (G 3), an f16
    # q (three e4m3 terms of Q); head_dim 64 with one head a group and 4-token chunks
    "dec_fp8_pair_feat": dict(seqs=[(1, 700), (2, 129), (1, 1), (1, 17), (1, 0), (2, 333)],
                              num_q_heads=8, num_kv_heads=4, kv_dtype=torch.float8_e4m3fn,
                              q_dtype=torch.bfloat16, softcap=25.0, alibi=True, qq_bias=True,
                              qq_bias_shape=(8, 16), sinks=True, window=260),
    "dec_fp8_pair_g3_f16q": dict(seqs=[(1, 900), (1, 65), (1, 31), (1, 200)], num_q_heads=12,
                                 num_kv_heads=4, block_size=32, kv_dtype=torch.float8_e4m3fn,
                                 sinks=True),
    "dec_fp8_pair_d64_mha": dict(seqs=[(4, 500), (1, 64), (3, 129)], num_q_heads=6,
                                 num_kv_heads=6, head_dim=64, q_dtype=torch.bfloat16,
                                 kv_dtype=torch.float8_e4m3fn, window=100, sinks=True),
    # 9 to 16 rows per kv-head, and head_dim 256: the 16-row tile kernel's decode path
    "tile16_bf16_g8_q2": dict(seqs=[(2, 700), (1, 300), (2, 45), (1, 1)], num_q_heads=16,
                              num_kv_heads=2, q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16,
                              window=300, sinks=True),
    "tile16_fp8_d256": dict(seqs=[(1, 900), (2, 260), (1, 3)], num_q_heads=12, num_kv_heads=2,
                            head_dim=256, kv_dtype=torch.float8_e4m3fn, softcap=30.0,
                            alibi=True),
}


@pytest.mark.parametrize("backend", ["auto", "2d", "split"])
@pytest.mark.parametrize("case", sorted(SMALL))
def test_small_cases(case, backend):
    spec = _small(100 + sorted(SMALL).index(case), **SMALL[case])
    inp = W.make(spec, poison=True)
    want = oracle.attention(threads=THREADS, **inp.oracle_kwargs())
    out = run(inp, backend=backend)
    err = max_err(out, want)
    assert err <= TOL[spec.kv_dtype], f"{case}/{backend}: {err:.3e}"


@pytest.mark.parametrize("n_part", [2, 3, 7, 16, 64])
def test_forced_partition_counts(n_part):
    inp = inputs(W.SWDECODE_BF16)
    want = oracle_out(inp, W.SWDECODE_BF16.name)
    out = run(inp, backend="split", num_splits=n_part)
    assert max_err(out, want) <= 2e-3


@pytest.mark.parametrize("kv,decode,tok", [(torch.float16, False, False),
                                           (torch.float8_e4m3fn, False, False),
                                           (torch.float8_e4m3fn, True, False),
                                           (torch.float8_e4m3fn, True, True)])
def test_block_table_permutation_is_bit_exact(kv, decode, tok):
    extra = dict(seqs=[(1, 300), (1, 45), (2, 100)], num_q_heads=8, num_kv_heads=4) if decode else {}
    spec = _small(7, kv_dtype=kv, window=100, sinks=True, num_blocks=80, per_token_scales=tok,
                  **extra)
    inp = W.make(spec)
    base = run(inp, backend="split").cpu()
    perm = torch.randperm(inp.k_cache.shape[0], generator=torch.Generator().manual_seed(5))
    k2, v2 = torch.empty_like(inp.k_cache), torch.empty_like(inp.v_cache)
    k2.view(torch.uint8)[perm] = inp.k_cache.view(torch.uint8)
    v2.view(torch.uint8)[perm] = inp.v_cache.view(torch.uint8)
    inp2 = replace(inp, k_cache=k2, v_cache=v2, block_table=perm[inp.block_table.long()].int())
    if tok:  # the scales move with their blocks
        ks2, vs2 = torch.empty_like(inp.k_scale_tok), torch.empty_like(inp.v_scale_tok)
        ks2[perm] = inp.k_scale_tok
        vs2[perm] = inp.v_scale_tok
        inp2 = replace(inp2, k_scale_tok=ks2, v_scale_tok=vs2)
    for backend in ("split", "2d"):
        ref = run(inp, backend=backend).cpu()
        got = run(inp2, backend=backend).cpu()
        assert torch.equal(ref.view(torch.int32), got.view(torch.int32))
    assert base.shape == ref.shape


def test_e4m3_dequant_of_all_codes_is_exact():
    """kv_len 1 makes out = V row * v_scale exactly: the device decode of every code."""
    spec = W.Spec("codes", [(1, 1), (1, 1)], 1, 1, 128, kv_dtype=torch.float8_e4m3fn,
                  q_dtype=torch.float16, seed=3, num_blocks=2)
    inp = W.make(spec)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    v = torch.zeros_like(inp.v_cache.view(torch.uint8))
    b0, b1 = int(inp.block_table[0, 0]), int(inp.block_table[1, 0])
    v[b0, 0, 0] = codes[:128]
    v[b1, 0, 0] = codes[128:]
    inp.v_cache = v.view(torch.float8_e4m3fn)
    inp.k_scale, inp.v_scale = 1.0, 1.0
    out = run(inp, backend="2d").cpu().double().numpy().reshape(-1)
    want = oracle.decode(codes.numpy(), oracle.E4M3)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(out), nan)
    assert np.array_equal(out[~nan], want[~nan])


def test_two_streams_share_nothing():
    a, b = inputs(W.SWDECODE_BF16), inputs(W.DECODE)
    da, db = to_dev(a), to_dev(b)
    wa, wb = oracle_out(a, W.SWDECODE_BF16.name), oracle_out(b, W.DECODE.name)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            oa = run(a, backend="split", dev_inputs=da)
        with torch.cuda.stream(s2):
            ob = run(b, backend="split", dev_inputs=db)
        outs.append((oa, ob))
    torch.cuda.synchronize()
    for oa, ob in outs:
        assert max_err(oa, wa) <= 2e-3 and max_err(ob, wb) <= 2e-3


def test_library_workspace_reuse_across_head_sizes():
    for d in (64, 128, 256, 64):
        spec = _small(20 + d, head_dim=d, seqs=[(1, 900), (2, 1500)], sinks=True)
        inp = W.make(spec, poison=True)
        want = oracle.attention(threads=THREADS, **inp.oracle_kwargs())
        assert max_err(run(inp, backend="split", num_splits=9), want) <= 2e-3


def test_caller_workspace_and_too_small_workspace():
    # 20 partitions: more than a cluster holds, so the merge kernel and its scratch
    inp = inputs(W.SWDECODE_BF16)
    want = oracle_out(inp, W.SWDECODE_BF16.name)
    need = ua.plan(num_seqs=inp.num_seqs, total_q=inp.total_q, max_seqlen_q=inp.max_seqlen_q,
                   max_seqlen_k=inp.max_seqlen_k, block_size=16, num_q_heads=32,
                   num_kv_heads=8, head_dim=128, window_left=inp.window_left,
                   kv_dtype=ua.UA_DT_BF16, backend="split", num_splits=20)["workspace_bytes"]
    assert need > 0
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN-filled scratch
    assert max_err(run(inp, backend="split", num_splits=20, workspace=ws), want) <= 2e-3
    with pytest.raises(ua.UaError) as e:
        run(inp, backend="split", num_splits=20, workspace=ws[: need - 256])
    assert e.value.code == ua._lib.UA_ERR_WORKSPACE


def test_cluster_merge_partition_counts():
    """Up to 16 partitions of a decode-shaped q-block merge inside their cluster through
    distributed shared memory (clusters of 2 to 16 CTAs, 1 to 4 kv-heads per cluster)."""
    for spec in (W.SWDECODE_BF16, W.SWDECODE_FP8, W.DECODE):
        inp = inputs(spec)
        want = oracle_out(inp, spec.name)
        for n_part in (2, 3, 5, 8, 11, 16):
            got = run(inp, backend="split", num_splits=n_part)
            assert max_err(got, want) <= TOL[spec.kv_dtype], (spec.name, n_part)


@pytest.mark.parametrize("spec,kw", [(W.SWDECODE_BF16, {}),
                                     (W.SWDECODE_FP8, dict(backend="split", num_splits=20)),
                                     (W.MIXED, {})],
                         ids=["cluster-merge", "merge-kernel-workspace", "tensor-memory-split"])
def test_cuda_graph_capture_and_replay(spec, kw):
    """A call captured in a CUDA graph replays with new inputs copied into the captured
    buffers (after one warm-up call has configured the kernels and sized the library's
    workspace): the in-cluster merge, the merge kernel over the library workspace, and
    the tensor-memory kernel's split."""
    inp = W.make(spec, poison=True, replicas=2)
    d = to_dev(inp)
    bt = d["block_table"][0].clone()
    q = d["q"].clone()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def call():
        ua.unified_attention(q, d["k_cache"], d["v_cache"], d["cu_seqlens_q"], d["seq_lens_k"],
                             bt, max_seqlen_q=inp.max_seqlen_q, max_seqlen_k=inp.max_seqlen_k,
                             scale=inp.scale, softcap=inp.softcap, window_left=inp.window_left,
                             alibi_slopes=d["alibi_slopes"], qq_bias=d["qq_bias"],
                             sinks=d["sinks"], kv_scale=d["kv_scale"], out=out, stream=stream,
                             **kw)

    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    for replica, qmul in ((1, 0.5), (0, 1.0)):
        bt.copy_(d["block_table"][replica])
        q.copy_(d["q"] * qmul)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        kwargs = inp.oracle_kwargs(replica)
        kwargs["q"] = inp.q * qmul
        want = oracle.attention(threads=THREADS, **kwargs)
        assert max_err(out, want) <= TOL[spec.kv_dtype], (spec.name, replica)


def test_per_token_scales_on_the_tile_kernel_are_unsupported():
    # 9 to 16 rows per kv-head (the 16-row tile kernel): no per-token scales there
    inp = W.make(_small(11, seqs=[(2, 300), (1, 40)], num_q_heads=16, num_kv_heads=2,
                        kv_dtype=torch.float8_e4m3fn, per_token_scales=True))
    assert _plan(inp)["kernel"] == 1
    with pytest.raises(ua.UaError) as e:
        run(inp)
    assert e.value.code == ua._lib.UA_ERR_UNSUPPORTED
    # pages not a multiple of 16 (the 64-row tile kernel): neither
    inp = W.make(_small(13, block_size=13, kv_dtype=torch.float8_e4m3fn, per_token_scales=True))
    assert _plan(inp)["kernel"] == 4
    with pytest.raises(ua.UaError) as e:
        run(inp)
    assert e.value.code == ua._lib.UA_ERR_UNSUPPORTED
    # only one of the two scale arrays
    inp = W.make(_small(12, seqs=[(1, 100)], kv_dtype=torch.float8_e4m3fn, per_token_scales=True))
    with pytest.raises(ValueError):
        run(replace(inp, v_scale_tok=None))


def test_both_decode_tile_widths_run():
    """The decode parity cases reach both widths of the decode tile on this device: four
    consumer warps (three CTAs an SM) on the sliding-window decode, eight (one CTA an SM)
    on a small decode grid."""
    assert _plan(inputs(W.SWDECODE_BF16))["kernel"] == 2
    spec = _small(100 + sorted(SMALL).index("dec_fp8_feat"), **SMALL["dec_fp8_feat"])
    inp = W.make(spec, poison=True)
    assert _plan(inp, "2d")["kernel"] == 32
    want = oracle.attention(threads=THREADS, **inp.oracle_kwargs())
    assert max_err(run(inp, backend="2d"), want) <= TOL[spec.kv_dtype]


def test_two_kv_heads_per_decode_tile():
    """fp8 decode batches of at most 4 rows per kv-head (an even kv-head count, per-tensor
    scales) run two kv-heads a CTA: the sliding-window fp8 decode and the pair cases above;
    8 rows a kv-head, or per-token scales, keep one head a CTA."""
    assert _plan(inputs(W.SWDECODE_FP8))["kernel"] == 64
    assert _plan(inputs(W.SWDECODE_FP8_TOK))["kernel"] == 2
    for case in ("dec_fp8_pair_feat", "dec_fp8_pair_g3_f16q", "dec_fp8_pair_d64_mha"):
        spec = _small(100 + sorted(SMALL).index(case), **SMALL[case])
        inp = W.make(spec, poison=True)
        for backend in ("auto", "2d", "split"):
            assert _plan(inp, backend)["kernel"] == 64, (case, backend)
    spec = _small(100 + sorted(SMALL).index("dec_fp8_feat"), **SMALL["dec_fp8_feat"])
    assert _plan(W.make(spec), "2d")["kernel"] in (2, 32)


def test_out_of_range_block_id_is_reported_not_read():
    inp = W.make(_small(9))
    bt = inp.block_table.clone()
    bt[2, 1] = 10 ** 6
    inp2 = replace(inp, block_table=bt)
    ua.device_status_reset()
    out = run(inp2, backend="2d")
    assert ua.device_status() == ua._lib.UA_ERR_DEVICE_CHECK
    ua.device_status_reset()
    assert ua.device_status() == 0
    assert torch.isfinite(out).all()

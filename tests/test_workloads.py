"""The seeded input recipe (CPU only): block tables over distinct physical blocks, the
1.25x cache, NaN in every slot no sequence owns, per-tensor and per-token fp8 scales of
absmax / 448, replicas on disjoint blocks, and the same draw for the same seed."""
import math
from dataclasses import replace

import torch

import workloads as W

SPEC = W.Spec("t", [(3, 40), (1, 17), (0, 5), (6, 6)], 8, 2, 64, block_size=16, seed=11)


def _owned(inp, bt):
    bs = inp.spec.block_size
    owned = torch.zeros(inp.k_cache.shape[:2], dtype=torch.bool)
    for s, (_, kv) in enumerate(inp.spec.seqs):
        for j in range(kv):
            owned[int(bt[s, j // bs]), j % bs] = True
    return owned


def test_block_table_uses_distinct_blocks_of_a_cache_a_quarter_larger():
    inp = W.make(SPEC)
    need = W.blocks_needed(SPEC.seqs, SPEC.block_size)
    assert inp.k_cache.shape[0] == math.ceil(1.25 * need)
    ids = [int(inp.block_table[s, j]) for s, (_, kv) in enumerate(SPEC.seqs)
           for j in range(math.ceil(kv / SPEC.block_size))]
    assert len(ids) == len(set(ids)) == need
    assert all(0 <= i < inp.k_cache.shape[0] for i in ids)
    assert inp.cu_seqlens_q.tolist() == [0, 3, 4, 4, 10]
    assert inp.seq_lens_k.tolist() == [40, 17, 5, 6]


def test_poison_fills_exactly_the_slots_no_sequence_owns():
    for kv_dtype in (torch.float16, torch.bfloat16, torch.float8_e4m3fn):
        inp = W.make(replace(SPEC, kv_dtype=kv_dtype), poison=True)
        owned = _owned(inp, inp.block_table)
        for cache in (inp.k_cache, inp.v_cache):
            nan = torch.isnan(cache.float()).any(dim=-1).any(dim=-1)
            assert torch.equal(nan, ~owned)
            assert torch.isnan(cache.float())[~owned].all()


def test_fp8_per_tensor_scales_are_absmax_over_448_of_the_owned_slots():
    inp = W.make(replace(SPEC, kv_dtype=torch.float8_e4m3fn))
    owned = _owned(inp, inp.block_table)
    for cache, scale in ((inp.k_cache, inp.k_scale), (inp.v_cache, inp.v_scale)):
        codes = cache.float()[owned]
        # the largest owned magnitude quantises to the top code
        assert float(codes.abs().max()) == W.F8_MAX
        assert scale > 0


def test_fp8_per_token_scales_put_every_row_maximum_on_the_top_code():
    inp = W.make(replace(SPEC, kv_dtype=torch.float8_e4m3fn, per_token_scales=True))
    assert inp.k_scale_tok.shape == inp.k_cache.shape[:3]
    assert inp.v_scale_tok.shape == inp.v_cache.shape[:3]
    assert inp.k_scale_tok.stride() != inp.v_scale_tok.stride()  # V's scales: other strides
    for cache in (inp.k_cache, inp.v_cache):
        row_max = cache.float().abs().amax(dim=-1)
        assert torch.all(row_max == W.F8_MAX)


def test_replicas_use_disjoint_blocks_and_one_seed_one_draw():
    reps = W.make(SPEC, replicas=3)
    assert reps.block_table.shape[0] == 3
    sets = []
    for r in range(3):
        bt = reps.block_table[r]
        sets.append({int(bt[s, j]) for s, (_, kv) in enumerate(SPEC.seqs)
                     for j in range(math.ceil(kv / SPEC.block_size))})
    assert not (sets[0] & sets[1]) and not (sets[1] & sets[2]) and not (sets[0] & sets[2])
    a, b = W.make(SPEC), W.make(SPEC)
    for x, y in ((a.q, b.q), (a.k_cache, b.k_cache), (a.block_table, b.block_table)):
        assert torch.equal(x.view(torch.uint8) if x.dtype.is_floating_point else x,
                           y.view(torch.uint8) if y.dtype.is_floating_point else y)

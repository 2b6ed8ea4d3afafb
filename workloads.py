"""Seeded synthetic inputs for unified paged varlen GQA attention.

This module only draws inputs; it holds none of the attention arithmetic.  Both
the CUDA path (tests, bench, smoke) and the CPU oracle read what it returns.

Workloads follow the scenario shapes of the pages: the RocKE unified-attention
harness scenario table ("Scenarios": decode_d128_b16, mixed_d128_b16 with ALiBi /
softcap / QQ-bias variants), the aiter split-K decode PR ("Performance": batch 8,
ctx ~6700, sliding window 4096, fp8 KV) and the FA-RDNA2 prefill benchmark
(prompts of 4k tokens, a 2k chunk behind a 16k prefix, heads 32/8 d128 and 24/4
d256).  Every tensor is drawn from a seeded ``torch.Generator`` on the CPU.

Layout (contiguous):
  q            [total_q, H_q, D]                 f16 / bf16
  k_cache      [num_blocks, block_size, H_kv, D] f16 / bf16 / float8_e4m3fn
  v_cache      same as k_cache
  block_table  [num_seqs, max_blocks_per_seq]    int32, a seeded permutation of
               physical blocks (with ``replicas`` > 1: [replicas, num_seqs, max_blocks],
               each replica a disjoint set of physical blocks)
  cu_seqlens_q [num_seqs + 1] int32, seq_lens_k [num_seqs] int32
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

F8_MAX = 448.0  # largest finite e4m3fn value


@dataclass
class Spec:
    """Shape and feature recipe of one workload."""
    name: str
    seqs: list                 # [(q_len, kv_len), ...]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int = 16
    q_dtype: torch.dtype = torch.float16
    kv_dtype: torch.dtype = torch.float16   # float8_e4m3fn for the fp8 cache
    seed: int = 0
    num_blocks: Optional[int] = None        # default: ceil(1.25 * needed)
    window: Optional[int] = None            # keys incl. self; window_left = window - 1
    softcap: float = 0.0
    alibi: bool = False
    qq_bias: bool = False
    qq_bias_shape: tuple = (256, 256)
    qq_bias_std: float = 0.1
    sinks: bool = False
    scale: Optional[float] = None           # default 1/sqrt(D)
    per_token_scales: bool = False          # fp8: one K and one V scale per cached token
    desc: str = ""


@dataclass
class Inputs:
    spec: Spec
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    cu_seqlens_q: torch.Tensor
    seq_lens_k: torch.Tensor
    block_table: torch.Tensor
    scale: float
    softcap: float
    window_left: int
    alibi_slopes: Optional[torch.Tensor]
    qq_bias: Optional[torch.Tensor]
    qq_bias_stride: int
    sinks: Optional[torch.Tensor]
    k_scale: float = 1.0
    v_scale: float = 1.0
    # fp8 per-token scales [num_blocks, block_size, H_kv] (float32; V's with other strides)
    k_scale_tok: Optional[torch.Tensor] = None
    v_scale_tok: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)

    @property
    def q_lens(self):
        return [a for a, _ in self.spec.seqs]

    @property
    def kv_lens(self):
        return [b for _, b in self.spec.seqs]

    @property
    def num_seqs(self):
        return len(self.spec.seqs)

    @property
    def total_q(self):
        return int(sum(self.q_lens))

    @property
    def max_seqlen_q(self):
        return max(self.q_lens) if self.spec.seqs else 0

    @property
    def max_seqlen_k(self):
        return max(self.kv_lens) if self.spec.seqs else 0

    def oracle_kwargs(self, replica: int = 0):
        """Keyword arguments of ``oracle.attention`` for this input set."""
        bt = self.block_table if self.block_table.dim() == 2 else self.block_table[replica]
        return dict(q=self.q, k_cache=self.k_cache, v_cache=self.v_cache,
                    cu_seqlens_q=self.cu_seqlens_q, seq_lens_k=self.seq_lens_k, block_table=bt,
                    scale=self.scale, softcap=self.softcap, window_left=self.window_left,
                    alibi_slopes=self.alibi_slopes, qq_bias=self.qq_bias,
                    qq_bias_stride=self.qq_bias_stride if self.qq_bias is not None else None,
                    sinks=self.sinks, k_scale=self.k_scale, v_scale=self.v_scale,
                    k_scale_tok=self.k_scale_tok, v_scale_tok=self.v_scale_tok)


def alibi_slopes(num_heads: int) -> torch.Tensor:
    """Geometric ALiBi slopes 2^(-8 (h+1) / H) for heads h = 0..H-1."""
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / num_heads) for h in range(num_heads)],
                        dtype=torch.float32)


def blocks_needed(seqs, block_size):
    return sum(math.ceil(kv / block_size) for _, kv in seqs)


def make(spec: Spec, *, poison: bool = False, replicas: int = 1) -> Inputs:
    """Draw one input set.

    poison:   fill every cache slot that no sequence owns (tails of last blocks and
              unused physical blocks) with NaN (e4m3 code 0x7F for fp8), so any
              read of it shows up in the output.
    replicas: number of independent block tables over disjoint physical blocks of
              one larger cache (used to rotate the working set past L2).
    """
    g = torch.Generator().manual_seed(spec.seed)
    seqs = spec.seqs
    H, Hk, D, bs = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    if H % Hk:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    per_seq = [math.ceil(kv / bs) for _, kv in seqs]
    need = sum(per_seq)
    nb_one = spec.num_blocks if spec.num_blocks is not None else max(1, math.ceil(1.25 * need))
    if nb_one < need:
        raise ValueError("num_blocks below the blocks the sequences need")
    nb = nb_one * replicas
    max_blocks = max([1] + per_seq)
    total_q = sum(a for a, _ in seqs)

    q = torch.randn((total_q, H, D), generator=g, dtype=torch.float32).to(spec.q_dtype)
    kf = torch.randn((nb, bs, Hk, D), generator=g, dtype=torch.float32)
    vf = torch.randn((nb, bs, Hk, D), generator=g, dtype=torch.float32)

    tables = []
    for r in range(replicas):
        perm = torch.randperm(nb_one, generator=g) + r * nb_one
        bt = torch.zeros((len(seqs), max_blocks), dtype=torch.int32)
        pos = 0
        for s, n in enumerate(per_seq):
            bt[s, :n] = perm[pos:pos + n].to(torch.int32)
            pos += n
        tables.append(bt)
    block_table = tables[0] if replicas == 1 else torch.stack(tables)

    used = torch.zeros((nb, bs), dtype=torch.bool)
    for bt in tables:
        for s, (_, kv) in enumerate(seqs):
            for j in range(per_seq[s]):
                n_slots = min(bs, kv - j * bs)
                used[int(bt[s, j]), :n_slots] = True

    k_scale = v_scale = 1.0
    k_tok = v_tok = None
    if spec.kv_dtype == torch.float8_e4m3fn and spec.per_token_scales:
        # one scale per (block, slot, kv-head) row: absmax / 448 (1 for an all-zero row);
        # V's scales live in a [H_kv, blocks, slots] buffer viewed as [blocks, slots, H_kv]
        # so that K and V scales have different strides
        def row_scale(x):
            s = x.abs().amax(dim=-1) / F8_MAX
            return torch.where(s > 0, s, torch.ones_like(s)).to(torch.float32)
        k_tok = row_scale(kf).contiguous()
        v_tok = row_scale(vf).permute(2, 0, 1).contiguous().permute(1, 2, 0)
        k_cache = (kf / k_tok[..., None]).clamp(-F8_MAX, F8_MAX).to(torch.float8_e4m3fn)
        v_cache = (vf / v_tok[..., None]).clamp(-F8_MAX, F8_MAX).to(torch.float8_e4m3fn)
        if poison:  # scales of slots no sequence owns: never read
            k_tok[~used] = float("nan")
            v_tok[~used] = float("nan")
    elif spec.kv_dtype == torch.float8_e4m3fn:
        k_scale = float(kf[used].abs().max()) / F8_MAX if used.any() else 1.0
        v_scale = float(vf[used].abs().max()) / F8_MAX if used.any() else 1.0
        k_cache = (kf / k_scale).clamp(-F8_MAX, F8_MAX).to(torch.float8_e4m3fn)
        v_cache = (vf / v_scale).clamp(-F8_MAX, F8_MAX).to(torch.float8_e4m3fn)
    else:
        k_cache = kf.to(spec.kv_dtype)
        v_cache = vf.to(spec.kv_dtype)
    if poison:
        mask = ~used
        if spec.kv_dtype == torch.float8_e4m3fn:
            k_cache.view(torch.uint8)[mask] = 0x7F
            v_cache.view(torch.uint8)[mask] = 0x7F
        else:
            k_cache[mask] = float("nan")
            v_cache[mask] = float("nan")

    cu = torch.zeros(len(seqs) + 1, dtype=torch.int32)
    for s, (a, _) in enumerate(seqs):
        cu[s + 1] = cu[s] + a
    sl = torch.tensor([kv for _, kv in seqs], dtype=torch.int32)

    alibi = alibi_slopes(H) if spec.alibi else None
    qq = None
    if spec.qq_bias:
        qq = torch.randn(spec.qq_bias_shape, generator=g, dtype=torch.float32) * spec.qq_bias_std
    sinks = torch.randn((H,), generator=g, dtype=torch.float32) if spec.sinks else None
    return Inputs(spec=spec, q=q, k_cache=k_cache, v_cache=v_cache, cu_seqlens_q=cu,
                  seq_lens_k=sl, block_table=block_table,
                  scale=spec.scale if spec.scale is not None else 1.0 / math.sqrt(D),
                  softcap=spec.softcap,
                  window_left=(spec.window - 1) if spec.window else -1,
                  alibi_slopes=alibi, qq_bias=qq,
                  qq_bias_stride=spec.qq_bias_shape[1] if spec.qq_bias else 0,
                  sinks=sinks, k_scale=k_scale, v_scale=v_scale, k_scale_tok=k_tok,
                  v_scale_tok=v_tok)


# --- the workloads ----------------------------------------------------------------

TINY = Spec("tiny_fp16", [(1, 37), (5, 18)], 4, 2, 64, block_size=16, num_blocks=8, seed=0,
            desc="2 seqs (1,37),(5,18); 4q/2kv; d64; bs16; 8 physical blocks; causal")
DECODE = Spec("decode_fp16", [(1, 512), (1, 1024), (1, 2048), (1, 4096)], 16, 2, 128, seed=1,
              desc="4 decode seqs kv 512..4096; 16q/2kv; d128; bs16; fp16")
MIXED = Spec("mixed_bf16", [(1, 1328), (5, 18), (129, 463), (64, 64), (128, 256)], 16, 2, 128,
             q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=2, softcap=50.0, alibi=True,
             qq_bias=True, desc="5 seqs mixed prefill+decode; ALiBi, softcap 50, QQ-bias; bf16")
SWDECODE_BF16 = Spec("swdecode_bf16", [(1, 6700)] * 8, 32, 8, 128, q_dtype=torch.bfloat16,
                     kv_dtype=torch.bfloat16, seed=3, window=4096, sinks=True,
                     desc="batch 8 decode, kv 6700, window 4096, sinks; 32q/8kv; bf16 KV")
SWDECODE_FP8 = replace(SWDECODE_BF16, name="swdecode_fp8", kv_dtype=torch.float8_e4m3fn,
                       desc="batch 8 decode, kv 6700, window 4096, sinks; 32q/8kv; fp8 e4m3 KV")
SWDECODE_FP8_TOK = replace(SWDECODE_FP8, name="swdecode_fp8_tok", per_token_scales=True,
                           desc="batch 8 decode, kv 6700, window 4096, sinks; 32q/8kv; fp8 e4m3 "
                                "KV with per-token K and V scales")
PREFILL_D128 = Spec("prefill_d128", [(4096, 4096)] * 4 + [(2048, 18432)], 32, 8, 128,
                    q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, seed=4,
                    desc="4x4096 prompts + 2048 chunk behind 16384 prefix; 32q/8kv d128; bf16")
PREFILL_D128_FP8 = replace(PREFILL_D128, name="prefill_d128_fp8", kv_dtype=torch.float8_e4m3fn,
                           desc="4x4096 prompts + 2048 chunk behind 16384 prefix; 32q/8kv d128; "
                                "bf16 q, fp8 e4m3 KV")
PREFILL_D256 = replace(PREFILL_D128, name="prefill_d256", num_q_heads=24, num_kv_heads=4,
                       head_dim=256,
                       desc="4x4096 prompts + 2048 chunk behind 16384 prefix; 24q/4kv d256; bf16")
PREFILL_D256_FP8 = replace(PREFILL_D256, name="prefill_d256_fp8", kv_dtype=torch.float8_e4m3fn,
                           desc="4x4096 prompts + 2048 chunk behind 16384 prefix; 24q/4kv d256; "
                                "bf16 q, fp8 e4m3 KV")

WORKLOADS = {s.name: s for s in (TINY, DECODE, MIXED, SWDECODE_BF16, SWDECODE_FP8,
                                 SWDECODE_FP8_TOK, PREFILL_D128, PREFILL_D128_FP8, PREFILL_D256,
                                 PREFILL_D256_FP8)}


def kv_bytes_read(inp: Inputs) -> int:
    """Algorithmic K+V bytes: every attended key's K and V row read once per kv-head (with
    per-token fp8 scales, also its two 4-byte scales)."""
    spec = inp.spec
    esz = torch.empty((), dtype=spec.kv_dtype).element_size()
    total = 0
    for a, kv in spec.seqs:
        ctx = kv - a
        lo_first = 0 if inp.window_left < 0 else max(0, ctx - inp.window_left)
        total += (kv - lo_first)  # keys touched by at least one row of the sequence
    per_key = spec.head_dim * esz + (4 if spec.per_token_scales else 0)
    return total * spec.num_kv_heads * per_key * 2


def causal_pairs(inp: Inputs) -> int:
    """Number of attended (query row, key) pairs per head."""
    n = 0
    for a, kv in inp.spec.seqs:
        ctx = kv - a
        for i in range(a):
            p = ctx + i
            lo = 0 if inp.window_left < 0 else max(0, p - inp.window_left)
            n += p + 1 - lo
    return n


def attention_flops(inp: Inputs) -> int:
    """Algorithmic FLOPs 4 * D * H_q * attended pairs (QK^T and P.V, 2 FLOPs per MAC)."""
    return 4 * inp.spec.head_dim * inp.spec.num_q_heads * causal_pairs(inp)

"""Seeded synthetic inputs for the paged KV cache hot path.

This module only draws inputs: sequence lengths, block tables, and bf16
query/key/value values.  It holds none of the method's arithmetic (no slot
mapping, no scatter, no attention), so both the CUDA path and the CPU oracle
can consume what it produces without sharing any of the computation.

Workloads are shaped like the attention layer of Qwen3-0.6B that the pages
walk through ("L17: Qwen3 attention sub-layer", §3: 16 query heads, 8 kv
heads, head_dim 128; §7: bf16 weights, block_size 256, a paged pool of
about two thousand blocks).  Values are fp32 N(0, 1) draws passed through a
per-head RMSNorm over head_dim (eps 1e-6, unit weight -- the norm of
"Nano-VLLM full-code notes (5): layernorm & attention") and rounded to bf16;
cache history that predates the step is plain N(0, 1) in bf16.

Block tables: a seeded permutation of the block pool; sequence i takes the
next ceil(len_i / block_size) entries of the permutation and the rest of its
row is -1 (the padding value of "Lesson 04: where exactly does the KV go",
§1).  Padding rows of a CUDA-graph decode batch have context length 0 and a
row of -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

SEED_BASE = 303


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, gen: torch.Generator, rmsnorm: bool = True) -> torch.Tensor:
    """fp32 N(0,1) draws, optionally RMS-normalised over the last dim, as bf16."""
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=gen.device)
    if rmsnorm:
        x = x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + 1e-6)
    return x.to(torch.bfloat16)


def fill_normal_(t: torch.Tensor, seed: int, chunk: int = 1 << 26) -> torch.Tensor:
    """Fill a bf16 tensor in place with seeded N(0,1) values, chunk by chunk,
    on whatever device it lives on."""
    g = generator(seed, t.device)
    flat = t.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=g, dtype=torch.float32,
                                    device=t.device).to(torch.bfloat16)
    return t


def block_tables_from_perm(nblocks_per_seq, num_blocks: int, gen: torch.Generator,
                           width: Optional[int] = None) -> torch.Tensor:
    perm = torch.randperm(num_blocks, generator=gen).to(torch.int32)
    need = int(sum(nblocks_per_seq))
    if need > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
    width = width or max(1, max(nblocks_per_seq) if len(nblocks_per_seq) else 1)
    bt = torch.full((len(nblocks_per_seq), width), -1, dtype=torch.int32)
    pos = 0
    for i, nb in enumerate(nblocks_per_seq):
        bt[i, :nb] = perm[pos:pos + nb]
        pos += nb
    return bt


@dataclass
class Heads:
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


@dataclass
class PrefillWork:
    """One prefill (or chunked / prefix-cache prefill) step.

    For sequence i the first ``prefix_lens[i]`` tokens are already in the
    cache; ``q_lens[i]`` new tokens are computed.  q/k/v hold the new tokens
    packed back to back (cu_seqlens_q order)."""
    heads: Heads
    q_lens: torch.Tensor          # [B] int32
    prefix_lens: torch.Tensor     # [B] int32 (cached tokens, 0 for a plain prefill)
    cu_seqlens_q: torch.Tensor    # [B+1] int32
    cu_seqlens_k: torch.Tensor    # [B+1] int32 (prefix + new)
    block_tables: torch.Tensor    # [B, width] int32, -1 padded
    q: torch.Tensor               # [N, Hq, d] bf16
    k: torch.Tensor               # [N, Hkv, d] bf16
    v: torch.Tensor               # [N, Hkv, d] bf16
    seed: int = 0
    name: str = ""

    @property
    def num_seqs(self) -> int:
        return int(self.q_lens.numel())

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_seqlen_q(self) -> int:
        return int(self.q_lens.max()) if self.num_seqs else 0

    @property
    def max_seqlen_k(self) -> int:
        return int((self.q_lens + self.prefix_lens).max()) if self.num_seqs else 0

    @property
    def has_prefix(self) -> bool:
        return bool((self.prefix_lens > 0).any())

    def causal_pairs(self) -> int:
        """Number of (query, key) pairs the causal mask admits."""
        c = self.q_lens.to(torch.int64)
        p = self.prefix_lens.to(torch.int64)
        return int((c * p + c * (c + 1) // 2).sum())


@dataclass
class DecodeWork:
    """One decode step: one new token per row.  ``context_lens`` counts the
    new token; a row with context length 0 is padding."""
    heads: Heads
    context_lens: torch.Tensor    # [B] int32
    block_tables: torch.Tensor    # [B, width] int32, -1 padded
    q: torch.Tensor               # [B, Hq, d] bf16
    k: torch.Tensor               # [B, Hkv, d] bf16 (the new token's key)
    v: torch.Tensor               # [B, Hkv, d] bf16
    seed: int = 0
    name: str = ""

    @property
    def batch(self) -> int:
        return int(self.context_lens.numel())

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.batch else 0


def _cu(lens: torch.Tensor) -> torch.Tensor:
    out = torch.zeros(lens.numel() + 1, dtype=torch.int32)
    out[1:] = torch.cumsum(lens.to(torch.int64), 0).to(torch.int32)
    return out


def prefill_work(heads: Heads, q_lens, prefix_lens=None, seed: int = SEED_BASE,
                 width: Optional[int] = None, name: str = "") -> PrefillWork:
    g = generator(seed)
    q_lens = torch.as_tensor(q_lens, dtype=torch.int32)
    prefix_lens = (torch.zeros_like(q_lens) if prefix_lens is None
                   else torch.as_tensor(prefix_lens, dtype=torch.int32))
    total = (q_lens + prefix_lens).tolist()
    nblk = [(t + heads.block_size - 1) // heads.block_size for t in total]
    bt = block_tables_from_perm(nblk, heads.num_blocks, g, width)
    n = int(q_lens.sum())
    q = normal_bf16((n, heads.num_heads, heads.head_dim), g)
    k = normal_bf16((n, heads.num_kv_heads, heads.head_dim), g)
    v = normal_bf16((n, heads.num_kv_heads, heads.head_dim), g)
    return PrefillWork(heads, q_lens, prefix_lens, _cu(q_lens), _cu(q_lens + prefix_lens),
                       bt, q, k, v, seed, name)


def decode_work(heads: Heads, context_lens, seed: int = SEED_BASE,
                width: Optional[int] = None, name: str = "") -> DecodeWork:
    g = generator(seed)
    ctx = torch.as_tensor(context_lens, dtype=torch.int32)
    nblk = [(c + heads.block_size - 1) // heads.block_size for c in ctx.tolist()]
    bt = block_tables_from_perm(nblk, heads.num_blocks, g, width)
    b = int(ctx.numel())
    q = normal_bf16((b, heads.num_heads, heads.head_dim), g)
    k = normal_bf16((b, heads.num_kv_heads, heads.head_dim), g)
    v = normal_bf16((b, heads.num_kv_heads, heads.head_dim), g)
    return DecodeWork(heads, ctx, bt, q, k, v, seed, name)


def empty_cache(heads: Heads, device="cpu"):
    shape = (heads.num_blocks, heads.block_size, heads.num_kv_heads, heads.head_dim)
    return (torch.zeros(shape, dtype=torch.bfloat16, device=device),
            torch.zeros(shape, dtype=torch.bfloat16, device=device))


def history_cache(heads: Heads, seed: int, device="cpu"):
    """A cache whose every slot holds seeded N(0,1) bf16 values (the history a
    decode or prefix-cache step reads)."""
    shape = (heads.num_blocks, heads.block_size, heads.num_kv_heads, heads.head_dim)
    kc = torch.empty(shape, dtype=torch.bfloat16, device=device)
    vc = torch.empty(shape, dtype=torch.bfloat16, device=device)
    fill_normal_(kc, seed * 2 + 1)
    fill_normal_(vc, seed * 2 + 2)
    return kc, vc


# ---------------------------------------------------------------------------
# The five workloads.
# ---------------------------------------------------------------------------
QWEN3_HEADS = dict(num_heads=16, num_kv_heads=8, head_dim=128, block_size=256)


def tiny(seed: int = SEED_BASE + 0):
    """4 q / 2 kv heads, head_dim 64, block_size 4, 16 blocks; prompts of 6 and
    3 tokens (seq0 owns blocks [7, 9], seq1 one other random block), then one
    decode step per sequence.  Returns (prefill, decode) sharing tables."""
    heads = Heads(4, 2, 64, 4, 16)
    g = generator(seed)
    others = [b for b in torch.randperm(16, generator=g).tolist() if b not in (7, 9)]
    bt = torch.tensor([[7, 9], [others[0], -1]], dtype=torch.int32)
    q_lens = torch.tensor([6, 3], dtype=torch.int32)
    n = 9
    pre = PrefillWork(heads, q_lens, torch.zeros(2, dtype=torch.int32), _cu(q_lens), _cu(q_lens),
                      bt.clone(),
                      normal_bf16((n, 4, 64), g), normal_bf16((n, 2, 64), g),
                      normal_bf16((n, 2, 64), g), seed, "tiny-prefill")
    dec = DecodeWork(heads, torch.tensor([7, 4], dtype=torch.int32), bt.clone(),
                     normal_bf16((2, 4, 64), g), normal_bf16((2, 2, 64), g),
                     normal_bf16((2, 2, 64), g), seed, "tiny-decode")
    return pre, dec


def qwen3_decode(seed: int = SEED_BASE + 1, batch: int = 64, num_blocks: int = 2048,
                 lo: int = 512, hi: int = 4096) -> DecodeWork:
    """Batch 64, context lengths uniform in [512, 4096], 2048-block pool."""
    g = generator(seed + 1000)
    ctx = torch.randint(lo, hi + 1, (batch,), generator=g, dtype=torch.int64)
    heads = Heads(num_blocks=num_blocks, **QWEN3_HEADS)
    return decode_work(heads, ctx, seed, name="qwen3-decode-b64")


def varlen_prefill(seed: int = SEED_BASE + 2, num_seqs: int = 8, lo: int = 128,
                   hi: int = 4096, num_blocks: int = 2048) -> PrefillWork:
    """8 prompts, lengths uniform in [128, 4096], packed, no prefix."""
    g = generator(seed + 1000)
    lens = torch.randint(lo, hi + 1, (num_seqs,), generator=g, dtype=torch.int64)
    heads = Heads(num_blocks=num_blocks, **QWEN3_HEADS)
    return prefill_work(heads, lens, None, seed, name="varlen-prefill-8x")


def prefix_prefill(seed: int = SEED_BASE + 3, num_seqs: int = 16, max_prefix_blocks: int = 12,
                   lo: int = 64, hi: int = 1024, num_blocks: int = 2048,
                   unaligned: bool = False) -> PrefillWork:
    """16 sequences, a block-aligned cached prefix of U{0..12} blocks and a new
    chunk of U[64, 1024] tokens.  ``unaligned`` adds U[1, 255] tokens to each
    prefix so the chunk starts mid-block."""
    g = generator(seed + 1000)
    bs = QWEN3_HEADS["block_size"]
    pblk = torch.randint(0, max_prefix_blocks + 1, (num_seqs,), generator=g, dtype=torch.int64)
    chunk = torch.randint(lo, hi + 1, (num_seqs,), generator=g, dtype=torch.int64)
    prefix = pblk * bs
    if unaligned:
        prefix = prefix + torch.randint(1, bs, (num_seqs,), generator=g, dtype=torch.int64)
    heads = Heads(num_blocks=num_blocks, **QWEN3_HEADS)
    return prefill_work(heads, chunk, prefix, seed,
                        name="prefix-prefill-16x" + ("-unaligned" if unaligned else ""))


def large_decode(seed: int = SEED_BASE + 4, batch: int = 256, pads: int = 32,
                 num_blocks: int = 40000, lo: int = 1024, hi: int = 32768,
                 sigma: float = 1.0) -> DecodeWork:
    """32 q / 8 kv heads (group 4); 256 rows plus 32 padding rows (context 0);
    context lengths lognormal with median 4096 and sigma 1, clipped to
    [1024, 32768]; a 40000-block pool."""
    g = generator(seed + 1000)
    z = torch.randn(batch, generator=g, dtype=torch.float64)
    ctx = torch.exp(math.log(4096.0) + sigma * z).round().clamp(lo, hi).to(torch.int64)
    ctx = torch.cat([ctx, torch.zeros(pads, dtype=torch.int64)])
    heads = Heads(32, 8, 128, 256, num_blocks)
    return decode_work(heads, ctx, seed, name="large-decode-b256p32")


def mixed_chunked(seed: int = SEED_BASE + 5, decode_rows: int = 64, chunks: int = 4,
                  chunk: int = 496, lo: int = 512, hi: int = 4096, max_prefix_chunks: int = 7,
                  num_blocks: int = 2048) -> PrefillWork:
    """A chunked-prefill step with a 2048-token budget, as one paged prefill
    call: 64 decode rows (one new token each, contexts uniform in [512, 4096]
    as in the decode workload, so a row's cached prefix is context - 1)
    followed by 4 prompt chunks of 496 tokens whose prompts already hold
    512 x U{0..7} tokens in the cache (their earlier chunks)."""
    g = generator(seed + 1000)
    ctx = torch.randint(lo, hi + 1, (decode_rows,), generator=g, dtype=torch.int64)
    pre = torch.randint(0, max_prefix_chunks + 1, (chunks,), generator=g, dtype=torch.int64) * 512
    q_lens = torch.cat([torch.ones(decode_rows, dtype=torch.int64),
                        torch.full((chunks,), chunk, dtype=torch.int64)])
    prefix = torch.cat([ctx - 1, pre])
    heads = Heads(num_blocks=num_blocks, **QWEN3_HEADS)
    return prefill_work(heads, q_lens, prefix, seed, name="mixed-chunked-2048")


CONFIGS = {
    "tiny": tiny,
    "qwen3-decode-b64": qwen3_decode,
    "varlen-prefill-8x": varlen_prefill,
    "prefix-prefill-16x": prefix_prefill,
    "large-decode-b256p32": large_decode,
    "mixed-chunked-2048": mixed_chunked,
}

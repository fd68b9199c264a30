"""Seeded synthetic workloads for paged decode attention.

This module only draws inputs: random K/V/q values, context lengths, block
tables scattered over a physical pool, slot mappings and copy-on-write lists.
It performs none of the attention arithmetic, so both the CUDA path and the
CPU oracle can take their inputs from it.

Seeds: data (q, K/V pool, new tokens) from seed 0, context lengths from seed 1,
the physical block permutation from seed 2. Values are N(0, 1) rounded to the
storage dtype. Context lengths, tables and slots are always drawn on the CPU, so
they are the same whatever device the data lands on.

The five shapes follow the workloads the pages describe:

``tiny``       4 sequences, MHA 4 heads, d 64, B 16, contexts {1, 17, 33, 100},
               fp32, a 64-block pool in random order, scale 1/8.
``opt13b``     OPT-13B layer: MHA 40 heads, d 128, fp16, B 16, 64 sequences with
               ShareGPT-like lengths (truncated lognormal, median 390, mean final
               length 493 as the CS349E Lecture 7 notes' §4.4 block-size demo
               states; 1..2048), pool of max(763, needed) blocks (763 blocks =
               the 12,207-token budget of the CMU 15-779 Lecture 16 notes, §0.4).
``llama8b``    Llama-3.1-8B layer: 32 q heads / 8 kv heads, d 128, bf16, B 16,
               256 sequences with contexts U[512, 4096], 100,000-block pool; one
               new token per sequence written by reshape_and_cache.
``shared``     64 prompts x 8 parallel samples on the Llama-3.1-8B shape: a
               2048-token prompt shared through ref-counted blocks, per-sample
               tails U[0, 512] appended after the fork.  ``cow=True`` makes the
               prompt 2048 + r (r ~ U{1..15}) tokens long so its last block is
               partial and the first append of 7 of the 8 samples copies it.
``long70b``    Llama-3.1-70B layer: 64 q heads / 8 kv heads, d 128, bf16,
               8 sequences with contexts U[32768, 131072], B 16 or 32, split into
               512-token partitions.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

from .block_manager import BlockManager

SEED_DATA, SEED_CTX, SEED_PERM = 0, 1, 2

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    S: int                      # sequences (one query token each)
    H: int                      # query heads
    G: int                      # kv heads
    d: int                      # head dim
    B: int                      # block size (tokens per physical block)
    dtype: torch.dtype
    num_blocks: int
    scale: float
    context_lens: torch.Tensor  # int32 [S], includes the new token
    block_tables: torch.Tensor  # int32 [S, max_blocks], -1 past the last used entry
    q: torch.Tensor             # [S, H, d]
    k_cache: torch.Tensor       # [num_blocks, G, B, d] (HND) or [num_blocks, B, G, d] (NHD)
    v_cache: torch.Tensor       # same layout as k_cache
    new_key: Optional[torch.Tensor] = None     # [N, G, d]
    new_value: Optional[torch.Tensor] = None   # [N, G, d]
    slot_mapping: Optional[torch.Tensor] = None  # int64 [N]
    copy_pairs: Optional[torch.Tensor] = None    # int64 [P, 2] (src, dst)
    partition_tokens: Optional[int] = None
    meta: dict = field(default_factory=dict)
    layout: str = "HND"         # pool layout of k_cache / v_cache

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context(self) -> int:
        return int(self.context_lens.max().item()) if self.S else 0

    def to(self, device) -> "Workload":
        def mv(t):
            return None if t is None else t.to(device)
        return Workload(self.name, self.S, self.H, self.G, self.d, self.B, self.dtype,
                        self.num_blocks, self.scale, mv(self.context_lens), mv(self.block_tables),
                        mv(self.q), mv(self.k_cache), mv(self.v_cache), mv(self.new_key),
                        mv(self.new_value), mv(self.slot_mapping), mv(self.copy_pairs),
                        self.partition_tokens, dict(self.meta), self.layout)


# ---------------------------------------------------------------------------
# random draws
# ---------------------------------------------------------------------------
def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn(shape, dtype, gen, device) -> torch.Tensor:
    """N(0, 1) rounded to ``dtype``."""
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def randn_big(shape, dtype, gen, device, chunk_rows=4096) -> torch.Tensor:
    """Like :func:`randn` but drawn row-chunk by row-chunk to bound temporaries."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(shape[0], -1)
    for r in range(0, shape[0], chunk_rows):
        e = min(shape[0], r + chunk_rows)
        flat[r:e] = torch.randn((e - r, flat.shape[1]), generator=gen, device=device,
                                dtype=torch.float32).to(dtype)
    return out


def lognormal_lengths(n, median, mean, lo, hi, gen) -> torch.Tensor:
    """Integer lengths from a lognormal with the given median and mean, resampled into [lo, hi]."""
    sigma = math.sqrt(2.0 * math.log(mean / median))
    mu = math.log(median)
    out = torch.empty(n, dtype=torch.int64)
    filled = 0
    while filled < n:
        draw = torch.exp(mu + sigma * torch.randn(4 * n, generator=gen, dtype=torch.float64))
        draw = torch.round(draw).to(torch.int64)
        ok = draw[(draw >= lo) & (draw <= hi)]
        take = min(n - filled, ok.numel())
        out[filled:filled + take] = ok[:take]
        filled += take
    return out


def uniform_lengths(n, lo, hi, gen) -> torch.Tensor:
    """Integers uniform on [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=gen, dtype=torch.int64)


# ---------------------------------------------------------------------------
# assembling a batch from a block manager
# ---------------------------------------------------------------------------
def _tables(bm: BlockManager, seq_ids, B) -> tuple:
    ctx = [bm.context_len(s) for s in seq_ids]
    width = max([1] + [-(-c // B) for c in ctx])
    bt = torch.full((len(seq_ids), width), -1, dtype=torch.int32)
    for i, s in enumerate(seq_ids):
        ids = bm.block_table(s)
        if ids:
            bt[i, :len(ids)] = torch.tensor(ids, dtype=torch.int32)
    return torch.tensor(ctx, dtype=torch.int32), bt


def batch_with_new_tokens(name, S, H, G, d, B, dtype, ctx, num_blocks, device,
                          new_token=True, scale=None, partition_tokens=None, meta=None,
                          pool_fill=None, rotate=0) -> Workload:
    """Independent sequences of lengths ``ctx`` scattered over a shuffled pool.

    With ``new_token`` the last position of every sequence is left for
    reshape_and_cache (its K/V are in ``new_key`` / ``new_value`` and its slot
    in ``slot_mapping``); the pool holds the earlier positions. ``rotate``
    starts handing out blocks ``rotate`` places into the shuffled free list, so
    two batches drawn with rotations far enough apart use disjoint blocks.
    """
    ctx = [int(c) for c in ctx]
    perm = torch.randperm(num_blocks, generator=_gen(SEED_PERM)).tolist()
    if rotate:
        perm = perm[rotate:] + perm[:rotate]
    bm = BlockManager(num_blocks, B, free_order=perm)
    slots = []
    for s, c in enumerate(ctx):
        if new_token and c > 0:
            bm.add_sequence(s, c - 1)
            slot, pair = bm.append_slot(s)
            assert pair is None
            slots.append(slot)
        else:
            bm.add_sequence(s, c)
    ctx_t, bt = _tables(bm, list(range(S)), B)

    g = _gen(SEED_DATA, device)
    kshape = (num_blocks, G, B, d)
    if pool_fill is None:
        k_cache = randn_big(kshape, dtype, g, device)
        v_cache = randn_big(kshape, dtype, g, device)
    else:
        k_cache = torch.full(kshape, pool_fill, dtype=dtype, device=device)
        v_cache = torch.full(kshape, pool_fill, dtype=dtype, device=device)
    q = randn((S, H, d), dtype, g, device)
    wl = Workload(name, S, H, G, d, B, dtype, num_blocks,
                  (1.0 / math.sqrt(d)) if scale is None else scale,
                  ctx_t.to(device), bt.to(device), q, k_cache, v_cache,
                  partition_tokens=partition_tokens, meta=dict(meta or {}))
    if slots:
        N = len(slots)
        wl.new_key = randn((N, G, d), dtype, g, device)
        wl.new_value = randn((N, G, d), dtype, g, device)
        wl.slot_mapping = torch.tensor(slots, dtype=torch.int64, device=device)
    wl.meta.setdefault("pool_blocks_used", num_blocks - bm.num_free())
    return wl


# ---------------------------------------------------------------------------
# the five shapes
# ---------------------------------------------------------------------------
def tiny(device="cpu", new_token=False) -> Workload:
    return batch_with_new_tokens("tiny", 4, 4, 4, 64, 16, torch.float32, [1, 17, 33, 100], 64,
                                 device, new_token=new_token, scale=1.0 / 8.0)


def opt13b(device="cpu", S=64, new_token=True) -> Workload:
    ctx = lognormal_lengths(S, 390.0, 493.0, 1, 2048, _gen(SEED_CTX)).tolist()
    need = sum(-(-c // 16) for c in ctx)
    nb = max(763, need)
    return batch_with_new_tokens("opt13b", S, 40, 40, 128, 16, torch.float16, ctx, nb, device,
                                 new_token=new_token,
                                 meta={"pool_reading": "max(763, blocks needed)"})


def llama8b(device="cpu", S=256, num_blocks=100_000, new_token=True, rotate=0) -> Workload:
    ctx = uniform_lengths(S, 512, 4096, _gen(SEED_CTX)).tolist()
    return batch_with_new_tokens("llama8b", S, 32, 8, 128, 16, torch.bfloat16, ctx, num_blocks,
                                 device, new_token=new_token, rotate=rotate)


def llama70b_short(device="cpu", S=256, num_blocks=100_000, new_token=True) -> Workload:
    """Plain decode at a GQA group of 8: the Llama-3.1-70B head layout (64 q / 8 kv
    heads, d 128, bf16, block 16) on the Llama-3.1-8B batch's lengths
    (U[512, 4096], 256 sequences) over a 100k-block shuffled pool. The KV bytes
    per token equal the 8B batch's (the same 8 kv heads); twice the query rows."""
    ctx = uniform_lengths(S, 512, 4096, _gen(SEED_CTX)).tolist()
    return batch_with_new_tokens("llama70b_short", S, 64, 8, 128, 16, torch.bfloat16, ctx, num_blocks,
                                 device, new_token=new_token)


def gemma_d256(device="cpu", S=256, num_blocks=50_000, new_token=True) -> Workload:
    """head_dim 256 with a group of 2 (16 q / 8 kv heads, the Gemma-2-9B layer
    shape), bf16, block 16: the Llama-3.1-8B batch's lengths (U[512, 4096]) and a
    shuffled pool of the same byte size (a block holds 2x the bytes)."""
    ctx = uniform_lengths(S, 512, 4096, _gen(SEED_CTX)).tolist()
    return batch_with_new_tokens("gemma_d256", S, 16, 8, 256, 16, torch.bfloat16, ctx, num_blocks,
                                 device, new_token=new_token)


def long70b(device="cpu", S=8, B=16, lo=32768, hi=131072, partition_tokens=512,
            new_token=True) -> Workload:
    ctx = uniform_lengths(S, lo, hi, _gen(SEED_CTX)).tolist()
    need = sum(-(-c // B) for c in ctx)
    nb = need + need // 8
    return batch_with_new_tokens(f"long70b_B{B}", S, 64, 8, 128, B, torch.bfloat16, ctx, nb,
                                 device, new_token=new_token, partition_tokens=partition_tokens)


def shared_prefix(device="cpu", prompts=64, samples=8, prefix=2048, tail_lo=0, tail_hi=512,
                  cow=False, num_blocks=None, H=32, G=8, d=128, B=16, dtype=torch.bfloat16) -> Workload:
    """Parallel sampling: ``prompts`` prompts forked into ``samples`` samples each.

    The prompt blocks are ref-counted and shared by all samples of the prompt.
    Each sample then appends ``tail`` tokens plus this step's token; those
    appends go through the block manager, which emits the copy-on-write pairs.
    The step is: copy_blocks(pairs), reshape_and_cache(all appended tokens),
    decode.  Before the step the pool holds the prompt tokens (and garbage
    elsewhere). The default head shape is the Llama-3.1-8B layer's.
    """
    gctx = _gen(SEED_CTX)
    r = (uniform_lengths(prompts, 1, B - 1, gctx) if cow
         else torch.zeros(prompts, dtype=torch.int64)).tolist()
    tails = uniform_lengths(prompts * samples, tail_lo, tail_hi, gctx).tolist()
    need = sum(-(-(prefix + r[p]) // B) for p in range(prompts))
    need += sum(-(-(tails[i] + 1 + B) // B) for i in range(prompts * samples))
    nb = num_blocks or (need + need // 8)
    perm = torch.randperm(nb, generator=_gen(SEED_PERM)).tolist()
    bm = BlockManager(nb, B, free_order=perm)
    seq_ids = []
    for p in range(prompts):
        base = p * samples
        bm.add_sequence(base, prefix + r[p])
        for j in range(1, samples):
            bm.fork(base, base + j)
        seq_ids.extend(range(base, base + samples))
    slots, pairs = [], []
    for s in seq_ids:
        for _ in range(tails[s] + 1):
            slot, pair = bm.append_slot(s)
            slots.append(slot)
            if pair is not None:
                pairs.append(pair)
    ctx_t, bt = _tables(bm, seq_ids, B)
    g = _gen(SEED_DATA, device)
    kshape = (nb, G, B, d)
    k_cache = randn_big(kshape, dtype, g, device)
    v_cache = randn_big(kshape, dtype, g, device)
    S = len(seq_ids)
    q = randn((S, H, d), dtype, g, device)
    N = len(slots)
    wl = Workload("shared_cow" if cow else "shared", S, H, G, d, B, dtype, nb,
                  1.0 / math.sqrt(d), ctx_t.to(device), bt.to(device), q, k_cache, v_cache,
                  new_key=randn((N, G, d), dtype, g, device),
                  new_value=randn((N, G, d), dtype, g, device),
                  slot_mapping=torch.tensor(slots, dtype=torch.int64, device=device),
                  copy_pairs=torch.tensor(pairs, dtype=torch.int64, device=device).view(-1, 2),
                  meta={"prompts": prompts, "samples": samples, "prefix": prefix,
                        "prefix_extra": r, "cow_copies": len(pairs),
                        "unique_tokens": sum(prefix + r[p] for p in range(prompts)) + N,
                        # groups for the shared-prefix decode: one per prompt, its samples in order
                        "group_starts": [p * samples for p in range(prompts + 1)],
                        "prefix_lens": [prefix + r[p] for p in range(prompts)]})
    return wl


def to_fp8(wl: Workload, k_scale=None, v_scale=None) -> Workload:
    """The same batch with an E4M3 KV pool: codes of clamp(x / scale, +-448).

    The scale defaults to max|x| / 448 over the pool (one fp32 per tensor). q
    and the new tokens keep their type (the fp8 cache write quantises them).
    """
    def codes(t, sc):
        out = torch.empty(t.shape, dtype=torch.uint8, device=t.device)
        flat, of = t.view(t.shape[0], -1), out.view(t.shape[0], -1)
        for r in range(0, t.shape[0], 4096):
            x = (flat[r:r + 4096].float() / sc).clamp_(-448.0, 448.0)
            of[r:r + 4096] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        return out
    ks = float(k_scale if k_scale is not None else wl.k_cache.abs().max().float().item() / 448.0)
    vs = float(v_scale if v_scale is not None else wl.v_cache.abs().max().float().item() / 448.0)
    meta = dict(wl.meta)
    meta.update(k_scale=ks, v_scale=vs, kv_dtype="fp8_e4m3")
    return Workload(wl.name + "_fp8", wl.S, wl.H, wl.G, wl.d, wl.B, wl.dtype, wl.num_blocks, wl.scale,
                    wl.context_lens, wl.block_tables, wl.q, codes(wl.k_cache, ks), codes(wl.v_cache, vs),
                    wl.new_key, wl.new_value, wl.slot_mapping, wl.copy_pairs, wl.partition_tokens, meta,
                    wl.layout)


def to_nhd(wl: Workload) -> Workload:
    """The same batch with its pools stored NHD, [num_blocks, B, G, d]: the same
    values, each block's token and head axes exchanged."""
    if wl.layout != "HND":
        raise ValueError("to_nhd expects an HND workload")

    def nhd(t):
        out = torch.empty((t.shape[0], t.shape[2], t.shape[1], t.shape[3]), dtype=t.dtype, device=t.device)
        for r in range(0, t.shape[0], 8192):
            out[r:r + 8192].copy_(t[r:r + 8192].transpose(1, 2))
        return out
    return Workload(wl.name + "_nhd", wl.S, wl.H, wl.G, wl.d, wl.B, wl.dtype, wl.num_blocks, wl.scale,
                    wl.context_lens, wl.block_tables, wl.q, nhd(wl.k_cache), nhd(wl.v_cache),
                    wl.new_key, wl.new_value, wl.slot_mapping, wl.copy_pairs, wl.partition_tokens,
                    dict(wl.meta), "NHD")


def by_name(name: str, device="cpu", **kw) -> Workload:
    table = {"tiny": tiny, "opt13b": opt13b, "llama8b": llama8b, "long70b": long70b, "gemma_d256": gemma_d256,
             "llama70b_short": llama70b_short,
             "shared": shared_prefix,
             "shared_cow": lambda device="cpu", **k: shared_prefix(device, cow=True, **k)}
    return table[name](device=device, **kw)

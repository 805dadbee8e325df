"""Seeded synthetic decode workloads shaped like the pages' examples.

This module only builds inputs: shapes, random bf16 values, which physical
block or request row each sequence owns, and where each new token goes.  It
holds none of the decode arithmetic (no gather-by-table for attention, no
softmax, no append or copy kernel); both the CUDA path and the CPU oracle take
what it produces as their input.

Shapes and workloads (page title, passage):
  * "Insights into LLM Serving Systems: KV-Cache Memory Allocation Patterns",
    section 4: Yi-6B, Llama-3-8B and Yi-34B decode with 1K-token contexts and
    batch 1..320; Observation-2 gives 64 KB, 128 KB and 240 KB of KV per
    token over all layers.
  * "Running Out of Cache": 16-token blocks, block tables, a new block only
    when the last is full; workshop lengths prompt ~ Exp(mean 1024), output
    ~ Exp(mean 256), at most 8192 tokens; shared blocks with copy on write.
  * "Leveraging Low-Level CUDA APIs for vAttention's Dynamic Memory",
    section 5.2.3: request sub-tensor at offset reqId x S.

Value recipe: Q, K, V ~ N(0, 1) rounded to bf16; scale = 1/sqrt(head_dim).
Physical blocks are handed out from a seeded random permutation of the pool,
sequence 0 first.  Seeds are 245 + workload index (tiny 245, Yi-6B 246,
Llama sweep 247, ragged 248, Yi-34B sharing 249); layer l of a workload draws
its values from a generator seeded with (seed * 1000 + l).
"""
from dataclasses import dataclass, field
import math
from typing import List, Optional

import numpy as np
import torch

TOKENS_PER_TILE = 16  # nothing here depends on it; kept for readers of tests


@dataclass(frozen=True)
class ModelShape:
    """KV geometry of one model: layers, query heads, KV heads, head_dim."""
    name: str
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int = 128

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def kv_bytes_per_token(self, elem_bytes: int = 2) -> int:
        """K and V of one token over all layers (the pages' per-token size)."""
        return (self.num_layers * self.num_kv_heads * self.head_dim * 2
                * elem_bytes)


TINY = ModelShape("tiny", 1, 8, 2)
YI_6B = ModelShape("Yi-6B", 32, 32, 4)
LLAMA3_8B = ModelShape("Llama-3-8B", 32, 32, 8)
YI_34B = ModelShape("Yi-34B", 60, 56, 8)
SHAPES = {s.name: s for s in (TINY, YI_6B, LLAMA3_8B, YI_34B)}

SEED_TINY, SEED_YI6B, SEED_LLAMA, SEED_RAGGED, SEED_YI34B = 245, 246, 247, 248, 249
LLAMA_SWEEP_BATCHES = (1, 8, 32, 64, 128, 256, 320)
RAGGED_BLOCK_SIZES = (16, 32, 64, 128)


def default_scale(shape: ModelShape) -> float:
    return 1.0 / math.sqrt(shape.head_dim)


@dataclass
class PagedBatch:
    """One decode batch laid out in a paged block pool.

    ctx[i] is the number of positions sequence i attends over after this
    step's token has been appended (ctx = ctx_pre + 1).  Each sequence owns
    ceil(ctx / bs) blocks; the new token of sequence i goes to slot
    slot_mapping[i] (block * bs + offset).  block_tables entries past a
    sequence's last block are filler (valid ids that must be ignored)."""
    shape: ModelShape
    seed: int
    block_size: int
    num_blocks: int
    ctx_pre: np.ndarray          # int32 [B]
    ctx: np.ndarray              # int32 [B]
    block_tables: np.ndarray     # int32 [B, max_blocks]
    slot_mapping: np.ndarray     # int64 [B]
    req_ids: np.ndarray          # int32 [B], the request row for contig use
    max_reqs: int = 0

    @property
    def B(self) -> int:
        return int(self.ctx.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context(self) -> int:
        return int(self.ctx.max()) if self.B else 0

    def kv_bytes(self) -> int:
        """Bytes of K and V the batch attends over in one layer."""
        s = self.shape
        return int(self.ctx.astype(np.int64).sum()) * s.num_kv_heads * s.head_dim * 4


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def assign_blocks(ctx: np.ndarray, block_size: int, seed: int,
                  spare_blocks: int = 0, filler: Optional[int] = None):
    """Hand each sequence ceil(ctx/bs) physical blocks from a random
    permutation of the pool (sequence 0 first).  Returns
    (block_tables [B, max_blocks] int32, num_blocks)."""
    ctx = np.asarray(ctx, dtype=np.int64)
    need = (ctx + block_size - 1) // block_size
    need = np.maximum(need, 0)
    total = int(need.sum())
    num_blocks = max(total + spare_blocks, 1)
    perm = torch.randperm(num_blocks, generator=_gen(seed)).numpy().astype(np.int32)
    max_blocks = max(int(need.max()) if len(need) else 1, 1)
    rng = np.random.default_rng(seed)
    tables = rng.integers(0, num_blocks, size=(len(ctx), max_blocks),
                          dtype=np.int64).astype(np.int32)
    if filler is not None:
        tables[:] = filler
    pos = 0
    for i, n in enumerate(need):
        tables[i, :n] = perm[pos:pos + n]
        pos += int(n)
    return tables, num_blocks


def make_paged_batch(shape: ModelShape, ctx, block_size: int, seed: int,
                     spare_blocks: int = 0) -> PagedBatch:
    """A decode step: sequence i already holds ctx[i]-1 tokens and appends
    one, so it attends over ctx[i] positions."""
    ctx = np.asarray(ctx, dtype=np.int32)
    ctx_pre = ctx - 1
    tables, nb = assign_blocks(ctx, block_size, seed, spare_blocks)
    slots = np.empty(len(ctx), dtype=np.int64)
    for i, p in enumerate(ctx_pre):
        # position p of sequence i: logical block p // bs, offset p % bs
        slots[i] = int(tables[i, p // block_size]) * block_size + int(p % block_size)
    return PagedBatch(shape=shape, seed=seed, block_size=block_size,
                      num_blocks=nb, ctx_pre=ctx_pre, ctx=ctx,
                      block_tables=tables, slot_mapping=slots,
                      req_ids=np.arange(len(ctx), dtype=np.int32),
                      max_reqs=len(ctx))


def bf16_randn(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """N(0,1) values rounded to bf16 (drawn on the CPU generator, so a seed
    gives the same values on every machine)."""
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16).to(device)


def bf16_randn_fast(shape, seed: int, device) -> torch.Tensor:
    """N(0,1) bf16 drawn with the generator of `device` (used for large
    caches where CPU generation would dominate; seeded, device-specific)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32,
                       device=device).to(torch.bfloat16)


@dataclass
class LayerInputs:
    q: torch.Tensor        # [B, Hq, D] bf16
    k_new: torch.Tensor    # [B, Hkv, D] bf16
    v_new: torch.Tensor    # [B, Hkv, D] bf16
    k_cache: torch.Tensor  # [NB, Hkv, bs, D] bf16
    v_cache: torch.Tensor  # [NB, Hkv, bs, D] bf16


def layer_inputs(batch: PagedBatch, layer: int, device="cpu",
                 fast_cache: bool = False) -> LayerInputs:
    """Random values for one layer of a batch.  The cache pool is filled
    everywhere, including the slot the new token will overwrite."""
    s = batch.shape
    seed = batch.seed * 1000 + layer
    g = _gen(seed)
    q = bf16_randn((batch.B, s.num_q_heads, s.head_dim), g, device)
    k_new = bf16_randn((batch.B, s.num_kv_heads, s.head_dim), g, device)
    v_new = bf16_randn((batch.B, s.num_kv_heads, s.head_dim), g, device)
    cshape = (batch.num_blocks, s.num_kv_heads, batch.block_size, s.head_dim)
    if fast_cache:
        k_cache = bf16_randn_fast(cshape, seed * 2 + 1, device)
        v_cache = bf16_randn_fast(cshape, seed * 2 + 2, device)
    else:
        k_cache = bf16_randn(cshape, g, device)
        v_cache = bf16_randn(cshape, g, device)
    return LayerInputs(q, k_new, v_new, k_cache, v_cache)


def paged_to_contig(cache: torch.Tensor, batch: PagedBatch, S: int,
                    max_reqs: Optional[int] = None) -> torch.Tensor:
    """Lay the same logical rows out contiguously: request i's rows go to
    buffer row req_ids[i] (offset reqId x S).  Built with torch indexing for
    input construction; positions past ctx hold zeros."""
    s = batch.shape
    nb, hkv, bs, d = cache.shape
    max_reqs = max_reqs or batch.max_reqs
    buf = torch.zeros((max_reqs, hkv, S, d), dtype=cache.dtype, device=cache.device)
    for i in range(batch.B):
        c = int(batch.ctx[i])
        if c <= 0:
            continue
        n = (c + bs - 1) // bs
        ids = torch.as_tensor(batch.block_tables[i, :n].astype(np.int64),
                              device=cache.device)
        rows = cache[ids].permute(1, 0, 2, 3).reshape(hkv, n * bs, d)[:, :c]
        buf[int(batch.req_ids[i]), :, :c] = rows
    return buf


# --------------------------------------------------------------------------
# The five workloads
# --------------------------------------------------------------------------

def tiny_batch(after_append: bool = True) -> PagedBatch:
    """Four sequences with contexts {1,17,33,100}, 8 query / 2 KV heads,
    block_size 16, 64 physical blocks.  after_append=True gives the step that
    appends one token to each (contexts {2,18,34,101})."""
    base = np.array([1, 17, 33, 100], dtype=np.int32)
    ctx = base + 1
    tables, nb = assign_blocks(ctx, 16, SEED_TINY, spare_blocks=64 - 13)
    assert nb == 64
    b = PagedBatch(shape=TINY, seed=SEED_TINY, block_size=16, num_blocks=nb,
                   ctx_pre=base.copy(), ctx=ctx, block_tables=tables,
                   slot_mapping=np.array([int(tables[i, p // 16]) * 16 + int(p % 16)
                                          for i, p in enumerate(base)], dtype=np.int64),
                   req_ids=np.arange(4, dtype=np.int32), max_reqs=4)
    if not after_append:
        b.ctx = base.copy()
    return b


def uniform_batch(shape: ModelShape, B: int, ctx: int = 1024, block_size: int = 16,
                  seed: int = SEED_LLAMA) -> PagedBatch:
    """B sequences, every one attending over exactly `ctx` positions (ctx-1
    already cached plus the appended token)."""
    return make_paged_batch(shape, np.full(B, ctx, dtype=np.int32), block_size, seed)


def ragged_lengths(B: int = 256, seed: int = SEED_RAGGED, max_len: int = 8192,
                   prompt_mean: float = 1024.0, output_mean: float = 256.0):
    """Context lengths of a serving batch caught mid-generation: prompt
    P = max(1, round(Exp(1024))), output O = round(Exp(256)), generated so far
    g ~ U{0..O}; the step attends over min(P + g + 1, max_len) positions."""
    g = _gen(seed)
    u1 = torch.rand(B, generator=g, dtype=torch.float64).numpy()
    u2 = torch.rand(B, generator=g, dtype=torch.float64).numpy()
    u3 = torch.rand(B, generator=g, dtype=torch.float64).numpy()
    P = np.maximum(1, np.rint(-prompt_mean * np.log1p(-u1))).astype(np.int64)
    O = np.rint(-output_mean * np.log1p(-u2)).astype(np.int64)
    gen_so_far = np.floor(u3 * (O + 1)).astype(np.int64)
    return np.minimum(P + gen_so_far + 1, max_len).astype(np.int32)


def ragged_batch(block_size: int = 16, B: int = 256) -> PagedBatch:
    return make_paged_batch(LLAMA3_8B, ragged_lengths(B), block_size, SEED_RAGGED)


@dataclass
class SharingScenario:
    """Yi-34B-shaped parallel sampling: each prompt is decoded n ways and the
    n branches share the prompt's physical blocks until one writes into a
    shared block, which it then copies (copy on write)."""
    shape: ModelShape
    block_size: int
    num_blocks: int
    prompt_lens: np.ndarray          # [P]
    n: int
    tables_shared: np.ndarray        # [B, max_blocks] before any copy
    cow_pairs: np.ndarray            # [n_copies, 2] int64 (src, dst)
    free_order: np.ndarray           # [num_blocks] int32: the order blocks are handed out
    tables: np.ndarray               # [B, max_blocks] after the copies
    steps: List[PagedBatch] = field(default_factory=list)  # one per decode step


def sharing_scenario(num_prompts: int = 32, n: int = 4, decode_steps: int = 64,
                     block_size: int = 16, shape: ModelShape = YI_34B,
                     min_len: int = 1024, max_len: int = 8192,
                     seed: int = SEED_YI34B) -> SharingScenario:
    """Block manager for prompts shared by reference count.

    Branch b of prompt p is sequence p*n + b.  All n branches point at the
    prompt's blocks (refcount n).  On the first decode step a branch that
    writes into a shared, partially filled last block while its refcount is
    above one takes a fresh block, copies the shared one into it and drops
    its reference; the last branch (refcount 1) writes in place.  If the
    prompt fills its last block exactly, every branch takes a fresh block and
    nothing is copied.  Later tokens go to private blocks, a fresh one each
    time the last fills."""
    g = _gen(seed)
    prompt_lens = torch.randint(min_len, max_len + 1, (num_prompts,),
                                generator=g).numpy().astype(np.int64)
    bs = block_size
    B = num_prompts * n
    final_ctx = prompt_lens + decode_steps
    # blocks: shared prompt blocks + per-branch private blocks (worst case)
    prompt_blocks = (prompt_lens + bs - 1) // bs
    private_blocks = (decode_steps + bs - 1) // bs + 1
    total = int(prompt_blocks.sum()) + B * int(private_blocks)
    perm = torch.randperm(total, generator=g).numpy().astype(np.int32)
    free = list(perm[::-1])  # pop() hands out perm[0], perm[1], ...

    max_blocks = int(((final_ctx + bs - 1) // bs).max())
    tables = np.zeros((B, max_blocks), dtype=np.int32)
    nblk = np.zeros(B, dtype=np.int64)
    refcount = {}
    for p in range(num_prompts):
        ids = [free.pop() for _ in range(int(prompt_blocks[p]))]
        for blk in ids:
            refcount[int(blk)] = n
        for b in range(n):
            tables[p * n + b, :len(ids)] = ids
            nblk[p * n + b] = len(ids)
    tables_shared = tables.copy()
    ctx_pre = np.repeat(prompt_lens, n).astype(np.int64)

    cow_pairs = []
    steps = []
    for step in range(decode_steps):
        slots = np.empty(B, dtype=np.int64)
        for i in range(B):
            pos = int(ctx_pre[i])
            lb, off = pos // bs, pos % bs
            if lb >= nblk[i]:
                # last block full: take a fresh private block
                blk = int(free.pop())
                refcount[blk] = 1
                tables[i, lb] = blk
                nblk[i] += 1
            else:
                blk = int(tables[i, lb])
                if refcount[blk] > 1:
                    new = int(free.pop())
                    refcount[new] = 1
                    refcount[blk] -= 1
                    cow_pairs.append((blk, new))
                    tables[i, lb] = new
                    blk = new
            slots[i] = blk * bs + off
        ctx = (ctx_pre + 1).astype(np.int32)
        steps.append(PagedBatch(shape=shape, seed=seed, block_size=bs,
                                num_blocks=total, ctx_pre=ctx_pre.astype(np.int32),
                                ctx=ctx, block_tables=tables.copy(),
                                slot_mapping=slots,
                                req_ids=np.arange(B, dtype=np.int32), max_reqs=B))
        ctx_pre = ctx_pre + 1
    # copies happen only on the first step (the first write to a shared block)
    pairs = np.array(cow_pairs, dtype=np.int64).reshape(-1, 2)
    return SharingScenario(shape=shape, block_size=bs, num_blocks=total,
                           prompt_lens=prompt_lens, n=n,
                           tables_shared=tables_shared, cow_pairs=pairs, free_order=perm,
                           tables=steps[0].block_tables if steps else tables,
                           steps=steps)


def shared_prefix_blocks(block_tables: np.ndarray, ctx: np.ndarray, block_size: int,
                         group_start: np.ndarray) -> np.ndarray:
    """For groups of consecutive sequences (group_start [G+1]), the number of
    leading block-table entries all members have in common and whose
    positions every member's context covers (0 for a singleton)."""
    out = []
    for g in range(len(group_start) - 1):
        rows = block_tables[group_start[g]:group_start[g + 1]]
        if len(rows) < 2:
            out.append(0)
            continue
        n = int(ctx[group_start[g]:group_start[g + 1]].min() // block_size)
        k = 0
        while k < n and np.all(rows[:, k] == rows[0, k]):
            k += 1
        out.append(k)
    return np.asarray(out, np.int32)


def to_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its uint16 bit patterns as a host numpy array."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def from_u16(a: np.ndarray, device="cpu") -> torch.Tensor:
    """uint16 bit patterns -> bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)

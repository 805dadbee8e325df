"""Helpers shared by the GPU parity tests: run a workload layer through the
CUDA path and through the CPU oracle from the same seeded inputs, and compare.

The oracle only ever sees inputs from the generators (copied to the host);
the CUDA path's outputs are only compared, never fed back."""
import numpy as np
import torch

import oracle
import paged_kv_cache_245_gb300 as pkv
import workloads as W

ATOL = 1e-2   # |err| <= ATOL + RTOL * |ref| per element, against fp64
RTOL = 1e-2


def assert_attention_close(got, ref, what=""):
    """got: bf16 tensor [B, Hq, D] from the GPU; ref: fp64 [B, Hq, D]."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "%s: non-finite output" % what
    excess = np.abs(g - ref) - (ATOL + RTOL * np.abs(ref))
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, ("%s: element %s got %.6g want %.6g (|err| %.3g)"
                               % (what, worst, g[worst], ref[worst], abs(g[worst] - ref[worst])))
    return float(np.abs(g - ref).max())


class DeviceLayer:
    """One layer of a paged batch resident on the GPU, with a host mirror of
    the caches maintained by the oracle."""

    def __init__(self, batch, layer, dev, fast_cache=False):
        self.b = batch
        li = W.layer_inputs(batch, layer, device="cpu" if not fast_cache else dev,
                            fast_cache=fast_cache)
        self.q = li.q.to(dev)
        self.k_new = li.k_new.to(dev)
        self.v_new = li.v_new.to(dev)
        self.k_cache = li.k_cache.to(dev)
        self.v_cache = li.v_cache.to(dev)
        # host copies for the oracle (taken before any kernel writes)
        self.h_q = W.to_u16(li.q)
        self.h_k_new = W.to_u16(li.k_new)
        self.h_v_new = W.to_u16(li.v_new)
        self.h_k = W.to_u16(li.k_cache).copy()
        self.h_v = W.to_u16(li.v_cache).copy()
        self.dev = dev
        self.tables = torch.as_tensor(batch.block_tables, device=dev)
        self.ctx = torch.as_tensor(batch.ctx, device=dev)
        self.slots = torch.as_tensor(batch.slot_mapping, device=dev)
        self.scale = W.default_scale(batch.shape)

    def set_step(self, batch):
        self.b = batch
        self.tables = torch.as_tensor(batch.block_tables, device=self.dev)
        self.ctx = torch.as_tensor(batch.ctx, device=self.dev)
        self.slots = torch.as_tensor(batch.slot_mapping, device=self.dev)

    def gpu_append(self, k_new=None, v_new=None):
        pkv.kv_append(self.slots, self.k_new if k_new is None else k_new,
                      self.v_new if v_new is None else v_new, self.k_cache, self.v_cache)

    def oracle_append(self, k_new=None, v_new=None):
        oracle.kv_append(self.b.slot_mapping, self.h_k_new if k_new is None else k_new,
                         self.h_v_new if v_new is None else v_new, self.h_k, self.h_v)

    def gpu_attend(self, q=None):
        return pkv.paged_decode_attention(self.q if q is None else q, self.k_cache, self.v_cache,
                                          self.tables, self.ctx, self.b.max_context, self.scale)

    def oracle_attend(self, q=None, nthreads=0):
        return oracle.paged_decode(self.h_q if q is None else q, self.h_k, self.h_v,
                                   self.b.block_tables, self.b.ctx, self.scale, nthreads)

    def assert_caches_equal(self):
        assert np.array_equal(W.to_u16(self.k_cache), self.h_k), "K cache differs"
        assert np.array_equal(W.to_u16(self.v_cache), self.h_v), "V cache differs"


def shared_groups_batch(hq, hkv, sizes, max_prompt_blocks, seed, own_max=70,
                        singleton_blocks=10):
    """Groups of consecutive sequences (sizes[g] members each) whose block
    tables begin with the same whole prompt blocks, then each member's own
    blocks (0 .. own_max - 1 positions); some members stop exactly at the
    shared blocks, singletons share nothing (at most singleton_blocks blocks
    of their own).  Block size 16, physical blocks from a seeded permutation.
    Returns (batch, group starts)."""
    rng = np.random.default_rng(seed)
    bs = 16
    shape = W.ModelShape("s%d_%d" % (hq, hkv), 1, hq, hkv)
    starts = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    B = int(starts[-1])
    prompt = rng.integers(1, max_prompt_blocks, size=len(sizes)) * bs   # whole shared blocks
    # a singleton shares nothing: all its positions are its own (keep them
    # within the in-merge bound)
    prompt[np.asarray(sizes) == 1] = np.minimum(prompt[np.asarray(sizes) == 1],
                                                singleton_blocks * bs)
    own_pos = [rng.integers(0, own_max, size=s) for s in sizes]
    own_pos[int(np.argmax(np.asarray(sizes) > 1))][0] = 0  # a member with no own positions
    ctx = np.concatenate([p + o for p, o in zip(prompt, own_pos)]).astype(np.int32)
    ctx = np.maximum(ctx, 1)
    max_blocks = int((ctx.max() + bs - 1) // bs)
    nb = int(sum((c + bs - 1) // bs for c in ctx)) + 8
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((B, max_blocks), np.int32)
    used = 0
    for g, s in enumerate(sizes):
        pb = int(prompt[g] // bs)
        pblocks = perm[used:used + pb]
        used += pb
        for k in range(s):
            i = int(starts[g]) + k
            tables[i, :pb] = pblocks
            rest = int((ctx[i] + bs - 1) // bs) - pb
            tables[i, pb:pb + rest] = perm[used:used + rest]
            used += rest
    b = W.PagedBatch(shape=shape, seed=1, block_size=bs, num_blocks=nb, ctx_pre=ctx - 1, ctx=ctx,
                     block_tables=tables, slot_mapping=np.full(B, -1, np.int64),
                     req_ids=np.arange(B, dtype=np.int32), max_reqs=B)
    return b, starts

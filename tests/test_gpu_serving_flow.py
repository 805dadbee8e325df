"""The calls working together the way a serving loop uses them, checked at
every stage against the oracle run on a host mirror of the cache:

  host block manager: prompts get blocks, forks share them, each decode step
  yields slots and copy-on-write pairs;
  kv_append of the prompts' rows, then causal prefill over the paged cache;
  decode steps: block_copy of the copy-on-write pairs, kv_append of the new
  rows, decode attention (the regular call and the shared-prefix call);
  a retired sequence's blocks reused by a new prompt;
  pre-emption when the pool runs out ("Running Out of Cache", closing
  paragraph): victims planned by the manager, swapped to a page-locked host
  pool with block_swap or dropped for recompute, then brought back (swap in,
  or kv_append of their rows again) once sequences retire.

The device cache must stay bit-identical to the mirror the oracle updates,
and every attention output must match the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_245_gb300 as pkv
import workloads as W
from parity import assert_attention_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
HQ, HKV, D, BS, NB, MAXB = 32, 8, 128, 16, 160, 40
SCALE = D ** -0.5


class Flow:
    def __init__(self, seed, nb=NB, nh=0):
        self.g = torch.Generator().manual_seed(seed)
        order = torch.randperm(nb, generator=self.g).numpy().astype(np.int32)
        self.bm = pkv.BlockManager(nb, BS, free_order=order)
        self.k_dev = torch.zeros((nb, HKV, BS, D), dtype=torch.bfloat16, device=DEV)
        self.v_dev = torch.zeros_like(self.k_dev)
        self.k_host = np.zeros((nb, HKV, BS, D), dtype=np.uint16)
        self.v_host = np.zeros_like(self.k_host)
        # the swap space: page-locked host pool and the oracle's mirror of it
        self.bm.set_swap_space(nh)
        self.k_swap = torch.zeros((max(nh, 1), HKV, BS, D), dtype=torch.bfloat16).pin_memory()
        self.v_swap = torch.zeros_like(self.k_swap).pin_memory()
        self.k_swap_m = np.zeros((max(nh, 1), HKV, BS, D), dtype=np.uint16)
        self.v_swap_m = np.zeros_like(self.k_swap_m)
        self.saved = {}           # sequences evicted for recompute: their rows

    def rand(self, *shape):
        return torch.randn(shape, generator=self.g).to(torch.bfloat16)

    def tables(self, seqs):
        return self.bm.export(seqs, MAXB)

    def append(self, slots, k, v):
        pkv.kv_append(torch.as_tensor(slots, device=DEV), k.to(DEV), v.to(DEV),
                      self.k_dev, self.v_dev)
        oracle.kv_append(slots, W.to_u16(k), W.to_u16(v), self.k_host, self.v_host)

    def copy(self, pairs):
        if len(pairs):
            pkv.block_copy(torch.as_tensor(pairs, device=DEV), [self.k_dev], [self.v_dev])
            oracle.block_copy(pairs, [self.k_host], [self.v_host])

    def assert_cache_mirrors(self, what):
        torch.cuda.synchronize()
        assert np.array_equal(W.to_u16(self.k_dev.cpu()), self.k_host), what + ": K cache"
        assert np.array_equal(W.to_u16(self.v_dev.cpu()), self.v_host), what + ": V cache"

    def prefill(self, seqs, lengths, what):
        """Append the prompts' rows at the slots their block tables give, then
        attend them causally; checks the output and the cache."""
        tables, ctx = self.tables(seqs)
        slots = np.concatenate([tables[i, np.arange(n) // BS].astype(np.int64) * BS +
                                np.arange(n) % BS for i, n in enumerate(lengths)])
        T = int(sum(lengths))
        self.append(slots, self.rand(T, HKV, D), self.rand(T, HKV, D))
        self.assert_cache_mirrors(what + " append")
        q = self.rand(T, HQ, D)
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        out = pkv.paged_prefill_attention(
            q.to(DEV), torch.as_tensor(cu, device=DEV), self.k_dev, self.v_dev,
            torch.as_tensor(tables, device=DEV), torch.as_tensor(ctx, device=DEV),
            int(max(lengths)), SCALE)
        ref = oracle.paged_prefill(W.to_u16(q), self.k_host, self.v_host, tables, ctx, cu, SCALE)
        assert_attention_close(out, ref, what + " prefill")

    def decode_step(self, seqs, groups=None, what=""):
        """One token per sequence: copy on write, append, attention."""
        slots, pairs = self.bm.append(seqs)
        self.copy(pairs)
        B = len(seqs)
        self.append(slots, self.rand(B, HKV, D), self.rand(B, HKV, D))
        self.assert_cache_mirrors(what + " append")
        tables, ctx = self.tables(seqs)
        q = self.rand(B, HQ, D)
        ref = oracle.paged_decode(W.to_u16(q), self.k_host, self.v_host, tables, ctx, SCALE)
        t_dev, c_dev = torch.as_tensor(tables, device=DEV), torch.as_tensor(ctx, device=DEV)
        out = pkv.paged_decode_attention(q.to(DEV), self.k_dev, self.v_dev, t_dev, c_dev,
                                         int(ctx.max()), SCALE)
        assert_attention_close(out, ref, what + " decode")
        if groups is not None:
            gs = np.asarray(groups, np.int32)
            sb = W.shared_prefix_blocks(tables, ctx, BS, gs).astype(np.int32)
            shared = pkv.paged_decode_attention_shared(
                q.to(DEV), self.k_dev, self.v_dev, t_dev, c_dev, int(ctx.max()), SCALE,
                torch.as_tensor(gs, device=DEV), torch.as_tensor(sb, device=DEV),
                int(np.diff(gs).max()))
            assert_attention_close(shared, ref, what + " shared decode")
        return pairs


    def rows(self, seq):
        """The logical K/V rows [len, Hkv, D] of a running sequence, read
        from the mirror through its table."""
        t = self.bm.block_table(seq)
        pos = np.arange(self.bm.length(seq))
        return (self.k_host[t[pos // BS], :, pos % BS], self.v_host[t[pos // BS], :, pos % BS])

    def preempt(self, seqs, mode):
        if mode == pkv.PREEMPT_RECOMPUTE:
            for s in seqs:
                self.saved[s] = self.rows(s)
        pairs = self.bm.preempt(seqs, mode)
        if len(pairs):
            pkv.block_swap(torch.as_tensor(pairs, device=DEV), [self.k_dev], [self.v_dev],
                           [self.k_swap], [self.v_swap])
            oracle.block_swap(pairs, [self.k_host], [self.v_host], [self.k_swap_m],
                              [self.v_swap_m])
            torch.cuda.synchronize()
            assert np.array_equal(W.to_u16(self.k_swap), self.k_swap_m), "swap out: K"
            assert np.array_equal(W.to_u16(self.v_swap), self.v_swap_m), "swap out: V"
        return pairs

    def resume(self, seqs):
        recompute = [s for s in seqs if self.bm.state(s) == pkv.BM_RECOMPUTE]
        pairs = self.bm.resume(seqs)
        if len(pairs):
            # pairs from page-locked host memory, read by the kernel directly
            pkv.block_swap(torch.as_tensor(pairs).pin_memory(), [self.k_swap], [self.v_swap],
                           [self.k_dev], [self.v_dev])
            oracle.block_swap(pairs, [self.k_swap_m], [self.v_swap_m], [self.k_host],
                              [self.v_host])
        for s in recompute:      # the recompute writes the sequence's rows again
            k, v = self.saved.pop(s)
            t = self.bm.block_table(s)
            pos = np.arange(k.shape[0])
            slots = t[pos // BS].astype(np.int64) * BS + pos % BS
            self.append(slots, W.from_u16(k), W.from_u16(v))
        self.assert_cache_mirrors("resume")
        return pairs


def test_prompts_forks_copy_on_write_and_block_reuse():
    f = Flow(seed=301)
    lengths = [37, 100, 16, 250]
    seqs = [f.bm.add_sequence(n) for n in lengths]
    f.prefill(seqs, lengths, "prompts")

    # two more branches of prompt 1 share its blocks (100 = 6 full blocks + 4)
    kids = [f.bm.fork(seqs[1]), f.bm.fork(seqs[1])]
    order = [seqs[0], seqs[1], kids[0], kids[1], seqs[2], seqs[3]]
    groups = [0, 1, 4, 5, 6]  # {0}, {1, kid, kid}, {2}, {3}
    pairs = f.decode_step(order, groups, "step 0")
    # the first write into the shared partial block copies it for all but one holder
    assert len(pairs) == 2
    for s in range(1, 4):
        pairs = f.decode_step(order, groups, "step %d" % s)
        assert len(pairs) == 0

    # retire sequence 3 (250 + 4 tokens, 16 blocks) and give its blocks to a new prompt
    free_before = f.bm.num_free_blocks()
    f.bm.free_sequence(seqs[3])
    assert f.bm.num_free_blocks() == free_before + 16
    new = f.bm.add_sequence(200)
    f.prefill([new], [200], "reused blocks")
    order = [seqs[0], seqs[1], kids[0], kids[1], seqs[2], new]
    f.decode_step(order, groups, "after reuse")


def test_prompt_that_fills_its_last_block_copies_nothing():
    f = Flow(seed=302)
    seqs = [f.bm.add_sequence(64)]
    f.prefill(seqs, [64], "prompt")
    kids = [f.bm.fork(seqs[0]) for _ in range(3)]
    order = seqs + kids
    pairs = f.decode_step(order, [0, 4], "step 0")
    assert len(pairs) == 0  # every branch starts a fresh block
    f.decode_step(order, [0, 4], "step 1")


def test_preemption_by_swap_and_by_recompute():
    # 30 blocks: the prompts take 23, so the decode steps exhaust the pool
    f = Flow(seed=303, nb=30, nh=24)
    lengths = [120, 60, 90, 44, 30]                    # 8 + 4 + 6 + 3 + 2 blocks
    seqs = [f.bm.add_sequence(n) for n in lengths]
    f.prefill(seqs, lengths, "prompts")
    kid = f.bm.fork(seqs[1])                           # shares 60 = 3 full + 12
    running = seqs + [kid]                             # priority: arrival order
    evicted, modes = [], [pkv.PREEMPT_SWAP, pkv.PREEMPT_RECOMPUTE]
    for step in range(40):
        k = f.bm.plan_preemption(running)
        if k:
            victims = running[len(running) - k:]
            f.preempt(victims, modes[len(evicted) % 2])
            evicted += victims
            running = running[:len(running) - k]
        f.decode_step(running, what="step %d" % step)
    c = f.bm.counters()
    assert c["preempted_swap"] >= 1 and c["preempted_recompute"] >= 1, c
    # two sequences retire; the evicted ones come back
    for s in running[:2]:
        f.bm.free_sequence(s)
    running = running[2:]
    f.resume(evicted)
    order = running + evicted
    for step in range(3):
        f.decode_step(order, what="after resume %d" % step)
    assert f.bm.num_free_host_blocks() == 24

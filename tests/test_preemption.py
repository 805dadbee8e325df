"""Pre-emption in the host block manager (include/pkv_block_manager.h), no
GPU.  "Running Out of Cache" (closing paragraph, and the glossary entry
"Pre-emption"): when even a paged cache runs out, a running request's cache is
evicted, to be recomputed or swapped back in later.

  * plan_preemption gives the fewest victims, from the back of the priority
    list, that let the rest append one token: on twin managers built by the
    same operations, evicting that many makes the append succeed and one
    fewer makes it fail;
  * a data model follows every block and host slot: token ids are written at
    the slots append gives, copy-on-write and swap pairs move them, resumed
    recomputes write them again.  After every operation each sequence's
    logical contents, read through its table, are exactly its tokens, so a
    wrong pair (or a block reused while still needed) shows at once;
  * swapping a family of forks out copies each shared block once, its host
    slot keeps one reference per holder, and swapping back restores the
    sharing;
  * device and host reference counts and free lists stay consistent under
    random operations; calls that cannot complete change nothing."""
import numpy as np
import pytest

from paged_kv_cache_245_gb300 import (BM_RECOMPUTE, BM_RETIRED, BM_RUNNING, BM_SWAPPED,
                                      PREEMPT_RECOMPUTE, PREEMPT_SWAP, BlockManager, PkvError)
from paged_kv_cache_245_gb300.build import build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()


class Model:
    """A block manager with the contents of its pools: dev[block, offset] and
    host[slot, offset] hold token ids (-1 = never written, -2 = freed)."""

    def __init__(self, nb, bs, nh, order=None):
        self.bm = BlockManager(nb, bs, free_order=order)
        self.bm.set_swap_space(nh)
        self.nb, self.bs, self.nh = nb, bs, nh
        self.dev = np.full((nb, bs), -1, np.int64)
        self.host = np.full((nh, bs), -1, np.int64)
        self.tokens = {}          # live sequence -> its token ids
        self.next = 0

    def _new_tokens(self, n):
        t = list(range(self.next, self.next + n))
        self.next += n
        return t

    def _write_all(self, s):
        t = self.bm.block_table(s)
        for p, tok in enumerate(self.tokens[s]):
            self.dev[t[p // self.bs], p % self.bs] = tok

    def _poison_free(self):
        for b in range(self.nb):
            if self.bm.ref_count(b) == 0:
                self.dev[b] = -2
        for h in range(self.nh):
            if self.bm.host_ref_count(h) == 0:
                self.host[h] = -2

    def add(self, n):
        s = self.bm.add_sequence(n)
        self.tokens[s] = self._new_tokens(n)
        self._write_all(s)            # the prompt's prefill writes its rows
        return s

    def fork(self, p):
        s = self.bm.fork(p)
        self.tokens[s] = list(self.tokens[p])
        return s

    def append(self, ids):
        slots, pairs = self.bm.append(ids)
        for src, dst in pairs:        # copies run before the step's writes
            self.dev[dst] = self.dev[src]
        for s, slot in zip(ids, slots):
            tok = self._new_tokens(1)[0]
            self.dev[slot // self.bs, slot % self.bs] = tok
            self.tokens[int(s)].append(tok)
        self._poison_free()
        return slots, pairs

    def preempt(self, ids, mode):
        pairs = self.bm.preempt(ids, mode)
        for b, h in pairs:
            self.host[h] = self.dev[b]
        self._poison_free()
        return pairs

    def resume(self, ids):
        recompute = [int(s) for s in ids if self.bm.state(int(s)) == BM_RECOMPUTE]
        pairs = self.bm.resume(ids)
        for h, d in pairs:
            self.dev[d] = self.host[h]
        for s in recompute:
            self._write_all(s)        # the recompute writes every row again
        self._poison_free()
        return pairs

    def free(self, s):
        self.bm.free_sequence(s)
        del self.tokens[s]
        self._poison_free()

    def check(self):
        dev_refs, host_refs = {}, {}
        for s, toks in self.tokens.items():
            st = self.bm.state(s)
            t = self.bm.block_table(s)
            assert self.bm.length(s) == len(toks)
            if st == BM_RECOMPUTE:
                assert len(t) == 0
                continue
            assert len(t) == (len(toks) + self.bs - 1) // self.bs
            pool, refs = (self.dev, dev_refs) if st == BM_RUNNING else (self.host, host_refs)
            assert st in (BM_RUNNING, BM_SWAPPED)
            got = [int(pool[t[p // self.bs], p % self.bs]) for p in range(len(toks))]
            assert got == toks, "sequence %d reads wrong rows" % s
            for x in t:
                refs[int(x)] = refs.get(int(x), 0) + 1
        for b in range(self.nb):
            assert self.bm.ref_count(b) == dev_refs.get(b, 0)
        for h in range(self.nh):
            assert self.bm.host_ref_count(h) == host_refs.get(h, 0)
        assert self.bm.num_free_blocks() == self.nb - len(dev_refs)
        assert self.bm.num_free_host_blocks() == self.nh - len(host_refs)

    def running(self):
        return [s for s in self.tokens if self.bm.state(s) == BM_RUNNING]

    def evicted(self):
        return [s for s in self.tokens if self.bm.state(s) in (BM_SWAPPED, BM_RECOMPUTE)]


def test_swapping_a_family_of_forks_keeps_its_sharing():
    m = Model(nb=20, bs=4, nh=10)
    root = m.add(10)                                   # blocks: 4 + 4 + 2 (partial)
    kids = [m.fork(root) for _ in range(3)]
    other = m.add(5)
    m.append([root] + kids)                            # three copy the partial block
    m.check()
    fam = [root] + kids
    held = {int(b) for s in fam for b in m.bm.block_table(s)}
    pairs = m.preempt(fam, PREEMPT_SWAP)
    assert sorted(int(b) for b in pairs[:, 0]) == sorted(held)   # each block once
    assert len(set(pairs[:, 1].tolist())) == len(held)
    m.check()
    # the two shared full blocks keep one host reference per holder
    t = m.bm.block_table(root)
    assert m.bm.host_ref_count(int(t[0])) == 4 and m.bm.host_ref_count(int(t[1])) == 4
    assert all(m.bm.state(s) == BM_SWAPPED for s in fam)
    m.append([other])
    back = m.resume(fam)
    assert back.shape[0] == len(held)
    m.check()
    assert m.bm.num_free_host_blocks() == 10
    tables = [m.bm.block_table(s) for s in fam]
    assert all(np.array_equal(tables[0][:2], x[:2]) for x in tables)   # shared again
    assert m.bm.ref_count(int(tables[0][0])) == 4
    m.append(fam + [other])
    m.check()
    c = m.bm.counters()
    assert c["preempted_swap"] == 4 and c["resumed"] == 4
    assert c["blocks_swapped_out"] == c["blocks_swapped_in"] == len(held)
    assert c["cow_copies"] == 3


def test_recompute_returns_the_blocks_and_keeps_the_length():
    m = Model(nb=12, bs=4, nh=0)
    a, b = m.add(9), m.add(7)
    free = m.bm.num_free_blocks()
    assert m.preempt([b], PREEMPT_RECOMPUTE).shape[0] == 0
    assert m.bm.state(b) == BM_RECOMPUTE and m.bm.length(b) == 7
    assert m.bm.num_free_blocks() == free + 2
    m.check()
    with pytest.raises(PkvError):
        m.bm.append([a, b])                            # an evicted sequence cannot step
    with pytest.raises(PkvError):
        m.bm.export([b], 4)
    m.append([a])
    m.resume([b])
    assert m.bm.state(b) == BM_RUNNING and len(m.bm.block_table(b)) == 2
    m.check()
    m.append([a, b])
    m.check()
    assert m.bm.counters()["tokens_recomputed"] == 7


def test_swap_with_a_running_sharer_copies_the_block_and_leaves_it_held():
    m = Model(nb=10, bs=4, nh=4)
    p = m.add(6)
    k = m.fork(p)
    pairs = m.preempt([k], PREEMPT_SWAP)
    assert pairs.shape[0] == 2
    assert all(m.bm.ref_count(int(b)) == 1 for b in m.bm.block_table(p))   # p keeps them
    m.append([p])                                      # p now writes in place: no copy
    assert m.bm.counters()["cow_copies"] == 0
    m.check()
    m.resume([k])
    m.check()
    assert not set(m.bm.block_table(k).tolist()) & set(m.bm.block_table(p).tolist())


@pytest.mark.parametrize("seed", range(6))
def test_plan_gives_the_fewest_victims(seed):
    def twin():
        rng = np.random.default_rng(seed)
        m = Model(nb=40, bs=4, nh=0, order=rng.permutation(40))
        live = []
        for _ in range(12):
            if live and rng.random() < 0.3:
                live.append(m.fork(int(rng.choice(live))))
            else:
                try:
                    live.append(m.add(int(rng.integers(1, 14))))
                except PkvError:
                    break
        for _ in range(30):                            # grow until steps stop fitting
            try:
                m.append(live)
            except PkvError:
                break
        prio = list(rng.permutation(live))
        return m, [int(s) for s in prio]

    m, prio = twin()
    k = m.bm.plan_preemption(prio)
    need_all = m.bm.step_blocks(prio)
    assert (k == 0) == (need_all <= m.bm.num_free_blocks())
    if k:
        m.preempt(prio[len(prio) - k:], PREEMPT_RECOMPUTE)
    keep = prio[:len(prio) - k]
    assert m.bm.step_blocks(keep) <= m.bm.num_free_blocks()
    m.append(keep)
    m.check()
    if k:
        m2, prio2 = twin()
        assert prio2 == prio
        m2.preempt(prio[len(prio) - k + 1:], PREEMPT_RECOMPUTE)
        with pytest.raises(PkvError, match="free blocks"):
            m2.append(prio[:len(prio) - k + 1])


def test_plan_counts_a_block_freed_only_when_all_its_holders_go():
    bm = BlockManager(5, 4)
    a = bm.add_sequence(8)           # blocks 0, 1: full, needs one
    b = bm.add_sequence(6)           # blocks 2, 3: partial, writes in place
    c = bm.fork(b)                   # shares 2, 3: one of b, c must copy
    bm.add_sequence(4)               # block 4: the pool is full
    assert bm.step_blocks([a, b, c]) == 2 and bm.num_free_blocks() == 0
    # evicting c alone frees nothing, but b then writes in place: a still needs one
    assert bm.plan_preemption([a, b, c]) == 2
    # evicting b and c frees blocks 2 and 3
    assert bm.plan_preemption([a, c, b]) == 2
    assert bm.plan_preemption([b, c, a]) == 1        # a's eviction frees 2 blocks
    assert bm.plan_preemption([]) == 0


def test_calls_that_cannot_complete_change_nothing():
    m = Model(nb=8, bs=4, nh=3)
    a = m.add(8)
    b = m.add(12)
    snap = lambda: ([m.bm.block_table(s).tolist() for s in (a, b)], m.bm.num_free_blocks(),
                    m.bm.num_free_host_blocks(), m.bm.state(a), m.bm.state(b))
    before = snap()
    with pytest.raises(PkvError, match="host blocks"):
        m.bm.preempt([a, b], PREEMPT_SWAP)             # 5 blocks, 3 slots
    assert snap() == before
    with pytest.raises(PkvError):
        m.bm.preempt([a, a], PREEMPT_SWAP)
    with pytest.raises(PkvError):
        m.bm.preempt([a], 7)
    with pytest.raises(PkvError):
        m.bm.resume([a])                               # running
    assert snap() == before
    m.preempt([b], PREEMPT_SWAP)
    with pytest.raises(PkvError):
        m.bm.set_swap_space(10)                        # slots in use
    with pytest.raises(PkvError):
        m.bm.preempt([b], PREEMPT_RECOMPUTE)           # already evicted
    m.add(20)                                          # takes every free block
    before = snap()
    with pytest.raises(PkvError, match="free blocks"):
        m.bm.resume([b])
    assert snap() == before
    m.check()
    # a swapped sequence that retires gives its host slots back
    m.free(b)
    assert m.bm.num_free_host_blocks() == 3 and m.bm.state(b) == BM_RETIRED
    m.bm.set_swap_space(10)
    m.nh, m.host = 10, np.full((10, m.bs), -1, np.int64)
    m.check()


def test_random_operations_with_preemption_keep_every_sequence_intact():
    rng = np.random.default_rng(2450)
    m = Model(nb=60, bs=4, nh=30, order=rng.permutation(60))
    for it in range(800):
        op = rng.integers(0, 12)
        run, ev = m.running(), m.evicted()
        try:
            if op < 2 or not m.tokens:
                m.add(int(rng.integers(0, 20)))
            elif op < 3 and run:
                m.fork(int(rng.choice(run)))
            elif op < 4:
                m.free(int(rng.choice(list(m.tokens))))
            elif op < 6 and run:
                ids = [int(s) for s in rng.choice(run, size=min(len(run), int(rng.integers(1, 4))),
                                                  replace=False)]
                m.preempt(ids, PREEMPT_SWAP if rng.random() < 0.6 else PREEMPT_RECOMPUTE)
            elif op < 8 and ev:
                ids = [int(s) for s in rng.choice(ev, size=min(len(ev), int(rng.integers(1, 4))),
                                                  replace=False)]
                m.resume(ids)
            elif run:
                prio = [int(s) for s in rng.permutation(run)]
                k = m.bm.plan_preemption(prio)
                if k:
                    m.preempt(prio[len(prio) - k:], PREEMPT_SWAP if rng.random() < 0.5
                              else PREEMPT_RECOMPUTE)
                m.append(prio[:len(prio) - k])
        except PkvError as e:
            assert "free blocks" in str(e) or "host blocks" in str(e), str(e)
        m.check()
    c = m.bm.counters()
    assert c["preempted_swap"] > 20 and c["preempted_recompute"] > 20 and c["resumed"] > 20

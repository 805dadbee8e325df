"""The host block manager (include/pkv_block_manager.h), no GPU:
  * it reproduces, step for step, the sharing scenario of the Yi-34B workload
    (32 prompts, 4 branches each, 64 decode steps): block tables, context
    lengths, slot mappings and copy-on-write pairs;
  * random sequences of add / fork / append / free keep the reference counts
    and the free list consistent, every sequence holds ceil(len / bs) blocks
    (less than one block wasted) and every new slot lies in its own table;
  * a step that needs more blocks than are free fails and changes nothing;
  * admitting requests of the workshop's length recipe into a 56 GB
    Llama-3-8B cache gives the workshop's counts ("Running Out of Cache",
    Workshop: 52 requests with 8192-token reservations at ~15 % fill, 333
    with 16-token blocks at 99 % fill, 6.4 times as many)."""
import json
import os

import numpy as np
import pytest

import workloads as W
from paged_kv_cache_245_gb300 import BlockManager, PkvError
from paged_kv_cache_245_gb300.build import build

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()


def test_reproduces_the_sharing_scenario():
    sc = W.sharing_scenario()
    bm = BlockManager(sc.num_blocks, sc.block_size, free_order=sc.free_order)
    B = len(sc.prompt_lens) * sc.n
    for p, plen in enumerate(sc.prompt_lens):
        root = bm.add_sequence(int(plen))
        assert root == p * sc.n
        for b in range(1, sc.n):
            assert bm.fork(root) == p * sc.n + b
    tables, _ = bm.export(np.arange(B), sc.tables_shared.shape[1])
    assert np.array_equal(tables, sc.tables_shared)
    for k, step in enumerate(sc.steps):
        slots, pairs = bm.append(np.arange(B))
        assert np.array_equal(slots, step.slot_mapping), k
        if k == 0:
            assert np.array_equal(pairs, sc.cow_pairs)
        else:
            assert pairs.shape[0] == 0
        tables, ctx = bm.export(np.arange(B), step.block_tables.shape[1])
        assert np.array_equal(ctx, step.ctx)
        assert np.array_equal(tables, step.block_tables), k


def _check_consistent(bm, live, num_blocks, bs):
    held = {}
    for s in live:
        t = bm.block_table(s)
        n = bm.length(s)
        assert len(t) == (n + bs - 1) // bs          # under one block of waste
        for blk in t:
            held[int(blk)] = held.get(int(blk), 0) + 1
    for blk in range(num_blocks):
        assert bm.ref_count(blk) == held.get(blk, 0)
    assert bm.num_free_blocks() == num_blocks - len(held)


def test_random_operations_keep_the_pool_consistent():
    rng = np.random.default_rng(245)
    nb, bs = 200, 4
    bm = BlockManager(nb, bs, free_order=rng.permutation(nb))
    live = []
    for it in range(600):
        op = rng.integers(0, 10)
        try:
            if op < 2 or not live:
                live.append(bm.add_sequence(int(rng.integers(0, 30))))
            elif op < 4:
                live.append(bm.fork(int(rng.choice(live))))
            elif op < 5:
                s = int(rng.choice(live))
                bm.free_sequence(s)
                live.remove(s)
            else:
                ids = rng.choice(live, size=min(len(live), int(rng.integers(1, 6))), replace=False)
                before = {int(s): bm.length(int(s)) for s in ids}
                slots, pairs = bm.append(ids)
                for s, slot in zip(ids, slots):
                    t = bm.block_table(int(s))
                    pos = before[int(s)]
                    assert slot == t[pos // bs] * bs + pos % bs   # the new slot is in its table
                    assert bm.length(int(s)) == pos + 1
                for src, dst in pairs:
                    assert bm.ref_count(int(dst)) >= 1 and src != dst
        except PkvError as e:
            assert "free blocks" in str(e)
        _check_consistent(bm, live, nb, bs)


def test_a_step_without_enough_blocks_changes_nothing():
    bm = BlockManager(6, 4)
    a = bm.add_sequence(8)          # blocks 0, 1 (both full)
    b = bm.add_sequence(3)          # block 2
    c = bm.fork(b)                  # shares block 2
    d = bm.add_sequence(12)         # blocks 3, 4, 5: none free now
    state = ([bm.block_table(s).tolist() for s in (a, b, c, d)], bm.num_free_blocks())
    with pytest.raises(PkvError, match="free blocks"):
        bm.append([a, b, c])        # a needs a block, b must copy block 2
    assert ([bm.block_table(s).tolist() for s in (a, b, c, d)], bm.num_free_blocks()) == state
    bm.free_sequence(d)
    slots, pairs = bm.append([a, b, c])
    assert pairs.tolist() == [[2, pairs[0, 1]]]     # b copies, c (last holder) writes in place
    assert slots[2] == 2 * 4 + 3
    with pytest.raises(PkvError):
        bm.append([a, a])           # a sequence may appear once per step


def _workshop_lengths(rng, n, g):
    prompt = np.maximum(1, np.rint(rng.exponential(g["mean_prompt_tokens"], n)))
    output = np.rint(rng.exponential(g["mean_output_tokens"], n))
    return np.minimum(prompt + output, g["max_tokens"]).astype(np.int64)


def test_workshop_capacity_through_the_block_manager():
    g = json.load(open(os.path.join(GOLDEN, "workshop_capacity.json")))
    per_token = W.SHAPES[g["model"]].kv_bytes_per_token()
    cache_tokens = int(g["cache_bytes"] // per_token)
    bs = g["block_tokens"]
    rng = np.random.default_rng(245)
    counts, fills = [], []
    for trial in range(5):
        bm = BlockManager(cache_tokens // bs, bs)
        lengths = _workshop_lengths(rng, 2000, g)
        admitted = 0
        for n in lengths:
            try:
                bm.add_sequence(int(n))
            except PkvError:
                break
            admitted += 1
        used = (cache_tokens // bs - bm.num_free_blocks()) * bs
        counts.append(admitted)
        fills.append(lengths[:admitted].sum() / used)
    # contiguous reservation: the printed arithmetic
    contig = cache_tokens // g["contiguous_reservation_tokens"]
    assert contig == g["contiguous_requests"]
    paged = float(np.mean(counts))
    assert abs(paged - g["paged_requests"]) <= 0.05 * g["paged_requests"], counts
    assert min(fills) >= g["paged_fill_percent"] / 100.0, fills
    assert abs(paged / contig - g["paged_over_contiguous"]) <= 0.35

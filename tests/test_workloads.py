"""Seeded input generators against the pages' printed shape figures and the
block-table bookkeeping rules.  No GPU."""
import json
import os

import numpy as np
import pytest

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_per_token_kv_footprint_matches_pages():
    g = _golden("kv_footprint.json")["per_token_kv_kib"]
    for name, kib in g.items():
        assert W.SHAPES[name].kv_bytes_per_token() == kib * 1024


def test_workshop_contiguous_capacity_arithmetic():
    g = _golden("workshop_capacity.json")
    per_token = W.SHAPES[g["model"]].kv_bytes_per_token()
    fit = int(g["cache_bytes"] // (g["contiguous_reservation_tokens"] * per_token))
    assert fit == g["contiguous_requests"]
    fill = (g["mean_prompt_tokens"] + g["mean_output_tokens"]) / g["contiguous_reservation_tokens"]
    assert abs(100 * fill - g["contiguous_fill_percent"]) < 1.0


@pytest.mark.parametrize("bs", [1, 5, 16, 128])
def test_blocks_cover_context_with_under_one_block_waste(bs):
    ctx = W.ragged_lengths(64)
    b = W.make_paged_batch(W.LLAMA3_8B, ctx, bs, seed=3)
    nblk = (b.ctx + bs - 1) // bs
    waste = nblk * bs - b.ctx
    assert np.all(waste >= 0) and np.all(waste < bs)
    used = np.concatenate([b.block_tables[i, :nblk[i]] for i in range(b.B)])
    assert len(np.unique(used)) == len(used), "no block belongs to two sequences"
    assert used.min() >= 0 and used.max() < b.num_blocks
    assert np.all(b.block_tables >= 0) and np.all(b.block_tables < b.num_blocks)
    # the new token's slot lies in the sequence's own last block
    assert np.all(np.isin(b.slot_mapping // bs, used))


def test_tiny_workload_matches_its_description():
    b = W.tiny_batch()
    assert list(b.ctx_pre) == [1, 17, 33, 100] and list(b.ctx) == [2, 18, 34, 101]
    assert b.num_blocks == 64 and b.block_size == 16
    assert sum((c + 15) // 16 for c in b.ctx) == 13
    assert W.tiny_batch(after_append=False).ctx.tolist() == [1, 17, 33, 100]


def test_generators_are_deterministic():
    a = W.layer_inputs(W.tiny_batch(), 0)
    b = W.layer_inputs(W.tiny_batch(), 0)
    assert all((x == y).all() for x, y in zip(
        (a.q, a.k_cache, a.v_cache, a.k_new), (b.q, b.k_cache, b.v_cache, b.k_new)))
    assert np.array_equal(W.ragged_lengths(), W.ragged_lengths())


def test_ragged_lengths_shape():
    ctx = W.ragged_lengths()
    assert ctx.shape == (256,) and ctx.min() >= 2 and ctx.max() <= 8192
    assert 700 < ctx.mean() < 1700  # prompt mean 1024 + about half of mean 256


def test_sharing_scenario_copy_on_write():
    sc = W.sharing_scenario(num_prompts=6, n=4, decode_steps=20, block_size=16)
    assert len(sc.steps) == 20 and sc.steps[0].B == 24
    partial = int(np.count_nonzero(sc.prompt_lens % 16))
    assert sc.cow_pairs.shape == (3 * partial, 2)
    first = sc.steps[0]
    for p in range(6):
        rows = first.block_tables[p * 4:(p + 1) * 4]
        full = int(sc.prompt_lens[p] // 16)
        # full prompt blocks stay shared by all four branches
        assert (rows[:, :full] == rows[0, :full]).all()
        # after step one, each branch's block holding its new token is its own
        last = first.slot_mapping[p * 4:(p + 1) * 4] // 16
        assert len(set(last.tolist())) == 4
    # copies go from a shared block to a fresh one
    assert len(set(sc.cow_pairs[:, 1].tolist())) == len(sc.cow_pairs)
    assert not set(sc.cow_pairs[:, 1].tolist()) & set(sc.tables_shared.ravel().tolist())

"""Block-table indexing, byte for byte: the library's gather (which locates
rows with the same address function as the append and decode kernels)
against the oracle's plain gather, for paged caches of many block sizes with
randomly placed blocks and for the contiguous reqId x S layout; checked mode
reports a bad block id."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_245_gb300 as pkv
import workloads as W
from paged_kv_cache_245_gb300 import binding

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _reset_modes():
    pkv.set_checked(False)
    yield
    pkv.set_checked(False)
    torch.cuda.synchronize()


def _batch(bs, seed):
    shape = W.ModelShape("g16_4", 1, 16, 4)
    ctx = np.array([0, 1, 2, 15, 16, 17, 33, 100, 255, 256, 257, 700], np.int32)
    return W.make_paged_batch(shape, ctx, bs, seed, spare_blocks=5)


@pytest.mark.parametrize("bs", [1, 3, 16, 24, 32, 128])
def test_paged_gather_matches_the_oracle(bs):
    b = _batch(bs, seed=100 + bs)
    li = W.layer_inputs(b, 0, device="cpu")
    cache = li.k_cache.to(DEV)
    tables = torch.as_tensor(b.block_tables, device=DEV)
    ctx = torch.as_tensor(b.ctx, device=DEV)
    got = W.to_u16(binding.debug_gather_paged(cache, tables, ctx, b.max_context))
    host = W.to_u16(li.k_cache)
    for i in range(b.B):
        c = int(b.ctx[i])
        for h in range(b.shape.num_kv_heads):
            ref = oracle.gather_paged(host, b.block_tables[i], c, bs, h)
            assert np.array_equal(got[i, h, :c], ref), (i, h)
            assert not got[i, h, c:].any()


def test_contig_gather_matches_the_oracle():
    b = _batch(16, seed=120)
    S = 1024
    # request rows in a shuffled order, with spare rows
    perm = np.random.default_rng(7).permutation(b.B + 3)[:b.B].astype(np.int32)
    b.req_ids = perm
    li = W.layer_inputs(b, 0, device="cpu")
    buf = W.paged_to_contig(li.k_cache, b, S, max_reqs=b.B + 3).to(DEV)
    req = torch.as_tensor(perm, device=DEV)
    ctx = torch.as_tensor(b.ctx, device=DEV)
    got = W.to_u16(binding.debug_gather_contig(buf, req, ctx, b.max_context))
    host = W.to_u16(buf.cpu())
    for i in range(b.B):
        c = int(b.ctx[i])
        for h in range(b.shape.num_kv_heads):
            ref = oracle.gather_contig(host, int(perm[i]), c, h)
            assert np.array_equal(got[i, h, :c], ref), (i, h)
            assert not got[i, h, c:].any()


def test_checked_gather_reports_a_bad_block_id():
    pkv.set_checked(True)
    b = _batch(16, seed=130)
    li = W.layer_inputs(b, 0, device="cpu")
    cache = li.k_cache.to(DEV)
    bad = b.block_tables.copy()
    bad[7, 0] = b.num_blocks + 5   # sequence 7 (ctx 100) reads its first block
    tables = torch.as_tensor(bad, device=DEV)
    ctx = torch.as_tensor(b.ctx, device=DEV)
    assert pkv.get_device_error() == "none"
    got = binding.debug_gather_paged(cache, tables, ctx, b.max_context)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == "block_id"
    assert torch.count_nonzero(got[7, :, :16]) == 0

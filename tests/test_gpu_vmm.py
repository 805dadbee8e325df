"""Contiguous (reqId x S) K/V buffers whose physical memory is mapped on
demand ("Leveraging Low-Level CUDA APIs for vAttention's Dynamic Memory",
5.2: reserve, create, map, set access; 5.2.3: a request's sub-tensor at
reqId x S): decode attention and the decode step on them match the CPU
oracle, and give the same bytes as on regular device memory; the append
writes the same rows the oracle's append writes; pages are mapped as a
request grows and unmapped when it ends, and released pages are reused.
Every kernel call is preceded by a host check that the rows it can touch
are backed."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_245_gb300 as pkv
import workloads as W
from parity import assert_attention_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
VARIANTS = [pkv.VARIANT_AUTO, pkv.VARIANT_SPLIT, pkv.VARIANT_TC_12X2]


@pytest.fixture(autouse=True)
def _reset_modes():
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    yield
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    torch.cuda.synchronize()


def _assert_backed(vm, ctx):
    for r, c in enumerate(ctx):
        assert vm.backed_tokens(r) >= c, "request %d: %d rows backed, %d needed" % (
            r, vm.backed_tokens(r), c)


@pytest.mark.parametrize("variant", VARIANTS)
def test_attention_and_step_on_mapped_memory_match_oracle_and_regular_memory(variant):
    pkv.set_decode_variant(variant)
    shape = W.ModelShape("v32_8", 1, 32, 8)
    ctx = np.array([1, 17, 300, 1024, 2047, 2048, 5000, 9000], np.int32)
    S = 16384   # 4 MiB per KV head: requests grow across page boundaries
    b = W.make_paged_batch(shape, ctx, 16, 301)
    li = W.layer_inputs(b, 0, device=DEV, fast_cache=True)
    kb = W.paged_to_contig(li.k_cache, b, S)
    vb = W.paged_to_contig(li.v_cache, b, S)
    vm = pkv.VmmBuffer(b.B, shape.num_kv_heads, S)
    try:
        for r, c in enumerate(ctx):
            vm.ensure(r, int(c))
        _assert_backed(vm, ctx)
        for r, c in enumerate(ctx):
            vm.k[r, :, :c].copy_(kb[r, :, :c])
            vm.v[r, :, :c].copy_(vb[r, :, :c])
        req = torch.arange(b.B, dtype=torch.int32, device=DEV)
        ctx_d = torch.as_tensor(ctx, device=DEV)
        scale = W.default_scale(shape)
        ref = pkv.contig_decode_attention(li.q, kb, vb, req, ctx_d, int(ctx.max()), scale)
        _assert_backed(vm, ctx)
        out = pkv.contig_decode_attention(li.q, vm.k, vm.v, req, ctx_d, int(ctx.max()), scale)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        # the oracle, from host copies of the inputs (nothing from the GPU path)
        h_q = W.to_u16(li.q)
        h_kb, h_vb = W.to_u16(kb).copy(), W.to_u16(vb).copy()
        h_req = np.arange(b.B, dtype=np.int32)
        assert_attention_close(out, oracle.contig_decode(h_q, h_kb, h_vb, h_req, ctx, scale),
                               "attention on mapped memory")
        # one more token per request: back it, then append + attend in one call
        ctx2 = ctx + 1
        for r, c in enumerate(ctx2):
            vm.ensure(r, int(c))
        _assert_backed(vm, ctx2)
        slots = torch.as_tensor(np.arange(b.B, dtype=np.int64) * S + ctx2 - 1, device=DEV)
        ctx2_d = torch.as_tensor(ctx2, device=DEV)
        kr, vr = kb.clone(), vb.clone()
        ref2 = pkv.contig_decode_step(slots, li.k_new, li.v_new, li.q, kr, vr, req, ctx2_d,
                                      int(ctx2.max()), scale)
        out2 = pkv.contig_decode_step(slots, li.k_new, li.v_new, li.q, vm.k, vm.v, req, ctx2_d,
                                      int(ctx2.max()), scale)
        torch.cuda.synchronize()
        assert torch.equal(out2, ref2)
        for r, c in enumerate(ctx2):
            assert torch.equal(vm.k[r, :, :c], kr[r, :, :c])
            assert torch.equal(vm.v[r, :, :c], vr[r, :, :c])
        # the oracle's append into its host copies, then its attention
        oracle.kv_append(slots.cpu().numpy(), W.to_u16(li.k_new), W.to_u16(li.v_new), h_kb, h_vb)
        for r, c in enumerate(ctx2):
            assert np.array_equal(W.to_u16(vm.k[r, :, :c]), h_kb[r, :, :c]), "K rows of %d" % r
            assert np.array_equal(W.to_u16(vm.v[r, :, :c]), h_vb[r, :, :c]), "V rows of %d" % r
        assert_attention_close(out2, oracle.contig_decode(h_q, h_kb, h_vb, h_req, ctx2, scale),
                               "decode step on mapped memory")
    finally:
        vm.close()


def test_pages_follow_the_requests():
    hkv, S = 8, 16384
    vm = pkv.VmmBuffer(4, hkv, S)
    try:
        st = vm.stats()
        rows_per_page = st["page_bytes"] // 256
        assert st["mapped_pages"] == 0
        # request 0 grows one token at a time past a page boundary
        for t in range(1, rows_per_page + 40):
            vm.ensure(0, t)
        per_head = (S * 256) // st["page_bytes"]   # pages per KV head region
        expect = hkv * min(2, per_head) if S * 256 >= st["page_bytes"] else None
        st = vm.stats()
        if expect is not None:
            assert st["mapped_pages"] == expect
        assert vm.backed_tokens(0) == ((rows_per_page + 39 + 15) // 16) * 16
        vm.ensure(1, 100)
        mapped = vm.stats()["mapped_pages"]
        created = vm.stats()["created_pages"]
        vm.release(0)
        assert vm.backed_tokens(0) == 0
        assert vm.stats()["mapped_pages"] < mapped
        vm.ensure(2, rows_per_page + 1)        # reuses the released physical pages
        assert vm.stats()["created_pages"] == created
        with pytest.raises(pkv.PkvError):
            vm.ensure(1, S + 1)
        with pytest.raises(pkv.PkvError):
            vm.ensure(4, 1)
    finally:
        vm.close()

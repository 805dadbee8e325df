"""Causal prefill over a paged cache (pkv_paged_prefill_attention) against
the oracle: every group size, several block sizes, chunks from one token to
several tiles over cached contexts of any length (and fresh prompts), a
chunk of one token against the decode kernel, and checked mode."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_245_gb300 as pkv
import workloads as W
from parity import assert_attention_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _reset_modes():
    pkv.set_checked(False)
    yield
    pkv.set_checked(False)
    torch.cuda.synchronize()


def _case(hq, hkv, cached, lq, bs, seed):
    """Paged K/V holding every sequence's full context (cached + chunk), the
    chunks' queries packed by cu_seqlens_q."""
    shape = W.ModelShape("p%d_%d" % (hq, hkv), 1, hq, hkv)
    ctx = np.asarray(cached, np.int32) + np.asarray(lq, np.int32)
    b = W.make_paged_batch(shape, ctx, bs, seed, spare_blocks=3)
    li = W.layer_inputs(b, 0, device="cpu")
    cu = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((int(cu[-1]), hq, 128), generator=g).to(torch.bfloat16)
    return b, li, q, cu


def _gpu(b, li, q, cu):
    return pkv.paged_prefill_attention(
        q.to(DEV), torch.as_tensor(cu, device=DEV), li.k_cache.to(DEV), li.v_cache.to(DEV),
        torch.as_tensor(b.block_tables, device=DEV), torch.as_tensor(b.ctx, device=DEV),
        int(np.diff(cu).max()), W.default_scale(b.shape))


def _oracle(b, li, q, cu):
    return oracle.paged_prefill(W.to_u16(q), W.to_u16(li.k_cache), W.to_u16(li.v_cache),
                                b.block_tables, b.ctx, cu, W.default_scale(b.shape))


@pytest.mark.parametrize("bs", [16, 32, 48, 64, 128, 256])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (32, 8), (16, 2)])
def test_chunks_against_oracle(hq, hkv, bs):
    cached = [0, 3, 100, 64, 17, 0]
    lq = [1, 5, 64, 65, 130, 33]
    b, li, q, cu = _case(hq, hkv, cached, lq, bs, seed=hq * 7 + hkv + bs)
    assert_attention_close(_gpu(b, li, q, cu), _oracle(b, li, q, cu),
                           "prefill G=%d bs=%d" % (hq // hkv, bs))


def test_llama_shaped_chunked_prefill():
    b, li, q, cu = _case(32, 8, [256, 44], [256, 256], 16, seed=91)
    assert_attention_close(_gpu(b, li, q, cu), _oracle(b, li, q, cu), "llama chunks")


def test_chunk_of_one_token_is_the_decode_call():
    b, li, q, cu = _case(32, 8, [0, 16, 99, 700], [1, 1, 1, 1], 16, seed=92)
    out = _gpu(b, li, q, cu)
    dec = pkv.paged_decode_attention(q.to(DEV), li.k_cache.to(DEV), li.v_cache.to(DEV),
                                     torch.as_tensor(b.block_tables, device=DEV),
                                     torch.as_tensor(b.ctx, device=DEV), b.max_context,
                                     W.default_scale(b.shape))
    ref = _oracle(b, li, q, cu)
    assert_attention_close(out, ref, "prefill, chunks of one")
    assert_attention_close(dec, ref, "decode")


def test_checked_mode_reports_a_chunk_longer_than_its_context():
    pkv.set_checked(True)
    b, li, q, cu = _case(8, 2, [10, 10], [4, 4], 16, seed=93)
    bad_ctx = b.ctx.copy()
    bad_ctx[1] = 2                       # shorter than its 4-token chunk
    assert pkv.get_device_error() == "none"
    pkv.paged_prefill_attention(q.to(DEV), torch.as_tensor(cu, device=DEV), li.k_cache.to(DEV),
                                li.v_cache.to(DEV), torch.as_tensor(b.block_tables, device=DEV),
                                torch.as_tensor(bad_ctx, device=DEV), 4, W.default_scale(b.shape))
    torch.cuda.synchronize()
    assert pkv.get_device_error() == "context"


def test_long_chunks_span_many_row_and_key_tiles():
    # 2800 / 2052 / 516 rows: several CTAs of 256 rows each; up to 9 key tiles
    b, li, q, cu = _case(32, 8, [0, 300, 1000], [700, 513, 129], 16, seed=94)
    assert_attention_close(_gpu(b, li, q, cu), _oracle(b, li, q, cu), "long chunks")


@pytest.mark.parametrize("hq,hkv", [(56, 8), (24, 8), (40, 8), (12, 2)])
def test_groups_that_do_not_divide_128(hq, hkv):
    # G = 7 (Yi-34B heads), 3, 5 and 6: row tiles of whole tokens (126 or 125
    # rows and zero padding), chunks that end inside a row tile and in the
    # second row tile of an item
    b, li, q, cu = _case(hq, hkv, [5, 0, 130], [100, 300, 37], 16, seed=95 + hq)
    assert_attention_close(_gpu(b, li, q, cu), _oracle(b, li, q, cu), "G=%d" % (hq // hkv))


def test_output_only_16_byte_aligned():
    # G = 7 writes rows with plain stores, 32 bytes at a time when out is
    # 32-byte aligned; an out 16 bytes off that uses 16-byte stores, same bytes
    b, li, q, cu = _case(56, 8, [5, 0], [100, 37], 16, seed=90)
    args = (q.to(DEV), torch.as_tensor(cu, device=DEV), li.k_cache.to(DEV), li.v_cache.to(DEV),
            torch.as_tensor(b.block_tables, device=DEV), torch.as_tensor(b.ctx, device=DEV),
            int(np.diff(cu).max()), W.default_scale(b.shape))
    ref = pkv.paged_prefill_attention(*args)
    flat = torch.zeros(q.numel() + 8, dtype=torch.bfloat16, device=DEV)
    out = flat[8:].view(q.shape)
    assert out.data_ptr() % 32 == 16
    pkv.paged_prefill_attention(*args, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert_attention_close(ref, _oracle(b, li, q, cu), "G=7, 32-byte stores")


@pytest.mark.parametrize("scale", [0.5, 2.0, 0.0, -0.3])
def test_growing_maxima_and_degenerate_scale(scale):
    # large scales make the running maximum jump between key tiles (the
    # rescale of O in tensor memory); scale 0 gives the mean of the visible V;
    # a negative scale takes the general (masked) softmax path on every tile
    b, li, q, cu = _case(16, 4, [0, 200, 513], [400, 129, 300], 16, seed=96)
    out = pkv.paged_prefill_attention(
        q.to(DEV), torch.as_tensor(cu, device=DEV), li.k_cache.to(DEV), li.v_cache.to(DEV),
        torch.as_tensor(b.block_tables, device=DEV), torch.as_tensor(b.ctx, device=DEV),
        int(np.diff(cu).max()), scale)
    ref = oracle.paged_prefill(W.to_u16(q), W.to_u16(li.k_cache), W.to_u16(li.v_cache),
                               b.block_tables, b.ctx, cu, scale)
    assert_attention_close(out, ref, "scale %g" % scale)


def test_short_chunk_after_a_long_context():
    # 157 key tiles of 128 behind a 64-token chunk, block_size 32
    b, li, q, cu = _case(8, 2, [20000, 7], [64, 40], 32, seed=97)
    assert_attention_close(_gpu(b, li, q, cu), _oracle(b, li, q, cu), "long context")


def test_sequences_without_new_tokens_are_skipped():
    # chunks of 0 tokens (repeated cu_seqlens_q entries) next to real ones
    b, li, q, cu = _case(32, 8, [50, 20, 300, 9], [0, 70, 0, 3], 16, seed=98)
    assert_attention_close(_gpu(b, li, q, cu), _oracle(b, li, q, cu), "empty chunks")


def test_checked_mode_reports_a_chunk_longer_than_the_host_bound():
    pkv.set_checked(True)
    b, li, q, cu = _case(8, 2, [10, 10], [4, 6], 16, seed=99)
    assert pkv.get_device_error() == "none"
    pkv.paged_prefill_attention(q.to(DEV), torch.as_tensor(cu, device=DEV), li.k_cache.to(DEV),
                                li.v_cache.to(DEV), torch.as_tensor(b.block_tables, device=DEV),
                                torch.as_tensor(b.ctx, device=DEV), 4, W.default_scale(b.shape))
    torch.cuda.synchronize()
    assert pkv.get_device_error() == "context"


def test_checked_mode_reports_a_block_id_outside_the_pool():
    pkv.set_checked(True)
    b, li, q, cu = _case(8, 2, [40, 10], [8, 8], 16, seed=100)
    tables = b.block_tables.copy()
    tables[0, 1] = li.k_cache.shape[0]  # one past the last block
    assert pkv.get_device_error() == "none"
    pkv.paged_prefill_attention(q.to(DEV), torch.as_tensor(cu, device=DEV), li.k_cache.to(DEV),
                                li.v_cache.to(DEV), torch.as_tensor(tables, device=DEV),
                                torch.as_tensor(b.ctx, device=DEV), 8, W.default_scale(b.shape))
    torch.cuda.synchronize()
    assert pkv.get_device_error() == "block_id"


def _contig_case(hq, hkv, S, max_reqs, req_ids, cached, lq, seed):
    g = torch.Generator().manual_seed(seed)
    kb = torch.randn((max_reqs, hkv, S, 128), generator=g).to(torch.bfloat16)
    vb = torch.randn((max_reqs, hkv, S, 128), generator=g).to(torch.bfloat16)
    ctx = (np.asarray(cached) + np.asarray(lq)).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    q = torch.randn((int(cu[-1]), hq, 128), generator=g).to(torch.bfloat16)
    return kb, vb, np.asarray(req_ids, np.int32), ctx, cu, q


@pytest.mark.parametrize("hq,hkv", [(32, 8), (56, 8)])
def test_contiguous_layout_against_oracle(hq, hkv):
    # request rows at reqId x S; the oracle reads the buffer as a paged cache
    # of max_reqs blocks of S rows and one-entry tables [reqId]
    kb, vb, req, ctx, cu, q = _contig_case(hq, hkv, 1024, 6, [4, 0, 5, 2], [0, 300, 17, 900],
                                           [200, 129, 40, 100], seed=101)
    out = pkv.contig_prefill_attention(q.to(DEV), torch.as_tensor(cu, device=DEV), kb.to(DEV),
                                       vb.to(DEV), torch.as_tensor(req, device=DEV),
                                       torch.as_tensor(ctx, device=DEV), int(np.diff(cu).max()),
                                       128 ** -0.5)
    ref = oracle.paged_prefill(W.to_u16(q), W.to_u16(kb), W.to_u16(vb), req[:, None], ctx, cu,
                               128 ** -0.5)
    assert_attention_close(out, ref, "contiguous prefill")


def test_contiguous_prefill_on_memory_mapped_on_demand():
    # only the rows each request needs are backed; the output is the same
    # bytes as on regular memory and matches the oracle
    S = 16384
    kb, vb, req, ctx, cu, q = _contig_case(32, 8, S, 3, [0, 1, 2], [8000, 0, 12000],
                                           [192, 70, 300], seed=102)
    vm = pkv.VmmBuffer(3, 8, S)
    try:
        for r in range(3):
            vm.ensure(int(req[r]), int(ctx[r]))
            assert vm.backed_tokens(int(req[r])) >= ctx[r]
            vm.k[int(req[r]), :, :ctx[r]].copy_(kb[int(req[r]), :, :ctx[r]])
            vm.v[int(req[r]), :, :ctx[r]].copy_(vb[int(req[r]), :, :ctx[r]])
        args = (torch.as_tensor(req, device=DEV), torch.as_tensor(ctx, device=DEV),
                int(np.diff(cu).max()), 128 ** -0.5)
        qd, cud = q.to(DEV), torch.as_tensor(cu, device=DEV)
        ref = pkv.contig_prefill_attention(qd, cud, kb.to(DEV), vb.to(DEV), *args)
        out = pkv.contig_prefill_attention(qd, cud, vm.k, vm.v, *args)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        # and against the oracle, from the host inputs alone (request rows at
        # reqId x S read as one-entry tables over blocks of S rows)
        want = oracle.paged_prefill(W.to_u16(q), W.to_u16(kb), W.to_u16(vb), req[:, None], ctx,
                                    cu, 128 ** -0.5)
        assert_attention_close(out, want, "contiguous prefill on mapped memory")
    finally:
        torch.cuda.synchronize()
        vm.close()

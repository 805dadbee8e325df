"""CUDA path against the CPU oracle on small and edge-case inputs, plus the
bit-exact invariances (block relabelling, block size, layout, append, copy).
Every call goes through the C ABI via the Python binding."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_245_gb300 as pkv
import workloads as W
from parity import DeviceLayer, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _reset_modes():
    pkv.set_split_tiles(0)
    pkv.set_checked(False)
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    yield
    pkv.set_split_tiles(0)
    pkv.set_checked(False)
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    torch.cuda.synchronize()


# every decode kernel: automatic choice, the split CUDA-core kernel, and the
# tensor-core kernel in both of its CTA shapes
VARIANTS = [pkv.VARIANT_AUTO, pkv.VARIANT_SPLIT, pkv.VARIANT_TC_8X3, pkv.VARIANT_TC_12X2]
TC_VARIANTS = (pkv.VARIANT_TC_8X3, pkv.VARIANT_TC_12X2)


def _batch(hq, hkv, ctx, bs, seed=5, spare=3):
    shape = W.ModelShape("t%d_%d" % (hq, hkv), 1, hq, hkv)
    return W.make_paged_batch(shape, np.asarray(ctx, np.int32), bs, seed, spare_blocks=spare)


def test_tiny_workload_before_and_after_append():
    """The tiny workload: attend at contexts {1,17,33,100}, append one token
    each, attend again at {2,18,34,101}."""
    before = W.tiny_batch(after_append=False)
    after = W.tiny_batch()
    L = DeviceLayer(after, 0, DEV)
    L.set_step(before)
    assert_attention_close(L.gpu_attend(), L.oracle_attend(), "before append")
    L.set_step(after)
    L.gpu_append()
    L.oracle_append()
    torch.cuda.synchronize()
    L.assert_caches_equal()
    assert_attention_close(L.gpu_attend(), L.oracle_attend(), "after append")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (6, 2), (8, 2), (10, 2), (12, 2), (14, 2),
                                    (16, 2), (56, 8), (32, 4)])
def test_every_group_size(hq, hkv, variant):
    pkv.set_decode_variant(variant)
    ctx = [1, 2, 15, 16, 17, 31, 33, 64, 100, 257, 700]
    L = DeviceLayer(_batch(hq, hkv, ctx, 16), 0, DEV)
    L.gpu_append()
    L.oracle_append()
    torch.cuda.synchronize()
    L.assert_caches_equal()
    assert_attention_close(L.gpu_attend(), L.oracle_attend(), "G=%d" % (hq // hkv))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("bs", [1, 3, 8, 16, 24, 32, 64, 128, 256])
def test_block_sizes(bs, variant):
    if variant in TC_VARIANTS and bs % 16:
        pytest.skip("the tensor-core kernel takes block sizes that are multiples of 16")
    pkv.set_decode_variant(variant)
    ctx = [1, 5, 16, 17, 48, 129, 300, 513]
    L = DeviceLayer(_batch(8, 2, ctx, bs, seed=bs), 0, DEV)
    L.gpu_append()
    L.oracle_append()
    torch.cuda.synchronize()
    L.assert_caches_equal()
    assert_attention_close(L.gpu_attend(), L.oracle_attend(), "bs=%d" % bs)


@pytest.mark.parametrize("tiles", [4, 8, 12, 16, 64])
def test_split_counts_agree_with_oracle(tiles):
    """Any number of context splits gives the oracle's result (the split
    combine is exercised whenever a context spans more than one split)."""
    pkv.set_decode_variant(pkv.VARIANT_SPLIT)
    pkv.set_split_tiles(tiles)
    ctx = [1, 63, 64, 65, 250, 1024, 2049]
    L = DeviceLayer(_batch(32, 8, ctx, 16, seed=11), 0, DEV)
    n = pkv.decode_num_splits(len(ctx), 32, 8, max(ctx))
    assert n == math.ceil(math.ceil(max(ctx) / 16) / tiles)
    assert_attention_close(L.gpu_attend(), L.oracle_attend(), "tiles=%d" % tiles)


@pytest.mark.parametrize("variant", VARIANTS)
def test_zero_and_single_contexts(variant):
    """ctx = 0 gives zeros; ctx = 1 returns v_0 exactly (bf16 round trip)."""
    pkv.set_decode_variant(variant)
    b = _batch(8, 2, [1, 1, 5], 16)
    b.ctx = np.array([0, 1, 5], np.int32)
    L = DeviceLayer(b, 0, DEV)
    L.set_step(b)
    out = L.gpu_attend()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[0]) == 0
    blk = int(b.block_tables[1, 0])
    v0 = L.v_cache[blk, :, 0, :]                      # [Hkv, D]
    expect = v0.repeat_interleave(4, dim=0)           # each query head reads h // G
    assert torch.equal(out[1], expect)
    assert_attention_close(out, L.oracle_attend(), "ctx 0/1/5")


@pytest.mark.parametrize("variant", VARIANTS)
def test_all_empty_batch_and_empty_call(variant):
    pkv.set_decode_variant(variant)
    b = _batch(8, 2, [3, 3], 16)
    b.ctx = np.zeros(2, np.int32)
    L = DeviceLayer(b, 0, DEV)
    L.set_step(b)
    out = pkv.paged_decode_attention(L.q, L.k_cache, L.v_cache, L.tables, L.ctx, 0, L.scale)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    empty_q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device=DEV)
    pkv.paged_decode_attention(empty_q, L.k_cache, L.v_cache, L.tables[:0], L.ctx[:0], 0, 1.0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_block_relabelling_is_bit_exact(variant):
    pkv.set_decode_variant(variant)
    ctx = [7, 100, 333, 1025]
    b = _batch(32, 8, ctx, 16, seed=21)
    L = DeviceLayer(b, 0, DEV)
    base = L.gpu_attend().clone()
    perm = torch.randperm(b.num_blocks, generator=torch.Generator().manual_seed(1)).to(DEV)
    k2 = torch.empty_like(L.k_cache)
    v2 = torch.empty_like(L.v_cache)
    k2[perm] = L.k_cache
    v2[perm] = L.v_cache
    t2 = perm[L.tables.long()].int()
    out = pkv.paged_decode_attention(L.q, k2, v2, t2, L.ctx, b.max_context, L.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, base)


@pytest.mark.parametrize("variant", VARIANTS)
def test_block_size_and_layout_do_not_change_bits(variant):
    """The kernels tile the logical sequence in 16-token tiles whatever the
    layout, so block sizes 16..128 and the contiguous layout give identical
    bits for identical logical K/V."""
    pkv.set_decode_variant(variant)
    ctx = W.ragged_lengths(24, seed=3, max_len=1500)
    ref = None
    base = W.make_paged_batch(W.LLAMA3_8B, ctx, 16, seed=9)
    L16 = DeviceLayer(base, 0, DEV)
    k_log = W.paged_to_contig(L16.k_cache, base, 1536)
    v_log = W.paged_to_contig(L16.v_cache, base, 1536)
    for bs in (16, 32, 64, 128):
        b = W.make_paged_batch(W.LLAMA3_8B, ctx, bs, seed=100 + bs)
        kc = torch.zeros((b.num_blocks, 8, bs, 128), dtype=torch.bfloat16, device=DEV)
        vc = torch.zeros_like(kc)
        for i in range(b.B):
            n = (int(ctx[i]) + bs - 1) // bs
            ids = torch.as_tensor(b.block_tables[i, :n].astype(np.int64), device=DEV)
            kpad = torch.zeros((8, n * bs, 128), dtype=torch.bfloat16, device=DEV)
            vpad = torch.zeros_like(kpad)
            kpad[:, :ctx[i]] = k_log[i, :, :ctx[i]]
            vpad[:, :ctx[i]] = v_log[i, :, :ctx[i]]
            kc[ids] = kpad.reshape(8, n, bs, 128).permute(1, 0, 2, 3)
            vc[ids] = vpad.reshape(8, n, bs, 128).permute(1, 0, 2, 3)
        out = pkv.paged_decode_attention(L16.q, kc, vc, torch.as_tensor(b.block_tables, device=DEV),
                                         L16.ctx, int(ctx.max()), L16.scale)
        torch.cuda.synchronize()
        if ref is None:
            ref = out.clone()
            assert_attention_close(out, L16.oracle_attend(), "bs=16")
        else:
            assert torch.equal(out, ref), "bs=%d changed the bits" % bs
    req = torch.arange(b.B, dtype=torch.int32, device=DEV)
    out = pkv.contig_decode_attention(L16.q, k_log, v_log, req, L16.ctx, int(ctx.max()), L16.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref), "contiguous layout changed the bits"


def test_contig_against_oracle_with_permuted_request_rows():
    rng = np.random.default_rng(4)
    S, max_reqs, hq, hkv = 320, 9, 16, 4
    ctx = np.array([1, 17, 320, 0, 99, 256], np.int32)
    req = rng.permutation(max_reqs)[:len(ctx)].astype(np.int32)
    g = torch.Generator().manual_seed(77)
    kb = torch.randn((max_reqs, hkv, S, 128), generator=g).to(torch.bfloat16)
    vb = torch.randn((max_reqs, hkv, S, 128), generator=g).to(torch.bfloat16)
    q = torch.randn((len(ctx), hq, 128), generator=g).to(torch.bfloat16)
    ref = oracle.contig_decode(W.to_u16(q), W.to_u16(kb), W.to_u16(vb), req, ctx, 0.1)
    for variant, tiles in ((0, 0), (1, 0), (1, 4), (3, 0)):
        pkv.set_decode_variant(variant)
        pkv.set_split_tiles(tiles)
        out = pkv.contig_decode_attention(q.to(DEV), kb.to(DEV), vb.to(DEV),
                                          torch.as_tensor(req, device=DEV),
                                          torch.as_tensor(ctx, device=DEV), S, 0.1)
        assert_attention_close(out, ref, "contig variant=%d tiles=%d" % (variant, tiles))


def test_contig_append_positions():
    """Append into the contiguous layout: slot = reqId * S + position."""
    S, hkv = 64, 2
    kb = torch.zeros((3, hkv, S, 128), dtype=torch.bfloat16, device=DEV)
    vb = torch.zeros_like(kb)
    g = torch.Generator().manual_seed(3)
    kn = torch.randn((2, hkv, 128), generator=g).to(torch.bfloat16)
    vn = torch.randn((2, hkv, 128), generator=g).to(torch.bfloat16)
    slots = np.array([2 * S + 7, 0 * S + 63], np.int64)
    pkv.kv_append(torch.as_tensor(slots, device=DEV), kn.to(DEV), vn.to(DEV), kb, vb)
    hk, hv = np.zeros((3, hkv, S, 128), np.uint16), np.zeros((3, hkv, S, 128), np.uint16)
    oracle.kv_append(slots, W.to_u16(kn), W.to_u16(vn), hk, hv)
    torch.cuda.synchronize()
    assert np.array_equal(W.to_u16(kb), hk) and np.array_equal(W.to_u16(vb), hv)


def test_append_skips_padding_and_touches_nothing_else():
    b = _batch(8, 4, [5, 16, 17, 40], 16)
    L = DeviceLayer(b, 0, DEV)
    slots = b.slot_mapping.copy()
    slots[1] = -1
    L.slots = torch.as_tensor(slots, device=DEV)
    L.b.slot_mapping = slots
    L.gpu_append()
    L.oracle_append()
    torch.cuda.synchronize()
    L.assert_caches_equal()


@pytest.mark.parametrize("layers", [1, 3, 70])
def test_block_copy_bit_exact(layers):
    nb, hkv, bs = 40, 2, 16
    g = torch.Generator().manual_seed(layers)
    ks = [torch.randn((nb, hkv, bs, 128), generator=g).to(torch.bfloat16) for _ in range(layers)]
    vs = [torch.randn((nb, hkv, bs, 128), generator=g).to(torch.bfloat16) for _ in range(layers)]
    pairs = np.array([[3, 7], [0, 39], [12, 2], [5, 6]], np.int64)
    dk = [t.to(DEV) for t in ks]
    dv = [t.to(DEV) for t in vs]
    pkv.block_copy(torch.as_tensor(pairs, device=DEV), dk, dv)
    hk = [W.to_u16(t).copy() for t in ks]
    hv = [W.to_u16(t).copy() for t in vs]
    oracle.block_copy(pairs, hk, hv)
    torch.cuda.synchronize()
    for l in range(layers):
        assert np.array_equal(W.to_u16(dk[l]), hk[l]) and np.array_equal(W.to_u16(dv[l]), hv[l])


def test_large_block_copy():
    """Copy-on-write at Yi-34B block size (8 KV heads x 16 x 128 = 32 KiB)."""
    nb = 300
    g = torch.Generator(device=DEV).manual_seed(5)
    ks = [torch.randn((nb, 8, 16, 128), generator=g, device=DEV).to(torch.bfloat16) for _ in range(2)]
    vs = [torch.randn((nb, 8, 16, 128), generator=g, device=DEV).to(torch.bfloat16) for _ in range(2)]
    src = torch.randperm(150, generator=torch.Generator().manual_seed(1))[:96]
    dst = 150 + torch.randperm(150, generator=torch.Generator().manual_seed(2))[:96]
    pairs = torch.stack([src, dst], 1).to(torch.int64)
    before = [t.clone() for t in ks + vs]
    pkv.block_copy(pairs.to(DEV), ks, vs)
    torch.cuda.synchronize()
    for t, b0 in zip(ks + vs, before):
        assert torch.equal(t[dst.to(DEV)], b0[src.to(DEV)])
        keep = torch.ones(nb, dtype=torch.bool)
        keep[dst] = False
        assert torch.equal(t[keep.to(DEV)], b0[keep.to(DEV)])


# ------------------------------------------------------------- checked mode

@pytest.mark.parametrize("variant", VARIANTS)
def test_checked_mode_reports_bad_block_id_without_fault(variant):
    pkv.set_decode_variant(variant)
    b = _batch(8, 2, [20, 40], 16)
    L = DeviceLayer(b, 0, DEV)
    assert pkv.get_device_error() == "none"
    pkv.set_checked(True)
    bad = L.tables.clone()
    bad[1, 1] = b.num_blocks + 5
    pkv.paged_decode_attention(L.q, L.k_cache, L.v_cache, bad, L.ctx, b.max_context, L.scale)
    assert pkv.get_device_error() == "block_id"
    assert pkv.get_device_error() == "none"   # reading clears it
    out = L.gpu_attend()                       # good tables still fine in checked mode
    assert_attention_close(out, L.oracle_attend(), "checked mode")
    assert pkv.get_device_error() == "none"


@pytest.mark.parametrize("variant", VARIANTS)
def test_checked_mode_reports_bad_slot_and_context_and_request(variant):
    pkv.set_decode_variant(variant)
    b = _batch(8, 2, [20, 40], 16)
    L = DeviceLayer(b, 0, DEV)
    pkv.set_checked(True)
    slots = L.slots.clone()
    slots[0] = b.num_blocks * 16 + 3
    pkv.kv_append(slots, L.k_new, L.v_new, L.k_cache, L.v_cache)
    assert pkv.get_device_error() == "slot"
    long_ctx = L.ctx.clone()
    long_ctx[1] = b.max_context + 100
    pkv.paged_decode_attention(L.q, L.k_cache, L.v_cache, L.tables, long_ctx, b.max_context, L.scale)
    assert pkv.get_device_error() == "context"
    kb = torch.zeros((2, 2, 64, 128), dtype=torch.bfloat16, device=DEV)
    req = torch.tensor([0, 7], dtype=torch.int32, device=DEV)
    c2 = torch.tensor([10, 10], dtype=torch.int32, device=DEV)
    out = pkv.contig_decode_attention(L.q, kb, kb, req, c2, 64, 0.1)
    assert pkv.get_device_error() == "req_id"
    assert torch.count_nonzero(out[1]) == 0
    pairs = torch.tensor([[0, b.num_blocks]], dtype=torch.int64, device=DEV)
    pkv.block_copy(pairs, [L.k_cache], [L.v_cache])
    assert pkv.get_device_error() == "copy_pair"


@pytest.mark.parametrize("variant", [pkv.VARIANT_SPLIT, pkv.VARIANT_TC_12X2])
def test_workspace_is_checked(variant):
    pkv.set_decode_variant(variant)
    b = _batch(32, 8, [4000, 4000], 16)
    L = DeviceLayer(b, 0, DEV)
    need = pkv.decode_workspace_size(2, 32, 8, b.max_context)
    assert need > 1024
    small = torch.empty(1024 if variant == pkv.VARIANT_TC_12X2 else 16, dtype=torch.uint8,
                        device=DEV)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attention(L.q, L.k_cache, L.v_cache, L.tables, L.ctx, b.max_context,
                                   L.scale, workspace=small)
    assert e.value.status == 3
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    out = pkv.paged_decode_attention(L.q, L.k_cache, L.v_cache, L.tables, L.ctx, b.max_context,
                                     L.scale, workspace=ws)
    assert_attention_close(out, L.oracle_attend(), "explicit workspace")


@pytest.mark.parametrize("variant", VARIANTS)
def test_large_batch_is_chunked(variant):
    """More sequences than one tensor-core launch takes (512) run as
    consecutive chunks; ragged short contexts, many of them empty."""
    pkv.set_decode_variant(variant)
    ctx = np.random.default_rng(8).integers(0, 40, size=1500).astype(np.int32)
    ctx[:3] = [1, 39, 0]
    b = _batch(16, 4, np.maximum(ctx, 1), 16, seed=12)
    b.ctx = ctx
    L = DeviceLayer(b, 0, DEV)
    L.set_step(b)
    assert_attention_close(L.gpu_attend(), L.oracle_attend(), "1500 sequences")


def test_variant_knob_rejects_tensor_core_for_odd_block_size():
    pkv.set_decode_variant(pkv.VARIANT_TC_8X3)
    b = _batch(8, 2, [20, 40], 24)
    L = DeviceLayer(b, 0, DEV)
    with pytest.raises(pkv.PkvError) as e:
        L.gpu_attend()
    assert e.value.status == 2


def test_wait_limit_reports_timeout_and_context_survives():
    """A wait that can never complete (test hook: one warp announces 16 bytes
    no copy brings) gives up after its time limit and reports a timeout in
    the device error word; the next call on the same context is correct."""
    pkv.set_decode_variant(pkv.VARIANT_TC_12X2)
    b = _batch(32, 8, [1024] * 64, 16, seed=31)
    L = DeviceLayer(b, 0, DEV)
    assert pkv.get_device_error() == "none"
    pkv.lib().pkv_debug_stall_next_decode()
    L.gpu_attend()
    assert pkv.get_device_error() == "timeout"
    out = L.gpu_attend()
    assert pkv.get_device_error() == "none"
    assert_attention_close(out, L.oracle_attend(), "after a timed-out call")


def test_merge_wait_limit_reports_timeout_and_context_survives():
    """The in-kernel merge of a pair cut by the CTA ranges re-reads a piece
    record that is not there yet for at most 2 s.  Test hook: CTA 1 writes
    no record in the next call, so CTA 0 (whose last segment holds the first
    tiles of the pair it shares with CTA 1) gives up and reports a timeout;
    the next call on the same context is correct."""
    pkv.set_decode_variant(pkv.VARIANT_TC_12X2)
    b = _batch(32, 8, [1024] * 64, 16, seed=37)
    L = DeviceLayer(b, 0, DEV)
    assert pkv.get_device_error() == "none"
    pkv.lib().pkv_debug_drop_next_piece_record()
    L.gpu_attend()
    assert pkv.get_device_error() == "timeout"
    out = L.gpu_attend()
    assert pkv.get_device_error() == "none"
    assert_attention_close(out, L.oracle_attend(), "after a merge that timed out")


def test_cuda_graph_replay_matches_direct_calls():
    """The decode step (append + attention) captured in a CUDA graph and
    replayed gives the same bytes as direct calls."""
    b = _batch(32, 8, [300, 1024, 17, 700] * 16, 16, seed=41)
    L = DeviceLayer(b, 0, DEV)
    k0, v0 = L.k_cache.clone(), L.v_cache.clone()
    ws = torch.empty(pkv.decode_workspace_size(b.B, 32, 8, b.max_context), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty_like(L.q)

    def step():
        pkv.kv_append(L.slots, L.k_new, L.v_new, L.k_cache, L.v_cache)
        pkv.paged_decode_attention(L.q, L.k_cache, L.v_cache, L.tables, L.ctx, b.max_context,
                                   L.scale, out=out, workspace=ws)

    step()
    torch.cuda.synchronize()
    direct = out.clone()
    L.k_cache.copy_(k0)
    L.v_cache.copy_(v0)
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    L.k_cache.copy_(k0)
    L.v_cache.copy_(v0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, direct)
    L.oracle_append()
    assert_attention_close(out, L.oracle_attend(), "graph replay")


@pytest.mark.parametrize("variant", VARIANTS)
def test_long_contexts(variant):
    """Contexts of 65K-131K positions next to tiny ones: a pair's tiles span
    many CTA ranges (many split records per pair)."""
    pkv.set_decode_variant(variant)
    ctx = [1, 131072, 65536 + 7, 5]
    L = DeviceLayer(_batch(32, 8, ctx, 16, seed=21), 0, DEV, fast_cache=True)
    L.gpu_append()
    L.oracle_append()
    assert_attention_close(L.gpu_attend(), L.oracle_attend(), "long contexts")


@pytest.mark.parametrize("variant", [pkv.VARIANT_AUTO, pkv.VARIANT_TC_12X2, pkv.VARIANT_TC_8X3])
def test_one_pair_across_every_cta(variant):
    """One sequence, one KV head, 200K positions: the only pair is cut by
    every CTA boundary, so its combine merges far more than 32 records."""
    pkv.set_decode_variant(variant)
    L = DeviceLayer(_batch(8, 1, [200000], 16, seed=22), 0, DEV, fast_cache=True)
    assert_attention_close(L.gpu_attend(), L.oracle_attend(), "one long pair")

"""The decode-step calls (append + attention of one layer in one call)
against the two separate calls -- the same bytes in the caches and the output
-- and against the oracle, for every kernel variant and both layouts, replayed
from a CUDA graph, in checked mode, and with a bad argument (nothing may be
launched: the append must not have run)."""
import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_cache_245_gb300 as pkv
import workloads as W
from parity import DeviceLayer, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
VARIANTS = [pkv.VARIANT_AUTO, pkv.VARIANT_SPLIT, pkv.VARIANT_TC_8X3, pkv.VARIANT_TC_12X2]


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


def _case(name):
    if name == "small":
        shape = W.ModelShape("t32_8", 1, 32, 8)
        ctx = [1, 2, 16, 17, 100, 257, 700, 1024]
        return W.make_paged_batch(shape, np.asarray(ctx, np.int32), 16, 71, spare_blocks=3), False
    if name == "ragged":
        return W.make_paged_batch(W.LLAMA3_8B, W.ragged_lengths(96, seed=72, max_len=3000), 16,
                                  72), True
    return W.uniform_batch(W.LLAMA3_8B, 64, 1024, 16, seed=73), True


def _separate_then_fused(L, b):
    """(caches and output of append + attention as two calls, the same from
    the step call), both from the same starting caches."""
    k0, v0 = L.k_cache.clone(), L.v_cache.clone()
    L.gpu_append()
    ref = L.gpu_attend()
    torch.cuda.synchronize()
    kr, vr = L.k_cache.clone(), L.v_cache.clone()
    L.k_cache.copy_(k0)
    L.v_cache.copy_(v0)
    out = pkv.paged_decode_step(L.slots, L.k_new, L.v_new, L.q, L.k_cache, L.v_cache, L.tables,
                                L.ctx, b.max_context, L.scale)
    torch.cuda.synchronize()
    return (kr, vr, ref), (L.k_cache, L.v_cache, out)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("case", ["small", "ragged", "llama_b64"])
def test_paged_step_is_append_then_attention(case, variant):
    pkv.set_decode_variant(variant)
    b, fast = _case(case)
    L = DeviceLayer(b, 0, DEV, fast_cache=fast)
    (kr, vr, ref), (kf, vf, out) = _separate_then_fused(L, b)
    assert torch.equal(kf, kr) and torch.equal(vf, vr), "caches differ"
    assert torch.equal(out, ref), "output differs from the two calls"
    L.oracle_append()
    L.assert_caches_equal()
    assert_attention_close(out, L.oracle_attend(), "%s step" % case)


@pytest.mark.parametrize("variant", VARIANTS)
def test_contig_step_is_append_then_attention(variant):
    pkv.set_decode_variant(variant)
    b, _ = _case("small")
    L = DeviceLayer(b, 0, DEV)
    S = 1024
    # rows of each request as they stand before this step's token
    pre = dataclasses.replace(b, ctx=b.ctx_pre)
    kb0 = W.paged_to_contig(L.k_cache, pre, S)
    vb0 = W.paged_to_contig(L.v_cache, pre, S)
    req = torch.as_tensor(b.req_ids, device=DEV)
    slots = torch.as_tensor(b.req_ids.astype(np.int64) * S + b.ctx.astype(np.int64) - 1,
                            device=DEV)
    kb, vb = kb0.clone(), vb0.clone()
    pkv.kv_append(slots, L.k_new, L.v_new, kb, vb)
    ref = pkv.contig_decode_attention(L.q, kb, vb, req, L.ctx, b.max_context, L.scale)
    kf, vf = kb0.clone(), vb0.clone()
    out = pkv.contig_decode_step(slots, L.k_new, L.v_new, L.q, kf, vf, req, L.ctx,
                                 b.max_context, L.scale)
    torch.cuda.synchronize()
    assert torch.equal(kf, kb) and torch.equal(vf, vb)
    assert torch.equal(out, ref)
    L.oracle_append()
    assert_attention_close(out, L.oracle_attend(), "contiguous step")


def test_step_in_a_cuda_graph_matches_direct_calls():
    b, fast = _case("llama_b64")
    L = DeviceLayer(b, 0, DEV, fast_cache=fast)
    k0, v0 = L.k_cache.clone(), L.v_cache.clone()
    ws = torch.empty(pkv.decode_workspace_size(b.B, 32, 8, b.max_context), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty_like(L.q)

    def step():
        pkv.paged_decode_step(L.slots, L.k_new, L.v_new, L.q, L.k_cache, L.v_cache, L.tables,
                              L.ctx, b.max_context, L.scale, out=out, workspace=ws)

    step()
    torch.cuda.synchronize()
    direct = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        L.k_cache.copy_(k0)
        L.v_cache.copy_(v0)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, direct)


def test_step_in_checked_mode_reports_nothing_on_valid_input():
    pkv.set_checked(True)
    b, fast = _case("ragged")
    L = DeviceLayer(b, 0, DEV, fast_cache=fast)
    assert pkv.get_device_error() == "none"
    (kr, vr, ref), (kf, vf, out) = _separate_then_fused(L, b)
    assert pkv.get_device_error() == "none"
    assert torch.equal(out, ref) and torch.equal(kf, kr)


def test_bad_attention_argument_launches_nothing():
    """A step whose attention arguments are invalid fails before the append
    is launched: the caches keep their bytes."""
    b, _ = _case("small")
    L = DeviceLayer(b, 0, DEV)
    k0, v0 = L.k_cache.clone(), L.v_cache.clone()
    too_long = L.tables.shape[1] * b.block_size + 1   # beyond what the tables hold
    with pytest.raises(pkv.PkvError):
        pkv.paged_decode_step(L.slots, L.k_new, L.v_new, L.q, L.k_cache, L.v_cache, L.tables,
                              L.ctx, too_long, L.scale)
    torch.cuda.synchronize()
    assert torch.equal(L.k_cache, k0) and torch.equal(L.v_cache, v0)


@pytest.mark.parametrize("variant", [pkv.VARIANT_TC_8X3, pkv.VARIANT_TC_12X2])
def test_step_with_sequences_without_a_new_token(variant):
    """With the tensor-core kernel the step is one launch that also does the
    append; a negative slot means no new token for that sequence: its
    attention then reads the cache as it stands, as after the two calls."""
    pkv.set_decode_variant(variant)
    b, _ = _case("small")
    L = DeviceLayer(b, 0, DEV)
    slots = L.slots.clone()
    slots[1::2] = -1
    k0, v0 = L.k_cache.clone(), L.v_cache.clone()
    pkv.kv_append(slots, L.k_new, L.v_new, L.k_cache, L.v_cache)
    ref = pkv.paged_decode_attention(L.q, L.k_cache, L.v_cache, L.tables, L.ctx, b.max_context,
                                     L.scale)
    torch.cuda.synchronize()
    kr, vr = L.k_cache.clone(), L.v_cache.clone()
    L.k_cache.copy_(k0)
    L.v_cache.copy_(v0)
    out = pkv.paged_decode_step(slots, L.k_new, L.v_new, L.q, L.k_cache, L.v_cache, L.tables,
                                L.ctx, b.max_context, L.scale)
    torch.cuda.synchronize()
    assert torch.equal(L.k_cache, kr) and torch.equal(L.v_cache, vr), "caches differ"
    assert torch.equal(out, ref), "output differs from the two calls"


def test_step_reports_a_slot_that_is_not_the_last_position():
    """Checked mode: with the append inside the tensor-core kernel, a slot in
    range that is not the sequence's position ctx - 1 is reported (the
    attention would read the new token there)."""
    pkv.set_checked(True)
    pkv.set_decode_variant(pkv.VARIANT_TC_12X2)
    b, _ = _case("small")
    L = DeviceLayer(b, 0, DEV)
    slots = L.slots.clone()
    i = int(np.argmax(b.ctx > 100))   # a sequence with several blocks
    slots[i] = slots[i] - 1           # the position before its last
    assert pkv.get_device_error() == "none"
    pkv.paged_decode_step(slots, L.k_new, L.v_new, L.q, L.k_cache, L.v_cache, L.tables, L.ctx,
                          b.max_context, L.scale)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == "slot"

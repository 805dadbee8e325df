"""Decode attention with shared prompt blocks read once per group of
sequences (pkv_paged_decode_attention_shared) against the regular paged call
and the oracle: the Yi-34B parallel-sampling scenario, synthetic groups over
every group size (singletons, empty suffixes, ragged members), and checked
mode's report for a member whose context does not cover the shared blocks."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_245_gb300 as pkv
import workloads as W
from parity import DeviceLayer, assert_attention_close, shared_groups_batch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _reset_modes():
    pkv.set_checked(False)
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    yield
    pkv.set_checked(False)
    torch.cuda.synchronize()


def shared_prefix_blocks(tables, ctx, bs, starts):
    return W.shared_prefix_blocks(tables, ctx, bs, np.asarray(starts))


def own_bound(b, starts, shared):
    """The largest number of own (unshared) positions of any sequence."""
    sizes = np.diff(np.asarray(starts))
    per_seq = np.repeat(shared, sizes) * b.block_size
    return int((b.ctx - per_seq).max())


def _run(b, starts, shared, L, own=-1):
    gs = torch.as_tensor(np.asarray(starts, np.int32), device=DEV)
    sb = torch.as_tensor(shared, device=DEV)
    maxg = int(np.max(np.diff(starts)))
    return pkv.paged_decode_attention_shared(L.q, L.k_cache, L.v_cache, L.tables, L.ctx,
                                             b.max_context, L.scale, gs, sb, maxg,
                                             max_own_tokens=own)


OWN = ["tensor_core_pass", "in_merge"]


@pytest.mark.parametrize("own", OWN + ["own_tiles"])
@pytest.mark.parametrize("step", [0, 1, 63])
def test_yi34b_sharing_scenario(step, own):
    """The exact own bound (<= 79 positions, 4 members) puts the own positions
    in masked key tiles of the prefix kernel, which with one chunk per group
    writes the output itself; a loose bound of 256 keeps them in the merge."""
    sc = W.sharing_scenario()
    b = sc.steps[step]
    L = DeviceLayer(b, 0, DEV, fast_cache=True)
    starts = np.arange(0, b.B + 1, sc.n)
    shared = shared_prefix_blocks(b.block_tables, b.ctx, b.block_size, starts)
    assert shared.min() > 0
    bound = {"tensor_core_pass": -1, "in_merge": 256,
             "own_tiles": own_bound(b, starts, shared)}[own]
    out = _run(b, starts, shared, L, bound)
    ref = L.gpu_attend()
    torch.cuda.synchronize()
    assert_attention_close(out, ref.float().cpu().numpy().astype(np.float64), "vs regular call")
    if step != 1:
        assert_attention_close(out, L.oracle_attend(), "vs oracle")


def _synthetic(hq, hkv, own, sizes, max_prompt_blocks, seed):
    if own == "own_tiles":  # few own positions: masked key tiles of the prefix kernel
        b, starts = shared_groups_batch(hq, hkv, sizes, max_prompt_blocks, seed, own_max=12,
                                        singleton_blocks=0)
    else:
        b, starts = shared_groups_batch(hq, hkv, sizes, max_prompt_blocks, seed)
    L = DeviceLayer(b, 0, DEV)
    shared = shared_prefix_blocks(b.block_tables, b.ctx, b.block_size, starts)
    bound = own_bound(b, starts, shared)
    assert bound <= 256   # singletons keep whole contexts: within the in-merge bound
    out = _run(b, starts, shared, L, -1 if own == OWN[0] else bound)
    assert_attention_close(out, L.oracle_attend(), "synthetic groups G=%d sizes %s"
                           % (hq // hkv, sizes))


@pytest.mark.parametrize("own", OWN + ["own_tiles"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (28, 4), (32, 4)])
def test_synthetic_groups(hq, hkv, own):
    """Groups of 1..5 sequences over one prompt each: members have their own
    tail blocks after the shared ones; some members stop exactly at the
    shared blocks."""
    _synthetic(hq, hkv, own, [1, 2, 3, 4, 5, 1, 3], 40, hq * 10 + hkv)


@pytest.mark.parametrize("own", OWN + ["own_tiles"])
def test_large_groups_and_long_shared_prompts(own):
    """A group of 24 members at G = 8 (192 rows: two row blocks of the prefix
    kernel) and shared prompts of up to 600 blocks (several chunks of the
    shared positions)."""
    _synthetic(32, 4, own, [24, 2, 1, 5], 600, 77)


@pytest.mark.parametrize("own", ["tensor_core_pass", "own_tiles"])
def test_checked_mode_reports_an_uncovered_member(own):
    pkv.set_checked(True)
    sc = W.sharing_scenario(num_prompts=4, decode_steps=1)
    b = sc.steps[0]
    L = DeviceLayer(b, 0, DEV, fast_cache=True)
    starts = np.arange(0, b.B + 1, sc.n)
    shared = shared_prefix_blocks(b.block_tables, b.ctx, b.block_size, starts)
    bound = own_bound(b, starts, shared)
    shared[0] = int(b.ctx[:sc.n].max() // b.block_size) + 1   # beyond every member's context
    assert pkv.get_device_error() == "none"
    _run(b, starts, shared, L, -1 if own == "tensor_core_pass" else bound)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == "context"


def test_checked_mode_reports_an_own_part_beyond_the_bound():
    pkv.set_checked(True)
    sc = W.sharing_scenario(num_prompts=4, decode_steps=8)
    b = sc.steps[7]
    L = DeviceLayer(b, 0, DEV, fast_cache=True)
    starts = np.arange(0, b.B + 1, sc.n)
    shared = shared_prefix_blocks(b.block_tables, b.ctx, b.block_size, starts)
    bound = own_bound(b, starts, shared)
    assert pkv.get_device_error() == "none"
    _run(b, starts, shared, L, bound)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == "none"
    _run(b, starts, shared, L, bound - 1)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == "context"


def test_launch_count_follows_the_own_mode():
    """The Yi-34B sharing step: the exact own bound makes the call one launch
    (own key tiles, one chunk per group), a loose bound of 256 two (prefix
    kernel, merge), no bound four (prep, prefix kernel, tensor-core pass,
    merge); a rejected shape reports -1."""
    sc = W.sharing_scenario()
    b = sc.steps[0]
    starts = np.arange(0, b.B + 1, sc.n)
    shared = shared_prefix_blocks(b.block_tables, b.ctx, b.block_size, starts)
    sh = b.shape

    def launches(own, bs=b.block_size):
        return pkv.shared_decode_launches(b.B, len(starts) - 1, sc.n, b.block_tables.shape[1],
                                          b.max_context, bs, own, sh.num_q_heads,
                                          sh.num_kv_heads)

    assert launches(own_bound(b, starts, shared)) == 1
    assert launches(256) == 2
    assert launches(-1) == 4
    assert launches(16, bs=8) == -1

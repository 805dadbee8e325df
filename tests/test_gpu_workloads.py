"""The five workloads at full size, in the launch configuration the benchmark
uses, against the CPU oracle.  Sampled where the oracle would be slow:
layers {0, last}; for the sharing workload decode steps {first, last}; every
sequence and head of a sampled layer/step is compared."""
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
def _modes():
    pkv.set_split_tiles(0)
    pkv.set_checked(False)
    yield
    torch.cuda.synchronize()


def _append_and_attend(batch, layer, fast=True):
    L = DeviceLayer(batch, layer, DEV, fast_cache=fast)
    L.gpu_append()
    out = L.gpu_attend()
    L.oracle_append()
    torch.cuda.synchronize()
    # append: the written slots hold the new rows, nothing else moved
    L.assert_caches_equal()
    return L, out


@pytest.mark.parametrize("layer", [0, 31])
def test_yi6b_batch64(layer):
    b = W.uniform_batch(W.YI_6B, 64, 1024, 16, seed=W.SEED_YI6B)
    L, out = _append_and_attend(b, layer)
    assert_attention_close(out, L.oracle_attend(), "Yi-6B layer %d" % layer)


@pytest.mark.parametrize("layer", [0, 31])
@pytest.mark.parametrize("B", W.LLAMA_SWEEP_BATCHES)
def test_llama_sweep(B, layer):
    b = W.uniform_batch(W.LLAMA3_8B, B, 1024, 16, seed=W.SEED_LLAMA)
    L, out = _append_and_attend(b, layer)
    assert_attention_close(out, L.oracle_attend(), "Llama b%d layer %d" % (B, layer))


def test_llama_b64_bench_configuration():
    """Exactly the benchmark's per-layer call (same seed, workspace, split
    plan), two layers."""
    b = W.uniform_batch(W.LLAMA3_8B, 64, 1024, 16, seed=W.SEED_LLAMA)
    for layer in (0, 31):
        L = DeviceLayer(b, layer, DEV, fast_cache=True)
        n = pkv.decode_workspace_size(64, 32, 8, 1024)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=DEV)
        L.gpu_append()
        out = pkv.paged_decode_attention(L.q, L.k_cache, L.v_cache, L.tables, L.ctx, 1024,
                                         L.scale, workspace=ws)
        L.oracle_append()
        assert_attention_close(out, L.oracle_attend(), "bench config layer %d" % layer)


@pytest.mark.parametrize("layer", [0, 31])
@pytest.mark.parametrize("bs", W.RAGGED_BLOCK_SIZES)
def test_ragged_paged_and_contiguous(bs, layer):
    """Ragged serving batch (prompt ~ Exp(1024), output ~ Exp(256), max 8192)
    in the paged layout, and the same logical K/V in the contiguous layout at
    S = 8192 (reqId x S): paged matches the oracle, contiguous matches paged
    bit for bit.  Layers 0 and 31 (first and last of the Llama-3-8B shape)."""
    b = W.ragged_batch(bs)
    L, out = _append_and_attend(b, layer)
    assert_attention_close(out, L.oracle_attend(), "ragged bs=%d layer %d" % (bs, layer))
    if bs == 16:
        S = 8192
        kb = W.paged_to_contig(L.k_cache, b, S)
        vb = W.paged_to_contig(L.v_cache, b, S)
        req = torch.as_tensor(b.req_ids, device=DEV)
        out_c = pkv.contig_decode_attention(L.q, kb, vb, req, L.ctx, b.max_context, L.scale)
        torch.cuda.synchronize()
        assert torch.equal(out_c, out)
        # the contiguous path against the oracle on a sample of requests
        idx = np.array([0, 1, 77, 255])
        ref = oracle.contig_decode(L.h_q[idx], W.to_u16(kb[idx]), W.to_u16(vb[idx]),
                                   np.arange(4, dtype=np.int32), b.ctx[idx], L.scale)
        assert_attention_close(out_c[torch.as_tensor(idx, device=DEV)], ref, "contig sample")


def test_yi34b_prefix_sharing_with_copy_on_write():
    """32 prompts ~ U[1024, 8192] decoded 4 ways (batch 128) over shared
    prompt blocks; block_copy on the first write into a shared partial
    block, then 64 decode steps of append + attention.  Layers {0, 59},
    attention checked at steps {0, 63}; copies and appends bit-exact."""
    sc = W.sharing_scenario()
    shape = sc.shape
    first, last = sc.steps[0], sc.steps[-1]
    layers = [DeviceLayer(first, l, DEV, fast_cache=True) for l in (0, 59)]
    pairs = torch.as_tensor(sc.cow_pairs, device=DEV)
    pkv.block_copy(pairs, [L.k_cache for L in layers], [L.v_cache for L in layers])
    oracle.block_copy(sc.cow_pairs, [L.h_k for L in layers], [L.h_v for L in layers])
    g = torch.Generator().manual_seed(W.SEED_YI34B)
    for step, batch in enumerate(sc.steps):
        kn = torch.randn((batch.B, shape.num_kv_heads, shape.head_dim), generator=g).to(torch.bfloat16)
        vn = torch.randn((batch.B, shape.num_kv_heads, shape.head_dim), generator=g).to(torch.bfloat16)
        for L in layers:
            L.set_step(batch)
            L.gpu_append(kn.to(DEV), vn.to(DEV))
            L.oracle_append(W.to_u16(kn), W.to_u16(vn))
            if step in (0, len(sc.steps) - 1):
                out = L.gpu_attend()
                torch.cuda.synchronize()
                assert_attention_close(out, L.oracle_attend(), "Yi-34B step %d" % step)
    torch.cuda.synchronize()
    for L in layers:
        L.assert_caches_equal()
    # branches of one prompt agree on the shared prefix: the last step's tables
    # still point branch 0..3 of prompt 0 at the same full prompt blocks
    full = int(sc.prompt_lens[0] // 16)
    assert (last.block_tables[0:4, :full] == last.block_tables[0, :full]).all()

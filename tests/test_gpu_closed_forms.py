"""Every decode kernel on inputs whose attention output has a closed form.

Standard attention softmax(scale * q K^T) V (the computation the paged and
the contiguous layouts both serve: "Running Out of Cache", PagedAttention;
"Leveraging Low-Level CUDA APIs for vAttention's Dynamic Memory", 5.2.3)
reduces to something a reader can check by eye when:

* every key of a KV head is the same vector: all logits tie, so the output
  is the mean of the context's V rows;
* the query is zero, or the scale is zero: the same mean of V;
* every V row of a KV head is the same vector c: the output is c;
* the query points along one key k_j with length 100 (q = 100 k_j/|k_j|):
  that logit exceeds every other by more than 30, so the output is v_j to
  within e^-30 of the total weight;
* scale 2 on N(0,1) data (no closed form): a sharply peaked softmax whose
  weights are far from uniform, which stresses the rounding of the
  probabilities to bf16 before the P.V product; compared with the oracle.

Each case runs every kernel: the automatic choice, the CUDA-core split
kernel, both tensor-core CTA shapes, the contiguous layout on the split and
the tensor-core kernels, and the shared-prefix call in each of its
own-position modes (a second tensor-core pass, CUDA cores in the merge, and
masked key tiles of the prefix kernel, which then writes the output).  The output is compared with the closed form and with
the fp64 oracle at |err| <= 1e-2 + 1e-2 |ref| per element; the closed form
is first checked against the oracle, so the inputs really realise it.
Expected values are computed from the host inputs alone."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_245_gb300 as pkv
import workloads as W
from parity import DeviceLayer, assert_attention_close, shared_groups_batch

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")

FORMS = ["identical_keys", "zero_query", "zero_scale", "constant_v", "dominant_logit", "scale_2"]
MODES = ["auto", "split", "tc_8x3", "tc_12x2", "contig_split", "contig_tc", "shared_tc_pass",
         "shared_in_merge", "shared_own_tiles"]
HEADS = [(32, 8), (56, 8), (32, 4)]
VARIANT = {"auto": pkv.VARIANT_AUTO, "split": pkv.VARIANT_SPLIT, "tc_8x3": pkv.VARIANT_TC_8X3,
           "tc_12x2": pkv.VARIANT_TC_12X2, "contig_split": pkv.VARIANT_SPLIT,
           "contig_tc": pkv.VARIANT_TC_12X2, "shared_tc_pass": pkv.VARIANT_AUTO,
           "shared_in_merge": pkv.VARIANT_AUTO, "shared_own_tiles": pkv.VARIANT_AUTO}
# contexts from one position to many tiles; with a tensor-core variant forced
# the few tiles spread over every SM, so pairs are cut by many CTA ranges
CTX = [1, 2, 15, 16, 17, 100, 257, 700, 1500]


@pytest.fixture(autouse=True)
def _reset_modes():
    pkv.set_split_tiles(0)
    pkv.set_checked(False)
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    yield
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    torch.cuda.synchronize()


def _f64(u16):
    """bf16 bit patterns -> float64 values (exact)."""
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_bits(x):
    """float64 values -> nearest bf16 bit patterns."""
    return W.to_u16(torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16))


def _rows(h_cache, tables, i, g, ctx, bs):
    """Logical rows [ctx, D] of KV head g of sequence i, by numpy indexing."""
    j = np.arange(ctx)
    return _f64(h_cache[tables[i, j // bs], g, j % bs])


def _make_form(form, L, b, seed):
    """Rewrite the host mirrors of q / K / V for the form, push them to the
    device, and return (scale, closed-form output or None)."""
    rng = np.random.default_rng(seed)
    hq, hkv = b.shape.num_q_heads, b.shape.num_kv_heads
    G, bs = hq // hkv, b.block_size
    scale = W.default_scale(b.shape)
    if form == "identical_keys":
        L.h_k[:] = _bf16_bits(rng.standard_normal((hkv, 128)))[None, :, None, :]
    elif form == "constant_v":
        L.h_v[:] = _bf16_bits(rng.standard_normal((hkv, 128)))[None, :, None, :]
    elif form == "zero_query":
        L.h_q[:] = 0
    elif form == "zero_scale":
        scale = 0.0
    elif form == "scale_2":
        scale = 2.0
    elif form == "dominant_logit":
        for i in range(b.B):
            for h in range(hq):
                K = _rows(L.h_k, b.block_tables, i, h // G, int(b.ctx[i]), bs)
                j = (7 * i + 13 * h) % int(b.ctx[i])
                L.h_q[i, h] = _bf16_bits(100.0 * K[j] / np.linalg.norm(K[j]))
    L.q = W.from_u16(L.h_q, DEV)
    L.k_cache = W.from_u16(L.h_k, DEV)
    L.v_cache = W.from_u16(L.h_v, DEV)
    if form == "scale_2":
        return scale, None
    want = np.zeros((b.B, hq, 128))
    for i in range(b.B):
        c = int(b.ctx[i])
        for h in range(hq):
            V = _rows(L.h_v, b.block_tables, i, h // G, c, bs)
            if form == "dominant_logit":
                K = _rows(L.h_k, b.block_tables, i, h // G, c, bs)
                j = (7 * i + 13 * h) % c
                s = scale * (K @ _f64(L.h_q[i, h]))
                if c > 1:   # the form holds: the chosen logit leads by more than 30
                    assert s[j] - np.max(np.delete(s, j)) > 30.0
                want[i, h] = V[j]
            elif form == "constant_v":
                want[i, h] = V[0]
            else:
                want[i, h] = V.mean(axis=0)
    return scale, want


def _paged_batch(hq, hkv, seed):
    shape = W.ModelShape("cf%d_%d" % (hq, hkv), 1, hq, hkv)
    return W.make_paged_batch(shape, np.asarray(CTX, np.int32), 16, seed, spare_blocks=3), None


def _run(mode, L, b, starts, scale):
    pkv.set_decode_variant(VARIANT[mode])
    if mode.startswith("contig"):
        S = (b.max_context + 15) // 16 * 16
        kb = W.paged_to_contig(L.k_cache, b, S)
        vb = W.paged_to_contig(L.v_cache, b, S)
        req = torch.as_tensor(b.req_ids, device=DEV)
        out = pkv.contig_decode_attention(L.q, kb, vb, req, L.ctx, b.max_context, scale)
        ref = oracle.contig_decode(L.h_q, W.to_u16(kb), W.to_u16(vb), b.req_ids, b.ctx, scale)
        return out, ref
    ref = oracle.paged_decode(L.h_q, L.h_k, L.h_v, b.block_tables, b.ctx, scale)
    if mode.startswith("shared"):
        shared = W.shared_prefix_blocks(b.block_tables, b.ctx, b.block_size, starts)
        own = -1
        if mode in ("shared_in_merge", "shared_own_tiles"):
            per_seq = np.repeat(shared, np.diff(starts)) * b.block_size
            own = int((b.ctx - per_seq).max())
        out = pkv.paged_decode_attention_shared(
            L.q, L.k_cache, L.v_cache, L.tables, L.ctx, b.max_context, scale,
            torch.as_tensor(np.asarray(starts, np.int32), device=DEV),
            torch.as_tensor(shared, device=DEV), int(np.max(np.diff(starts))),
            max_own_tokens=own)
        return out, ref
    out = pkv.paged_decode_attention(L.q, L.k_cache, L.v_cache, L.tables, L.ctx, b.max_context,
                                     scale)
    return out, ref


@pytest.mark.parametrize("hq,hkv", HEADS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("form", FORMS)
def test_closed_form(form, mode, hq, hkv):
    seed = 1000 + 17 * FORMS.index(form) + hq + hkv
    if mode == "shared_own_tiles":
        # few own positions: they ride as masked key tiles of the prefix
        # kernel, which (one chunk per group here) writes the output itself
        b, starts = shared_groups_batch(hq, hkv, [1, 2, 3, 4], 40, seed, own_max=20,
                                        singleton_blocks=1)
    elif mode.startswith("shared"):
        # groups of 1..4 sequences over shared prompt blocks of up to 40 blocks
        b, starts = shared_groups_batch(hq, hkv, [1, 2, 3, 4], 40, seed)
    else:
        b, starts = _paged_batch(hq, hkv, seed)
    L = DeviceLayer(b, 0, DEV)
    scale, want = _make_form(form, L, b, seed)
    out, ref = _run(mode, L, b, starts, scale)
    torch.cuda.synchronize()
    what = "%s / %s / G=%d" % (form, mode, hq // hkv)
    if want is not None:
        # the inputs realise the closed form (the oracle agrees to ~1e-10)
        assert np.max(np.abs(ref - want)) <= 1e-9 * max(1.0, np.max(np.abs(want))), what
        assert_attention_close(out, want, what + " vs closed form")
    assert_attention_close(out, ref, what + " vs oracle")

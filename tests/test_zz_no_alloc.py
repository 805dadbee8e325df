"""The allocation-free decode entry point.

pkv_paged_decode_attention_noalloc serves callers that cannot allocate
device memory (an engine whose allocator owns all of the GPU's memory, or a
latency-critical caller that must not call cudaMalloc/cudaFree).  Its split
partials live in a fixed device array inside the library.  These tests call
it through the C ABI and check it against the regular entry point (which
takes a caller workspace) on two calls in a row, the second with different
inputs, so stale scratch from the first call cannot leak into the second.

This file is collected last on purpose: it must pass alone in a fresh
process and after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_245_gb300 as pkv
import workloads as W
from paged_kv_cache_245_gb300.binding import Heads
from paged_kv_cache_245_gb300.build import build
from parity import ATOL, RTOL

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SCRATCH_BYTES = 16 * 1024 * 1024   # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h


def _entry():
    build()
    L = pkv.lib()
    f = L.pkv_paged_decode_attention_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [vp, vp, vp, vp, i32, i32, vp, i32, i32, i32, ctypes.c_float, Heads, vp, vp]
    f.restype = ctypes.c_int
    return L, f


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call_noalloc(f, q, kc, vc, tables, ctx, max_context, bs, scale, out):
    hq, hkv = q.shape[1], kc.shape[1]
    return f(_ptr(q), _ptr(kc), _ptr(vc), _ptr(tables), tables.shape[1], kc.shape[0],
             _ptr(ctx), q.shape[0], int(max_context), bs, float(scale), Heads(hq, hkv, 128),
             _ptr(out), ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    L, f = _entry()
    pkv.set_split_tiles(0)
    pkv.set_checked(False)
    cases = [(W.LLAMA3_8B, W.ragged_lengths(48, seed=31, max_len=4096), 31),
             (W.YI_34B, W.ragged_lengths(24, seed=32, max_len=6000), 32)]
    for shape, ctx, seed in cases:
        b = W.make_paged_batch(shape, ctx, 16, seed)
        nsplit = pkv.decode_num_splits(b.B, shape.num_q_heads, shape.num_kv_heads,
                                       b.max_context)
        need = pkv.decode_workspace_size(b.B, shape.num_q_heads, shape.num_kv_heads,
                                         b.max_context)
        assert nsplit > 1 and 0 < need <= SCRATCH_BYTES  # the scratch is really used
        li = W.layer_inputs(b, 0, device=DEV, fast_cache=True)
        tables = torch.as_tensor(b.block_tables, device=DEV)
        ctx_d = torch.as_tensor(b.ctx, device=DEV)
        scale = W.default_scale(shape)
        ref = pkv.paged_decode_attention(li.q, li.k_cache, li.v_cache, tables, ctx_d,
                                         b.max_context, scale)
        out = torch.full_like(li.q, float("nan"))
        st = _call_noalloc(f, li.q, li.k_cache, li.v_cache, tables, ctx_d, b.max_context, 16,
                           scale, out)
        assert st == 0, L.pkv_last_error().decode()
        torch.cuda.synchronize()
        g = out.float().cpu().numpy().astype(np.float64)
        r = ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(g))
        assert np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r)), shape.name


def test_noalloc_rejects_batches_beyond_the_scratch():
    L, f = _entry()
    pkv.set_split_tiles(0)
    B, hq, hkv, max_ctx = 2048, 32, 8, 8192
    need = pkv.decode_workspace_size(B, hq, hkv, max_ctx)
    assert need > SCRATCH_BYTES
    # real buffers; every context is 0, so nothing would be read even if a
    # kernel ran, but the call must stop before launching anything
    q = torch.zeros((B, hq, 128), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((4, hkv, 16, 128), dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros((B, max_ctx // 16), dtype=torch.int32, device=DEV)
    ctx = torch.zeros(B, dtype=torch.int32, device=DEV)
    out = torch.full_like(q, 7.0)
    st = _call_noalloc(f, q, kc, kc, tables, ctx, max_ctx, 16, 0.1, out)
    torch.cuda.synchronize()
    assert st == 3
    assert b"fixed maximum" in L.pkv_last_error()
    assert torch.all(out == 7.0)   # nothing was launched

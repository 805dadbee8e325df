"""The allocation-free decode entry point.

pkv_paged_decode_attention_noalloc serves callers that cannot allocate
device memory (an engine whose allocator owns all of the GPU's memory, or a
latency-critical caller that must not call cudaMalloc/cudaFree).  Its split
partials live in a fixed device array inside the library.  These tests call
it through the C ABI and check it against the regular entry point (which
takes a caller workspace) and against the CPU oracle, on two calls in a
row, the second with different inputs, so stale scratch from the first call
cannot leak into the second.  Both decode kernels are covered: the
tensor-core kernel (its split records) and the CUDA-core split kernel (its
partials and combine).

This file is collected last on purpose: it must pass alone in a fresh
process and after every other test."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import paged_kv_cache_245_gb300 as pkv
import workloads as W
from paged_kv_cache_245_gb300.binding import Heads
from paged_kv_cache_245_gb300.build import build
from parity import ATOL, RTOL, DeviceLayer, assert_attention_close

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
SCRATCH_BYTES = 16 * 1024 * 1024   # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(autouse=True)
def _modes():
    pkv.set_split_tiles(0)
    pkv.set_checked(False)
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    yield
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    torch.cuda.synchronize()


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


CASES = [(W.LLAMA3_8B, 48, 4096, 31), (W.YI_34B, 24, 6000, 32)]


@pytest.mark.parametrize("variant", [pkv.VARIANT_AUTO, pkv.VARIANT_SPLIT])
def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls(variant):
    """Two calls in a row with different batches: each output equals the
    regular call's within the attention tolerance and matches the fp64
    oracle.  VARIANT_SPLIT forces the CUDA-core split kernel, whose partials
    (several splits per sequence here) go through the fixed array."""
    L, f = _entry()
    pkv.set_decode_variant(variant)
    for shape, B, max_len, seed in CASES:
        b = W.make_paged_batch(shape, W.ragged_lengths(B, seed=seed, max_len=max_len), 16, seed)
        need = pkv.decode_workspace_size(b.B, shape.num_q_heads, shape.num_kv_heads,
                                         b.max_context)
        assert 0 < need <= SCRATCH_BYTES
        if variant == pkv.VARIANT_SPLIT:   # the split kernel really writes partials
            assert pkv.decode_num_splits(b.B, shape.num_q_heads, shape.num_kv_heads,
                                         b.max_context) > 1
        Ld = DeviceLayer(b, 0, DEV, fast_cache=True)
        ref = Ld.gpu_attend()
        out = torch.full_like(Ld.q, float("nan"))
        st = _call_noalloc(f, Ld.q, Ld.k_cache, Ld.v_cache, Ld.tables, Ld.ctx, b.max_context, 16,
                           Ld.scale, out)
        assert st == 0, L.pkv_last_error().decode()
        torch.cuda.synchronize()
        g = out.float().cpu().numpy().astype(np.float64)
        r = ref.float().cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(g))
        assert np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r)), shape.name
        assert_attention_close(out, Ld.oracle_attend(), "noalloc %s vs oracle" % shape.name)


def test_noalloc_rejects_only_what_the_chosen_kernel_cannot_hold():
    """A batch of 2048 sequences x 8192 positions: the split kernel's
    partials would need far more than the fixed array, so forcing that
    kernel is rejected before any launch; the automatic choice (the
    tensor-core kernel, whose records fit) runs it."""
    L, f = _entry()
    B, hq, hkv, max_ctx = 2048, 32, 8, 8192
    # real buffers; every context is 0, so nothing would be read even if a
    # kernel ran
    q = torch.zeros((B, hq, 128), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((4, hkv, 16, 128), dtype=torch.bfloat16, device=DEV)
    tables = torch.zeros((B, max_ctx // 16), dtype=torch.int32, device=DEV)
    ctx = torch.zeros(B, dtype=torch.int32, device=DEV)
    pkv.set_decode_variant(pkv.VARIANT_SPLIT)
    out = torch.full_like(q, 7.0)
    st = _call_noalloc(f, q, kc, kc, tables, ctx, max_ctx, 16, 0.1, out)
    torch.cuda.synchronize()
    assert st == 3
    assert b"fixed maximum" in L.pkv_last_error()
    assert torch.all(out == 7.0)   # nothing was launched
    pkv.set_decode_variant(pkv.VARIANT_AUTO)
    st = _call_noalloc(f, q, kc, kc, tables, ctx, max_ctx, 16, 0.1, out)
    torch.cuda.synchronize()
    assert st == 0, L.pkv_last_error().decode()
    assert torch.count_nonzero(out) == 0   # empty contexts give zeros


_CHILD = r"""
import ctypes, sys, threading
import numpy as np, torch
sys.path.insert(0, ".")
sys.path.insert(0, "tests")
import paged_kv_cache_245_gb300 as pkv
import workloads as W
from paged_kv_cache_245_gb300.binding import Heads
from parity import ATOL, RTOL
dev = torch.device("cuda:0")
L = pkv.lib()
f = L.pkv_paged_decode_attention_noalloc
vp, i32 = ctypes.c_void_p, ctypes.c_int32
f.argtypes = [vp, vp, vp, vp, i32, i32, vp, i32, i32, i32, ctypes.c_float, Heads, vp, vp]
f.restype = ctypes.c_int
shape = W.LLAMA3_8B
b = W.make_paged_batch(shape, W.ragged_lengths(40, seed=5, max_len=3000), 16, 5)
li = W.layer_inputs(b, 0, device=dev, fast_cache=True)
tables = torch.as_tensor(b.block_tables, device=dev)
ctx = torch.as_tensor(b.ctx, device=dev)
scale = W.default_scale(shape)
ref = pkv.paged_decode_attention(li.q, li.k_cache, li.v_cache, tables, ctx, b.max_context, scale)
stream = torch.cuda.Stream(dev)      # one stream: the threads' kernels never overlap
torch.cuda.synchronize()
n = 8
outs = [torch.full_like(li.q, float("nan")) for _ in range(n)]
status = [None] * n
gate = threading.Barrier(n)
def run(t):
    gate.wait()   # every thread makes its first call at once
    status[t] = f(ctypes.c_void_p(li.q.data_ptr()), ctypes.c_void_p(li.k_cache.data_ptr()),
                  ctypes.c_void_p(li.v_cache.data_ptr()), ctypes.c_void_p(tables.data_ptr()),
                  tables.shape[1], li.k_cache.shape[0], ctypes.c_void_p(ctx.data_ptr()), b.B,
                  int(b.max_context), 16, float(scale), Heads(32, 8, 128),
                  ctypes.c_void_p(outs[t].data_ptr()), ctypes.c_void_p(stream.cuda_stream))
ths = [threading.Thread(target=run, args=(t,)) for t in range(n)]
for t in ths: t.start()
for t in ths: t.join()
torch.cuda.synchronize()
assert status == [0] * n, status
r = ref.float().cpu().numpy().astype(np.float64)
for o in outs:
    g = o.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(g)) and np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r))
print("ok", n)
"""


def test_noalloc_first_calls_from_many_threads_in_a_fresh_process():
    """In a fresh process, eight host threads make their first call at the
    same moment (the scratch address lookup runs under a lock); all calls
    go to one stream, and every output equals the regular call's."""
    build()
    r = subprocess.run([sys.executable, "-c", _CHILD], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok 8" in r.stdout

"""The C-ABI library loads on a machine without a GPU and exports every
symbol include/pkv.h declares; host-side validation rejects bad arguments
before any CUDA call.  No GPU."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_245_gb300 as pkv
from paged_kv_cache_245_gb300 import binding
from paged_kv_cache_245_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build()
    return pkv.lib()


def _declared():
    inc = os.path.join(ROOT, "include")
    text = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc))
                   if f.endswith(".h"))
    return set(re.findall(r"PKV_API[^;(]*?\b(pkv_\w+)\s*\(", text))


def test_header_declares_the_calls(L):
    names = _declared()
    for call in ("pkv_kv_append", "pkv_paged_decode_attention", "pkv_contig_decode_attention",
                 "pkv_block_copy", "pkv_decode_workspace_size", "pkv_get_device_error",
                 "pkv_paged_decode_step", "pkv_debug_gather_paged", "pkv_bm_create",
                 "pkv_bm_append"):
        assert call in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name
    assert set(binding.EXPORTED) <= _declared()


def _h(hq=8, hkv=2, d=128):
    return binding.Heads(hq, hkv, d)


FAKE = ctypes.c_void_p(0x10000)        # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x10008)


def test_status_strings(L):
    assert L.pkv_status_string(0) == b"ok"
    assert L.pkv_status_string(3).startswith(b"workspace")


def test_decode_rejects_bad_heads(L):
    st = L.pkv_paged_decode_attention(FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, 2, 64, 16, 0.1,
                                      _h(d=64), FAKE, None, 0, None)
    assert st == 2 and b"head_dim" in L.pkv_last_error()
    st = L.pkv_paged_decode_attention(FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, 2, 64, 16, 0.1,
                                      _h(32, 2), FAKE, None, 0, None)
    assert st == 2
    st = L.pkv_paged_decode_attention(FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, 2, 64, 16, 0.1,
                                      _h(9, 2), FAKE, None, 0, None)
    assert st == 1


def test_decode_rejects_null_and_misaligned(L):
    st = L.pkv_paged_decode_attention(None, FAKE, FAKE, FAKE, 4, 10, FAKE, 2, 64, 16, 0.1,
                                      _h(), FAKE, None, 0, None)
    assert st == 1
    st = L.pkv_paged_decode_attention(MISALIGNED, FAKE, FAKE, FAKE, 4, 10, FAKE, 2, 64, 16,
                                      0.1, _h(), FAKE, None, 0, None)
    assert st == 1 and b"aligned" in L.pkv_last_error()
    st = L.pkv_paged_decode_attention(FAKE, FAKE, FAKE, FAKE, 3, 10, FAKE, 2, 64, 16, 0.1,
                                      _h(), FAKE, None, 0, None)
    assert st == 1 and b"max_blocks" in L.pkv_last_error()
    st = L.pkv_paged_decode_attention(FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, 2, 64, 0, 0.1,
                                      _h(), FAKE, None, 0, None)
    assert st == 1
    st = L.pkv_paged_decode_attention(FAKE, FAKE, FAKE, FAKE, 4, 10, FAKE, 2, 64, 16,
                                      float("nan"), _h(), FAKE, None, 0, None)
    assert st == 1


def test_contig_rejects_context_beyond_S(L):
    st = L.pkv_contig_decode_attention(FAKE, FAKE, FAKE, FAKE, 4, FAKE, 2, 65, 64, 0.1, _h(),
                                       FAKE, None, 0, None)
    assert st == 1 and b"S" in L.pkv_last_error()


def test_empty_batch_is_a_no_op(L):
    st = L.pkv_paged_decode_attention(None, None, None, None, 0, 0, None, 0, 0, 16, 0.1, _h(),
                                      None, None, 0, None)
    assert st == 0
    assert L.pkv_kv_append(None, 0, None, None, None, None, 0, 16, _h(), None) == 0
    assert L.pkv_block_copy(None, 0, None, None, 3, 10, 1024, None) == 0


def test_append_and_copy_validation(L):
    assert L.pkv_kv_append(FAKE, 4, FAKE, FAKE, FAKE, FAKE, 100, 0, _h(), None) == 1
    assert L.pkv_kv_append(MISALIGNED, 4, FAKE, FAKE, FAKE, MISALIGNED, 100, 16, _h(), None) == 1
    assert L.pkv_kv_append(FAKE, 4, FAKE, FAKE, FAKE, FAKE, 100, 16, _h(d=256), None) == 2
    arr = (ctypes.c_void_p * 2)(0x10000, 0x10008)
    assert L.pkv_block_copy(FAKE, 2, arr, arr, 2, 10, 1024, None) == 1
    assert L.pkv_block_copy(FAKE, 2, arr, arr, 1, 10, 1000, None) == 1


def test_checked_flag_and_split_override_round_trip(L):
    pkv.set_checked(True)
    assert pkv.get_checked()
    pkv.set_checked(False)
    assert not pkv.get_checked()
    pkv.set_split_tiles(0)


def test_prefill_validation(L):
    # paged: (q, cu, T, k, v, tables, max_blocks, num_blocks, ctx, B, max_q, bs, scale, heads, out, stream)
    args = lambda **kw: dict(dict(q=FAKE, cu=FAKE, T=8, k=FAKE, v=FAKE, tab=FAKE, mb=4, nb=10,
                                  ctx=FAKE, B=2, mq=4, bs=16, sc=0.1, h=_h(), out=FAKE), **kw)

    def paged(**kw):
        a = args(**kw)
        return L.pkv_paged_prefill_attention(a["q"], a["cu"], a["T"], a["k"], a["v"], a["tab"],
                                             a["mb"], a["nb"], a["ctx"], a["B"], a["mq"], a["bs"],
                                             a["sc"], a["h"], a["out"], None)

    assert paged(h=_h(d=64)) == 2
    assert paged(q=None) == 1
    assert paged(out=MISALIGNED) == 1 and b"aligned" in L.pkv_last_error()
    assert paged(bs=8) == 2 and b"block_size" in L.pkv_last_error()
    assert paged(sc=float("inf")) == 1
    assert paged(mb=0) == 1
    assert paged(T=0) == 0 and paged(B=0) == 0  # nothing to attend
    # contiguous: (q, cu, T, k_buf, v_buf, req_ids, max_reqs, ctx, B, max_q, S, scale, heads, out, stream)
    assert L.pkv_contig_prefill_attention(FAKE, FAKE, 8, FAKE, FAKE, FAKE, 4, FAKE, 2, 4, 1000,
                                          0.1, _h(), FAKE, None) == 2  # S % 16 != 0
    assert L.pkv_contig_prefill_attention(FAKE, FAKE, 8, FAKE, FAKE, FAKE, 4, FAKE, 2, 4, 0,
                                          0.1, _h(), FAKE, None) == 2
    assert L.pkv_contig_prefill_attention(FAKE, FAKE, 8, MISALIGNED, FAKE, FAKE, 4, FAKE, 2, 4,
                                          1024, 0.1, _h(), FAKE, None) == 1


def test_block_swap_validation(L):
    one = (ctypes.c_void_p * 1)(FAKE)
    # (pairs, n, src_k, src_v, src_blocks, dst_k, dst_v, dst_blocks, layers, block_bytes, stream)
    assert L.pkv_block_swap(FAKE, -1, one, one, 4, one, one, 4, 1, 64, None) == 1
    assert L.pkv_block_swap(FAKE, 0, one, one, 4, one, one, 4, 1, 64, None) == 0  # no pairs
    assert L.pkv_block_swap(FAKE, 2, None, one, 4, one, one, 4, 1, 64, None) == 1
    assert L.pkv_block_swap(FAKE, 2, one, one, 4, one, one, 4, 1, 24, None) == 1
    assert b"multiple of 16" in L.pkv_last_error()
    assert L.pkv_block_swap(FAKE, 2, one, one, 0, one, one, 4, 1, 64, None) == 1
    assert L.pkv_block_swap(FAKE, 2, one, one, 4, one, one, 0, 1, 64, None) == 1

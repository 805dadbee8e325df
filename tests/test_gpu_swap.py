"""Block swap between the device cache and a pool in page-locked host memory
(pkv_block_swap), for pre-emption ("Running Out of Cache", closing paragraph:
an evicted request's cache is swapped out and brought back later), against
the oracle: bit-exact in every layer, pairs in device or pinned host memory,
pageable memory rejected on the host, ids outside a pool reported in checked
mode."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_245_gb300 as pkv
import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
HKV, BS, D = 8, 16, 128


@pytest.fixture(autouse=True)
def _reset_modes():
    pkv.set_checked(False)
    yield
    pkv.set_checked(False)
    torch.cuda.synchronize()


def _pools(g, layers, blocks, pinned):
    mk = lambda: torch.randn((blocks, HKV, BS, D), generator=g).to(torch.bfloat16)
    ks, vs = [mk() for _ in range(layers)], [mk() for _ in range(layers)]
    if pinned:
        return [t.pin_memory() for t in ks], [t.pin_memory() for t in vs]
    return [t.to(DEV) for t in ks], [t.to(DEV) for t in vs]


def _u16(ts):
    return [W.to_u16(t.cpu()).copy() for t in ts]


@pytest.mark.parametrize("pairs_on_host", [False, True])
def test_swap_out_and_back_is_bit_exact(pairs_on_host):
    g = torch.Generator().manual_seed(7)
    L, NB, NH = 3, 64, 20
    dk, dv = _pools(g, L, NB, pinned=False)
    hk, hv = _pools(g, L, NH, pinned=True)
    mdk, mdv, mhk, mhv = _u16(dk), _u16(dv), _u16(hk), _u16(hv)
    rng = np.random.default_rng(8)
    out = np.stack([rng.choice(NB, 12, replace=False), rng.choice(NH, 12, replace=False)], 1)
    back = np.stack([out[:, 1], rng.choice(NB, 12, replace=False)], 1)

    def pairs(p):
        t = torch.as_tensor(p.astype(np.int64))
        return t.pin_memory() if pairs_on_host else t.to(DEV)

    pkv.block_swap(pairs(out), dk, dv, hk, hv)
    torch.cuda.synchronize()
    oracle.block_swap(out, mdk, mdv, mhk, mhv)
    for l in range(L):
        assert np.array_equal(W.to_u16(hk[l]), mhk[l]) and np.array_equal(W.to_u16(hv[l]), mhv[l])
    for l in range(L):                    # the device blocks are reused meanwhile
        dk[l][out[:, 0]] = 0
        dv[l][out[:, 0]] = 0
        mdk[l][out[:, 0]] = 0
        mdv[l][out[:, 0]] = 0
    pkv.block_swap(pairs(back), hk, hv, dk, dv)
    torch.cuda.synchronize()
    oracle.block_swap(back, mhk, mhv, mdk, mdv)
    for l in range(L):
        assert np.array_equal(W.to_u16(dk[l].cpu()), mdk[l])
        assert np.array_equal(W.to_u16(dv[l].cpu()), mdv[l])


def test_pageable_host_memory_is_rejected():
    g = torch.Generator().manual_seed(9)
    dk, dv = _pools(g, 1, 8, pinned=False)
    hk = [torch.zeros((4, HKV, BS, D), dtype=torch.bfloat16)]      # not page-locked
    hv = [torch.zeros((4, HKV, BS, D), dtype=torch.bfloat16)]
    with pytest.raises(pkv.PkvError, match="page-locked"):
        pkv.block_swap(torch.tensor([[1, 2]], device=DEV), dk, dv, hk, hv)
    assert not hk[0].any()


def test_checked_mode_reports_an_id_outside_the_host_pool():
    pkv.set_checked(True)
    g = torch.Generator().manual_seed(10)
    dk, dv = _pools(g, 2, 8, pinned=False)
    hk, hv = _pools(g, 2, 4, pinned=True)
    before = [t.clone() for t in hk]
    assert pkv.get_device_error() == "none"
    pkv.block_swap(torch.tensor([[1, 4]], device=DEV), dk, dv, hk, hv)   # slot 4 of 4
    torch.cuda.synchronize()
    assert pkv.get_device_error() == "copy_pair"
    assert all(torch.equal(a, b) for a, b in zip(hk, before))


def test_many_pairs_and_layers_cross_the_launch_slices():
    # more pairs than one launch's grid takes (65535) and more layers than
    # one launch's parameters hold (64): 16-byte blocks keep the pools small
    rng = np.random.default_rng(11)
    nb, n = 140000, 70000
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:n], perm[n:]], 1).astype(np.int64)
    g = torch.Generator().manual_seed(12)
    k = torch.randn((nb, 8), generator=g).to(torch.bfloat16)
    v = torch.randn((nb, 8), generator=g).to(torch.bfloat16)
    # copy on write within one pool
    dk, dv = k.to(DEV), v.to(DEV)
    pkv.block_copy(torch.as_tensor(pairs, device=DEV), [dk], [dv])
    mk, mv = W.to_u16(k).copy(), W.to_u16(v).copy()
    oracle.block_copy(pairs, [mk], [mv])
    torch.cuda.synchronize()
    assert np.array_equal(W.to_u16(dk), mk) and np.array_equal(W.to_u16(dv), mv)
    # swap out to a page-locked pool, slots in order
    out = np.stack([perm[:n], np.arange(n)], 1).astype(np.int64)
    hk = torch.zeros((n, 8), dtype=torch.bfloat16).pin_memory()
    hv = torch.zeros((n, 8), dtype=torch.bfloat16).pin_memory()
    pkv.block_swap(torch.as_tensor(out, device=DEV), [dk], [dv], [hk], [hv])
    torch.cuda.synchronize()
    assert np.array_equal(W.to_u16(hk), mk[perm[:n]]) and np.array_equal(W.to_u16(hv), mv[perm[:n]])
    # 70 layers back in, one launch per 64 layers
    L = 70
    src_k = [torch.randn((6, 8), generator=g).to(torch.bfloat16).pin_memory() for _ in range(L)]
    src_v = [torch.randn((6, 8), generator=g).to(torch.bfloat16).pin_memory() for _ in range(L)]
    dst_k = [torch.zeros((10, 8), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    dst_v = [torch.zeros((10, 8), dtype=torch.bfloat16, device=DEV) for _ in range(L)]
    back = np.array([[5, 0], [0, 9], [3, 4]], np.int64)
    pkv.block_swap(torch.as_tensor(back, device=DEV), src_k, src_v, dst_k, dst_v)
    mdk = [np.zeros((10, 8), np.uint16) for _ in range(L)]
    mdv = [np.zeros((10, 8), np.uint16) for _ in range(L)]
    oracle.block_swap(back, _u16(src_k), _u16(src_v), mdk, mdv)
    torch.cuda.synchronize()
    for l in range(L):
        assert np.array_equal(W.to_u16(dst_k[l]), mdk[l]) and np.array_equal(W.to_u16(dst_v[l]), mdv[l])

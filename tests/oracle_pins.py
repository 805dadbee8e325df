"""Pins for the CPU oracle: checks against what the pages and mathematics fix,
never against a retyping of the oracle's own formula.

Each pin is a plain function of the oracle module (so the mutation test can
run the same pins against deliberately broken builds of the oracle).  They
raise AssertionError when the oracle is wrong.

  * closed forms of softmax attention: one position returns V; identical keys,
    a zero query or a zero scale return the mean of V; two positions give the
    logistic weights; constant V returns the constant; one dominant logit
    returns that position's V;
  * an independent library routine (torch fp64 softmax) on tiny inputs;
  * gather special cases that reduce to array reshapes (identity block
    table, request rows), plus invariance under relabelling physical blocks,
    plus contiguous == paged with bs = S and a one-entry table
    ("Leveraging Low-Level CUDA APIs for vAttention's Dynamic Memory",
    section 5.2.3; "Running Out of Cache", block tables);
  * GQA: repeating each KV head G times (plain MHA) gives the same result;
  * append then gather finds the new token at the last position; untouched
    bytes stay untouched; copy on write makes dst equal src; a swap out to
    another pool and back into new blocks gives the same logical rows;
  * causal prefill: torch fp64 attention with an explicit causal mask; a
    chunk of one token is the decode step; the last token of a chunk equals
    decode; a query ignores later positions and depends on its own.
"""
import math

import numpy as np
import torch

D = 128


def _bf16(x):
    """float array -> uint16 bf16 bits (round to nearest even via torch)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _val(u16):
    """uint16 bf16 bits -> float64 values (exact)."""
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def _rand_bf16(rng, shape, scale=1.0):
    return _bf16(rng.standard_normal(shape) * scale)


# ---------------------------------------------------------------- closed forms

def pin_single_position_returns_v(orc):
    rng = np.random.default_rng(1)
    for _ in range(5):
        q, K, V = _rand_bf16(rng, D), _rand_bf16(rng, (1, D)), _rand_bf16(rng, (1, D))
        o = orc.attend(q, K, V, 1 / math.sqrt(D))
        assert np.array_equal(o, _val(V[0])), "ctx=1 must return v_0 exactly"


def pin_identical_keys_give_mean(orc):
    rng = np.random.default_rng(2)
    k = _rand_bf16(rng, D)
    K = np.tile(k, (37, 1))
    V = _rand_bf16(rng, (37, D))
    q = _rand_bf16(rng, D, 3.0)
    o = orc.attend(q, K, V, 1 / math.sqrt(D))
    assert np.allclose(o, _val(V).mean(axis=0), rtol=0, atol=1e-12)


def pin_zero_query_or_scale_gives_mean(orc):
    rng = np.random.default_rng(3)
    K, V = _rand_bf16(rng, (23, D)), _rand_bf16(rng, (23, D))
    mean = _val(V).mean(axis=0)
    o = orc.attend(np.zeros(D, np.uint16), K, V, 0.7)
    assert np.allclose(o, mean, rtol=0, atol=1e-12)
    o = orc.attend(_rand_bf16(rng, D), K, V, 0.0)
    assert np.allclose(o, mean, rtol=0, atol=1e-12)


def pin_two_positions_logistic(orc):
    rng = np.random.default_rng(4)
    for trial in range(6):
        q, K, V = _rand_bf16(rng, D), _rand_bf16(rng, (2, D)), _rand_bf16(rng, (2, D))
        scale = [0.088, 0.5, 1.0, 0.01, 0.3, 2.0][trial]
        qv, Kv, Vv = _val(q), _val(K), _val(V)
        delta = scale * (math.fsum(qv * Kv[0]) - math.fsum(qv * Kv[1]))
        w0 = 1.0 / (1.0 + math.exp(-delta))   # logistic sigma(s0 - s1)
        w1 = 1.0 / (1.0 + math.exp(delta))
        expect = w0 * Vv[0] + w1 * Vv[1]
        o = orc.attend(q, K, V, scale)
        assert np.allclose(o, expect, rtol=1e-12, atol=1e-12)


def pin_constant_v(orc):
    rng = np.random.default_rng(5)
    K = _rand_bf16(rng, (50, D))
    row = _rand_bf16(rng, D)
    V = np.tile(row, (50, 1))
    o = orc.attend(_rand_bf16(rng, D), K, V, 1 / math.sqrt(D))
    assert np.allclose(o, _val(row), rtol=1e-14, atol=1e-14)


def pin_dominant_logit(orc):
    rng = np.random.default_rng(6)
    ctx = 100
    K = np.zeros((ctx, D), np.float64)
    for j in range(ctx):
        K[j, j % D] = 1.0
    V = _rand_bf16(rng, (ctx, D))
    for star in (0, 41, 99):
        q = np.zeros(D)
        q[star % D] = 1000.0
        o = orc.attend(_bf16(q), _bf16(K), V, 1 / math.sqrt(D))
        assert np.allclose(o, _val(V[star]), rtol=1e-12, atol=1e-12)


def pin_empty_context_gives_zeros(orc):
    o = orc.attend(np.ones(D, np.uint16), np.zeros((0, D), np.uint16),
                   np.zeros((0, D), np.uint16), 1.0)
    assert np.array_equal(o, np.zeros(D))


def pin_library_softmax(orc):
    """torch fp64 softmax(q K^T * scale) V on random tiny inputs."""
    rng = np.random.default_rng(7)
    for ctx in (1, 2, 3, 17, 64, 130):
        q, K, V = _rand_bf16(rng, D, 2.0), _rand_bf16(rng, (ctx, D)), _rand_bf16(rng, (ctx, D))
        scale = 1 / math.sqrt(D)
        qt, Kt, Vt = (torch.from_numpy(_val(a)) for a in (q, K, V))
        ref = (torch.softmax((Kt @ qt) * scale, dim=0) @ Vt).numpy()
        o = orc.attend(q, K, V, scale)
        assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------- gathers

def _pool(rng, nb, hkv, bs):
    return _rand_bf16(rng, (nb, hkv, bs, D))


def pin_identity_table_is_reshape(orc):
    """With block table [0, 1, 2, ...] the logical rows of KV head h are the
    pool's head-h rows read in order (a reshape)."""
    rng = np.random.default_rng(8)
    for bs in (1, 5, 16):
        nb, hkv = 9, 3
        cache = _pool(rng, nb, hkv, bs)
        table = np.arange(nb, dtype=np.int32)
        for ctx in (1, bs, nb * bs - 2, nb * bs):
            for h in range(hkv):
                got = orc.gather_paged(cache, table, ctx, bs, h)
                assert np.array_equal(got, cache[:, h].reshape(-1, D)[:ctx])


def pin_request_rows_are_subtensors(orc):
    rng = np.random.default_rng(9)
    buf = _rand_bf16(rng, (4, 2, 33, D))
    for r in range(4):
        for h in range(2):
            got = orc.gather_contig(buf, r, 20, h)
            assert np.array_equal(got, buf[r, h, :20])


def pin_block_relabel_invariance(orc):
    """Relabelling physical blocks (moving storage and table together) leaves
    the decode output bit-identical."""
    rng = np.random.default_rng(10)
    hq, hkv, bs, nb = 8, 2, 16, 40
    ctx = np.array([1, 16, 17, 100, 33], np.int32)
    need = (ctx + bs - 1) // bs
    table = np.zeros((len(ctx), need.max()), np.int32)
    ids = rng.permutation(nb)
    pos = 0
    for i, n in enumerate(need):
        table[i, :n] = ids[pos:pos + n]
        pos += n
    kc, vc = _pool(rng, nb, hkv, bs), _pool(rng, nb, hkv, bs)
    q = _rand_bf16(rng, (len(ctx), hq, D))
    base = orc.paged_decode(q, kc, vc, table, ctx, 1 / math.sqrt(D))
    perm = rng.permutation(nb)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    out = orc.paged_decode(q, kc2, vc2, perm[table].astype(np.int32), ctx,
                           1 / math.sqrt(D))
    assert np.array_equal(out, base)
    # and the output really depends on the table (guards a table-blind oracle)
    shuffled = table.copy()
    shuffled[3, :2] = shuffled[3, [1, 0]]
    other = orc.paged_decode(q, kc, vc, shuffled, ctx, 1 / math.sqrt(D))
    assert not np.array_equal(other[3], base[3])


def pin_contig_equals_paged_with_bs_S(orc):
    """[max_reqs, Hkv, S, D] read at reqId x S is the paged pool with bs = S
    and the one-entry table [reqId]."""
    rng = np.random.default_rng(11)
    max_reqs, hkv, hq, S = 6, 2, 8, 48
    kb, vb = _rand_bf16(rng, (max_reqs, hkv, S, D)), _rand_bf16(rng, (max_reqs, hkv, S, D))
    req = np.array([4, 0, 5, 2], np.int32)
    ctx = np.array([48, 1, 30, 0], np.int32)
    q = _rand_bf16(rng, (4, hq, D))
    a = orc.contig_decode(q, kb, vb, req, ctx, 0.1)
    b = orc.paged_decode(q, kb, vb, req.reshape(-1, 1), ctx, 0.1)
    assert np.array_equal(a, b)
    assert np.array_equal(a[3], np.zeros((hq, D)))


def pin_paged_equals_logical_attend(orc):
    """Paged decode of one (sequence, head) equals attention over the rows the
    identity-table reshape exposes (brute force on a contiguous copy)."""
    rng = np.random.default_rng(12)
    nb, hkv, hq, bs = 7, 1, 3, 4
    kc, vc = _pool(rng, nb, hkv, bs), _pool(rng, nb, hkv, bs)
    table = np.arange(nb, dtype=np.int32).reshape(1, -1)
    ctx = np.array([25], np.int32)
    q = _rand_bf16(rng, (1, hq, D))
    out = orc.paged_decode(q, kc, vc, table, ctx, 0.2)
    Kl, Vl = kc[:, 0].reshape(-1, D)[:25], vc[:, 0].reshape(-1, D)[:25]
    for h in range(hq):
        assert np.array_equal(out[0, h], orc.attend(q[0, h], Kl, Vl, 0.2))


def pin_gqa_equals_repeated_mha(orc):
    rng = np.random.default_rng(13)
    hkv, G, bs, nb = 3, 4, 8, 30
    hq = hkv * G
    ctx = np.array([9, 40, 1], np.int32)
    table = rng.permutation(nb)[:15].reshape(3, 5).astype(np.int32)
    kc, vc = _pool(rng, nb, hkv, bs), _pool(rng, nb, hkv, bs)
    q = _rand_bf16(rng, (3, hq, D))
    gqa = orc.paged_decode(q, kc, vc, table, ctx, 0.09)
    kr = np.ascontiguousarray(np.repeat(kc, G, axis=1))  # head h -> h // G
    vr = np.ascontiguousarray(np.repeat(vc, G, axis=1))
    mha = orc.paged_decode(q, kr, vr, table, ctx, 0.09)
    assert np.array_equal(gqa, mha)


def pin_threads_do_not_change_results(orc):
    rng = np.random.default_rng(14)
    kc, vc = _pool(rng, 20, 2, 16), _pool(rng, 20, 2, 16)
    table = rng.permutation(20)[:12].reshape(3, 4).astype(np.int32)
    ctx = np.array([64, 3, 50], np.int32)
    q = _rand_bf16(rng, (3, 8, D))
    a = orc.paged_decode(q, kc, vc, table, ctx, 0.1, nthreads=1)
    b = orc.paged_decode(q, kc, vc, table, ctx, 0.1, nthreads=7)
    assert np.array_equal(a, b)


# ------------------------------------------------------------ append and copy

def pin_append_then_gather(orc):
    """Observation-1: each step adds exactly one token.  After appending at the
    slot of position ctx-1, the gather through the block table returns the new
    row last, every earlier row unchanged, and no other byte of the pool moved."""
    rng = np.random.default_rng(15)
    hkv, bs, nb = 2, 16, 24
    kc, vc = _pool(rng, nb, hkv, bs), _pool(rng, nb, hkv, bs)
    table = rng.permutation(nb)[:12].reshape(3, 4).astype(np.int32)
    ctx_pre = np.array([0, 16, 40], np.int64)
    slots = np.array([table[i, p // bs] * bs + p % bs for i, p in enumerate(ctx_pre)],
                     np.int64)
    k_new, v_new = _rand_bf16(rng, (3, hkv, D)), _rand_bf16(rng, (3, hkv, D))
    before_k = [[orc.gather_paged(kc, table[i], int(ctx_pre[i]), bs, h)
                 for h in range(hkv)] for i in range(3)]
    k0, v0 = kc.copy(), vc.copy()
    orc.kv_append(slots, k_new, v_new, kc, vc)
    for i in range(3):
        c = int(ctx_pre[i]) + 1
        for h in range(hkv):
            gk = orc.gather_paged(kc, table[i], c, bs, h)
            gv = orc.gather_paged(vc, table[i], c, bs, h)
            assert np.array_equal(gk[-1], k_new[i, h])
            assert np.array_equal(gv[-1], v_new[i, h])
            assert np.array_equal(gk[:-1], before_k[i][h])
    changed = np.count_nonzero(kc != k0) + np.count_nonzero(vc != v0)
    assert changed <= 2 * 3 * hkv * D
    # a padding slot (-1) writes nothing
    k1 = kc.copy()
    orc.kv_append(np.array([-1], np.int64), k_new[:1], v_new[:1], kc, vc)
    assert np.array_equal(kc, k1)


def pin_append_contig_positions(orc):
    """In the contiguous layout slot reqId*S + pos puts the row at position pos
    of request reqId's sub-tensor."""
    rng = np.random.default_rng(16)
    S, hkv = 12, 2
    kb, vb = _rand_bf16(rng, (3, hkv, S, D)), _rand_bf16(rng, (3, hkv, S, D))
    k_new, v_new = _rand_bf16(rng, (2, hkv, D)), _rand_bf16(rng, (2, hkv, D))
    orc.kv_append(np.array([2 * S + 7, 0 * S + 11], np.int64), k_new, v_new, kb, vb)
    for h in range(hkv):
        assert np.array_equal(orc.gather_contig(kb, 2, 8, h)[7], k_new[0, h])
        assert np.array_equal(orc.gather_contig(vb, 0, 12, h)[11], v_new[1, h])


def pin_block_copy(orc):
    rng = np.random.default_rng(17)
    L, nb, hkv, bs = 3, 10, 2, 4
    ks = [_pool(rng, nb, hkv, bs) for _ in range(L)]
    vs = [_pool(rng, nb, hkv, bs) for _ in range(L)]
    k0, v0 = [a.copy() for a in ks], [a.copy() for a in vs]
    pairs = np.array([[3, 7], [0, 9], [5, 2]], np.int64)
    orc.block_copy(pairs, ks, vs)
    for l in range(L):
        for src, dst in pairs:
            assert np.array_equal(ks[l][dst], k0[l][src])
            assert np.array_equal(vs[l][dst], v0[l][src])
        untouched = [b for b in range(nb) if b not in pairs[:, 1]]
        assert np.array_equal(ks[l][untouched], k0[l][untouched])
        assert np.array_equal(vs[l][untouched], v0[l][untouched])


def pin_block_swap(orc):
    # out of a device-like pool into a host-like pool of another size, then
    # back into new blocks: the sequence read through its new table is the
    # one it was; blocks no pair names are untouched
    rng = np.random.default_rng(19)
    L, nb, nh, hkv, bs = 2, 9, 5, 2, 4
    dk = [_pool(rng, nb, hkv, bs) for _ in range(L)]
    dv = [_pool(rng, nb, hkv, bs) for _ in range(L)]
    hk = [_pool(rng, nh, hkv, bs) for _ in range(L)]
    hv = [_pool(rng, nh, hkv, bs) for _ in range(L)]
    table = np.array([6, 1, 4], np.int32)
    before = [orc.gather_paged(dk[l], table, 11, bs, h) for l in range(L) for h in range(hkv)]
    h0 = [a.copy() for a in hk]
    out = np.array([[6, 3], [1, 0], [4, 4]], np.int64)
    orc.block_swap(out, dk, dv, hk, hv)
    for l in range(L):
        assert np.array_equal(hk[l][[1, 2]], h0[l][[1, 2]])
        assert np.array_equal(hk[l][3], dk[l][6]) and np.array_equal(hv[l][0], dv[l][1])
    for l in range(L):                                  # the device blocks are reused
        dk[l][[6, 1, 4]] = 0
        dv[l][[6, 1, 4]] = 0
    new_table = np.array([2, 8, 0], np.int32)
    orc.block_swap(np.array([[3, 2], [0, 8], [4, 0]], np.int64), hk, hv, dk, dv)
    after = [orc.gather_paged(dk[l], new_table, 11, bs, h) for l in range(L) for h in range(hkv)]
    for a, b in zip(before, after):
        assert np.array_equal(a, b)
    # within one pool it is the copy on write
    ks = [_pool(rng, nb, hkv, bs) for _ in range(L)]
    vs = [_pool(rng, nb, hkv, bs) for _ in range(L)]
    ks2, vs2 = [a.copy() for a in ks], [a.copy() for a in vs]
    pairs = np.array([[3, 7], [0, 5]], np.int64)
    orc.block_swap(pairs, ks, vs, ks, vs)
    orc.block_copy(pairs, ks2, vs2)
    for l in range(L):
        assert np.array_equal(ks[l], ks2[l]) and np.array_equal(vs[l], vs2[l])


# --------------------------------------------------------------------- prefill

def _prefill_case(rng, ctx, lq, hq=8, hkv=2, bs=16, nb=None):
    """A paged batch whose sequence i's last lq[i] positions are new tokens."""
    ctx = np.asarray(ctx, np.int32)
    need = (ctx + bs - 1) // bs
    nb = nb or int(need.sum()) + 3
    table = np.zeros((len(ctx), need.max()), np.int32)
    ids = rng.permutation(nb)
    pos = 0
    for i, n in enumerate(need):
        table[i, :n] = ids[pos:pos + n]
        pos += n
    kc, vc = _pool(rng, nb, hkv, bs), _pool(rng, nb, hkv, bs)
    cu = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    q = _rand_bf16(rng, (int(cu[-1]), hq, D))
    return ctx, cu, table, kc, vc, q


def pin_prefill_library_causal(orc):
    """torch fp64 causal attention (explicit mask) on one sequence laid out
    with an identity table: new token j at position ctx - lq + j sees
    positions 0 .. ctx - lq + j."""
    rng = np.random.default_rng(21)
    bs, hkv, hq = 16, 2, 4
    for ctx, lq in ((1, 1), (5, 5), (40, 7), (70, 33)):
        nb = (ctx + bs - 1) // bs
        table = np.arange(nb, dtype=np.int32)[None, :]
        kc, vc = _pool(rng, nb, hkv, bs), _pool(rng, nb, hkv, bs)
        q = _rand_bf16(rng, (lq, hq, D))
        scale = 1 / math.sqrt(D)
        out = orc.paged_prefill(q, kc, vc, table, np.array([ctx], np.int32),
                                np.array([0, lq], np.int32), scale)
        K = torch.from_numpy(_val(kc)).permute(1, 0, 2, 3).reshape(hkv, nb * bs, D)[:, :ctx]
        V = torch.from_numpy(_val(vc)).permute(1, 0, 2, 3).reshape(hkv, nb * bs, D)[:, :ctx]
        Q = torch.from_numpy(_val(q))                     # [lq, hq, D]
        posn = torch.arange(ctx - lq, ctx)[:, None]       # query positions
        mask = torch.arange(ctx)[None, :] > posn          # [lq, ctx]
        for h in range(hq):
            s = (Q[:, h] @ K[h // (hq // hkv)].T) * scale
            s = s.masked_fill(mask, float("-inf"))
            ref = torch.softmax(s, dim=1) @ V[h // (hq // hkv)]
            assert np.allclose(out[:, h], ref.numpy(), rtol=1e-12, atol=1e-12)


def pin_prefill_chunk_of_one_is_decode(orc):
    """A chunk of one new token per sequence is the decode step."""
    rng = np.random.default_rng(22)
    ctx, cu, table, kc, vc, q = _prefill_case(rng, [1, 16, 17, 100, 33], [1] * 5)
    scale = 1 / math.sqrt(D)
    a = orc.paged_prefill(q, kc, vc, table, ctx, cu, scale)
    b = orc.paged_decode(q, kc, vc, table, ctx, scale)
    assert np.array_equal(a, b)


def pin_prefill_last_token_is_decode(orc):
    """The last new token of each chunk attends the whole context, exactly
    as the decode step with that context does."""
    rng = np.random.default_rng(23)
    lq = [3, 16, 1, 40]
    ctx, cu, table, kc, vc, q = _prefill_case(rng, [3, 50, 17, 120], lq)
    scale = 1 / math.sqrt(D)
    a = orc.paged_prefill(q, kc, vc, table, ctx, cu, scale)
    last = cu[1:] - 1
    b = orc.paged_decode(q[last], kc, vc, table, ctx, scale)
    assert np.array_equal(a[last], b)


def pin_prefill_is_causal(orc):
    """A query's output ignores every later position and depends on its own."""
    rng = np.random.default_rng(24)
    ctx, cu, table, kc, vc, q = _prefill_case(rng, [48], [20], hq=2, hkv=1)
    scale = 1 / math.sqrt(D)
    base = orc.paged_prefill(q, kc, vc, table, ctx, cu, scale)
    bs = kc.shape[2]
    j = 9                                   # query at position 48 - 20 + 9 = 37
    p = 48 - 20 + j
    later_k, later_v = kc.copy(), vc.copy()
    for pos in range(p + 1, 48):            # change every later position
        blk, off = table[0, pos // bs], pos % bs
        later_k[blk, :, off] = _rand_bf16(rng, (kc.shape[1], D))
        later_v[blk, :, off] = _rand_bf16(rng, (kc.shape[1], D))
    out = orc.paged_prefill(q, later_k, later_v, table, ctx, cu, scale)
    assert np.array_equal(out[:j + 1], base[:j + 1])
    assert not np.array_equal(out[-1], base[-1])
    own_v = vc.copy()
    own_v[table[0, p // bs], :, p % bs] = _rand_bf16(rng, (kc.shape[1], D))
    out2 = orc.paged_prefill(q, kc, own_v, table, ctx, cu, scale)
    assert not np.array_equal(out2[j], base[j])
    assert np.array_equal(out2[:j], base[:j])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

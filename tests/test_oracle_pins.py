"""Pins for the CPU oracle, independent of the oracle's own formulas.

Each check ties an oracle function to something the pages or mathematics fix:
a procedural re-construction of the interleaved layout ("Decode Context
Parallel (DCP)", section "KV-cache layout"), closed forms, library routines
(scipy's logsumexp / softmax), special cases with textbook answers
(dcp_size = 1 is ordinary paged attention; interleave 1 is token round-robin;
interleave = block_size is page-cyclic ownership as on the TokenSpeed page,
section "Cache ownership"), and the exactness of the LSE merge that the
"Backend structure" and "Decode" sections rely on.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

LAYOUTS = [(dcp, bs, I) for dcp in (1, 2, 3, 4, 8) for bs in (1, 2, 4, 16, 64)
           for I in (1, 2, 4, 16, 64) if bs % I == 0]


def deal_tokens(L, dcp, bs, I):
    """Procedural placement: inside each run of bs*dcp tokens, consecutive
    groups of I tokens are dealt to ranks 0, 1, ..., dcp-1, 0, 1, ...; every
    rank appends the tokens it receives to its own local sequence."""
    local = [[] for _ in range(dcp)]
    x = 0
    while x < L:
        for g in range(bs * dcp // I):
            for _ in range(I):
                if x < L:
                    local[g % dcp].append(x)
                    x += 1
    return local


@pytest.mark.parametrize("dcp,bs,I", LAYOUTS)
def test_layout_matches_dealing(dcp, bs, I):
    L = 4 * bs * dcp + 3
    local = deal_tokens(L, dcp, bs, I)
    for r in range(dcp):
        for p, x in enumerate(local[r]):
            assert O.target_rank(x, bs, dcp, I) == r
            assert O.local_position(x, bs, dcp, I) == p
            assert O.global_token(p, r, bs, dcp, I) == x
    # each rank receives exactly bs tokens per full virtual block
    full = L // (bs * dcp)
    for r in range(dcp):
        assert sum(1 for x in local[r] if x < full * bs * dcp) == full * bs


@pytest.mark.parametrize("dcp,bs,I", LAYOUTS)
def test_local_seq_lens_closed_form_and_sum(dcp, bs, I):
    for L in [0, 1, I, bs, bs * dcp - 1, bs * dcp, bs * dcp + 1, 3 * bs * dcp + I + 1, 977]:
        enum = O.local_seq_lens([L], dcp, bs, I)[0]
        assert enum.sum() == L
        for r in range(dcp):
            assert O.local_seq_len_closed_form(L, r, dcp, bs, I) == enum[r]
        assert list(enum) == [len(v) for v in deal_tokens(L, dcp, bs, I)]


def test_layout_golden_table():
    rows = np.loadtxt(os.path.join(GOLDEN, "layout_dcp2_bs4_i2.txt"), dtype=np.int64)
    for x, vb, off, lbi, r, loc, p in rows:
        assert O.virtual_block_index(x, 4, 2) == vb
        assert O.offset_in_virtual_block(x, 4, 2) == off
        assert O.local_block_index(x, 4, 2, 2) == lbi
        assert O.target_rank(x, 4, 2, 2) == r
        assert O.local_offset(x, 4, 2, 2) == loc
        assert O.local_position(x, 4, 2, 2) == p


def test_special_cases():
    x = np.arange(5000)
    for dcp in (1, 2, 3, 8):
        # interleave 1: token round-robin
        assert (O.target_rank(x, 16, dcp, 1) == x % dcp).all()
        assert (O.local_position(x, 16, dcp, 1) == x // dcp).all()
        # interleave == block_size: whole pages cycle over the ranks
        assert (O.target_rank(x, 64, dcp, 64) == (x // 64) % dcp).all()
        assert (O.local_position(x, 64, dcp, 64) == (x // (64 * dcp)) * 64 + x % 64).all()
    # dcp 1: textbook paged attention, slot = BT[x // bs] * bs + x % bs
    rng = np.random.default_rng(0)
    bt = rng.permutation(40).astype(np.int32).reshape(1, 1, 40)
    pos = np.arange(40 * 16)
    rank, slot = O.slot_mapping(np.zeros_like(pos), pos, bt, None, 1, 16, 4, 40)
    assert (rank == 0).all()
    assert (slot[0] == bt[0, 0, pos // 16] * 16 + pos % 16).all()


def test_layout_constraint():
    with pytest.raises(ValueError):
        O.check_layout(2, 16, 3)
    with pytest.raises(ValueError):
        O.check_layout(0, 16, 1)
    O.check_layout(2, 16, 8)


@pytest.mark.parametrize("dcp,bs,I", [(2, 4, 2), (3, 16, 4), (8, 16, 1), (8, 64, 64), (4, 8, 8)])
def test_slot_mapping_ownership(dcp, bs, I):
    import workloads as W
    lens = np.array([1, bs * dcp, 3 * bs * dcp + 5, 101])
    bt, nb = W.make_block_tables(lens, dcp, bs, "random", seed=3)
    req = np.concatenate([np.full(L, b) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    rank, slot = O.slot_mapping(req, pos, bt, lens, dcp, bs, I, nb)
    # every token lands on exactly one rank, and only that rank has a slot
    assert (rank >= 0).all()
    assert ((slot >= 0).sum(axis=0) == 1).all()
    assert (slot[rank, np.arange(len(req))] >= 0).all()
    # (rank, slot) pairs are unique and inside the pool
    pairs = set()
    for t in range(len(req)):
        s = int(slot[rank[t], t])
        assert 0 <= s < nb * bs
        pairs.add((int(rank[t]), s))
    assert len(pairs) == len(req)
    # a rank's tokens of one request fill its blocks in local-position order
    for b, L in enumerate(lens):
        for r in range(dcp):
            toks = [x for x in range(L) if O.target_rank(x, bs, dcp, I) == r]
            for p, x in enumerate(toks):
                t = int(np.nonzero((req == b) & (pos == x))[0][0])
                assert slot[r, t] == bt[r, b, p // bs] * bs + p % bs
    # invalid inputs are masked
    rk, sl = O.slot_mapping([0, 9, 0], [-1, 0, 10 ** 9], bt, lens, dcp, bs, I, nb)
    assert (rk == -1).all() and (sl == -1).all()


def test_build_caches_writes_owner_only():
    rows = np.arange(12, dtype=np.int64).reshape(6, 2) + 100
    slot = np.array([[0, -1, 3, -1, 5, -1], [-1, 1, -1, 2, -1, 7]])
    c = O.build_caches(rows, slot, 2, 2, 4, -7)
    for t in range(6):
        r = 0 if slot[0, t] >= 0 else 1
        assert (c[r, slot[r, t]] == rows[t]).all()
    assert (c == -7).all(axis=2).sum() == 2 * 8 - 6


# ---------------------------------------------------------------------------
# attention and merge
# ---------------------------------------------------------------------------

def rnd(rng, *shape):
    return rng.standard_normal(shape)


def test_attention_against_library_routines():
    rng = np.random.default_rng(1)
    for n, dk, dv in [(1, 4, 4), (7, 5, 3), (300, 64, 64), (33, 576, 512)]:
        q, K, V = rnd(rng, dk), rnd(rng, n, dk), rnd(rng, n, dv)
        scale = 0.37
        o, lse = O.attention(q, K, V, scale)
        s = scale * np.einsum("d,nd->n", q, K)
        assert lse == pytest.approx(scipy.special.logsumexp(s), rel=1e-13, abs=1e-13)
        w = scipy.special.softmax(s)
        np.testing.assert_allclose(o, np.einsum("n,nv->v", w, V), rtol=1e-12, atol=1e-13)


def test_attention_closed_forms():
    rng = np.random.default_rng(2)
    q, k, v = rnd(rng, 8), rnd(rng, 8), rnd(rng, 6)
    # one key: o = v, lse = scale * q.k
    o, lse = O.attention(q, k[None], v[None], 0.5)
    np.testing.assert_allclose(o, v, rtol=1e-14)
    assert lse == pytest.approx(0.5 * float(np.dot(q, k)), rel=1e-14)
    # n identical keys: o = mean(v), lse = s + ln n
    V = rnd(rng, 9, 6)
    o, lse = O.attention(q, np.tile(k, (9, 1)), V, 0.5)
    np.testing.assert_allclose(o, V.mean(axis=0), rtol=1e-12)
    assert lse == pytest.approx(0.5 * float(np.dot(q, k)) + math.log(9), rel=1e-13)
    # two keys: weights are a logistic function of the score difference
    K2 = np.stack([k, -k])
    s1 = 0.25 * float(np.dot(q, k))
    o, lse = O.attention(q, K2, V[:2], 0.25)
    w1 = 1.0 / (1.0 + math.exp(-2 * s1))
    np.testing.assert_allclose(o, w1 * V[0] + (1 - w1) * V[1], rtol=1e-12)
    assert lse == pytest.approx(s1 + math.log1p(math.exp(-2 * s1)), rel=1e-13)
    # empty
    o, lse = O.attention(q, np.zeros((0, 8)), np.zeros((0, 6)), 1.0)
    assert lse == -math.inf and (o == 0).all()


@pytest.mark.parametrize("dcp,bs,I", [(1, 16, 1), (2, 16, 1), (2, 4, 2), (8, 16, 1), (8, 64, 64),
                                      (3, 8, 4)])
def test_sharded_merge_equals_unsharded(dcp, bs, I):
    rng = np.random.default_rng(dcp * 100 + bs + I)
    for L in [1, 2, dcp, bs * dcp, bs * dcp + 1, 777]:
        q, K, V = rnd(rng, 32), rnd(rng, L, 32), rnd(rng, L, 24)
        o_ref, lse_ref = O.attention(q, K, V, 0.2)
        o, lse, po, pl = O.sharded_attention(q, K, V, 0.2, L, dcp, bs, I)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
        assert lse == pytest.approx(lse_ref, rel=1e-13)
        for r in range(dcp):
            if O.local_seq_len_closed_form(L, r, dcp, bs, I) == 0:
                assert pl[r] == -math.inf and (po[r] == 0).all()


def test_sink_is_one_extra_zero_value_key():
    rng = np.random.default_rng(5)
    q, K, V = rnd(rng, 16), rnd(rng, 50, 16), rnd(rng, 50, 8)
    scale, sigma = 0.3, 1.7
    o, lse, _, _ = O.sharded_attention(q, K, V, scale, 50, 4, 4, 2, sink=sigma)
    k_star = q * sigma / (scale * float(np.dot(q, q)))
    o2, lse2 = O.attention(q, np.vstack([K, k_star]), np.vstack([V, np.zeros(8)]), scale)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-14)
    assert lse == pytest.approx(lse2, rel=1e-13)
    # one key with a sink: o = v e^s / (e^s + e^sigma)
    s = scale * float(np.dot(q, K[0]))
    o, lse = O.lse_merge(V[:1], [s], sink=sigma)
    np.testing.assert_allclose(o, V[0] * math.exp(s) / (math.exp(s) + math.exp(sigma)), rtol=1e-13)
    assert lse == pytest.approx(math.log(math.exp(s) + math.exp(sigma)), rel=1e-14)
    # sink -> -inf is no sink
    oa, la = O.lse_merge(V[:3], [0.1, -2.0, 0.5], sink=-math.inf)
    ob, lb = O.lse_merge(V[:3], [0.1, -2.0, 0.5])
    np.testing.assert_allclose(oa, ob, rtol=0, atol=0)
    assert la == lb


def test_merge_edge_cases_and_associativity():
    rng = np.random.default_rng(6)
    P = rnd(rng, 5, 7)
    lses = rnd(rng, 5) * 3
    o, lse = O.lse_merge(P, lses)
    oa, la = O.lse_merge(P[:2], lses[:2])
    ob, lb = O.lse_merge(P[2:], lses[2:])
    o2, l2 = O.lse_merge(np.stack([oa, ob]), [la, lb])
    np.testing.assert_allclose(o, o2, rtol=1e-13)
    assert lse == pytest.approx(l2, rel=1e-14)
    assert lse == pytest.approx(scipy.special.logsumexp(lses), rel=1e-14)
    # empty parts are ignored
    o3, l3 = O.lse_merge(np.vstack([P, np.zeros(7)]), list(lses) + [-math.inf])
    np.testing.assert_allclose(o3, o, rtol=1e-14)
    # nothing at all
    o4, l4 = O.lse_merge(np.zeros((2, 7)), [-math.inf, -math.inf])
    assert l4 == -math.inf and (o4 == 0).all()
    o5, l5 = O.lse_merge(np.zeros((2, 7)), [-math.inf, -math.inf], sink=0.3)
    assert l5 == 0.3 and (o5 == 0).all()


# ---------------------------------------------------------------------------
# SFA remap
# ---------------------------------------------------------------------------

def test_sfa_remap_matches_slot_mapping_and_sparse_merge():
    import workloads as W
    dcp, bs, I = 4, 8, 8
    lens = np.array([200, 77])
    bt, nb = W.make_block_tables(lens, dcp, bs, "random", seed=9)
    rng = np.random.default_rng(3)
    topk = np.stack([rng.choice(200, 40, replace=False), np.r_[rng.choice(77, 38, replace=False), -1, 77]])
    rank, slot = O.sfa_remap(topk, lens, bt, dcp, bs, I, nb)
    for b in range(2):
        for k in range(topk.shape[1]):
            g = int(topk[b, k])
            if g < 0 or g >= lens[b]:
                assert rank[b, k] == -1 and slot[b, k] == -1
                continue
            rk, sl = O.slot_mapping([b], [g], bt, lens, dcp, bs, I, nb)
            assert rank[b, k] == rk[0] and slot[b, k] == sl[rk[0], 0]
    # remapped slots address exactly the selected tokens' rows in the built caches
    req = np.concatenate([np.full(L, b) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    rows = np.arange(len(req))[:, None] * 10 + np.arange(3)[None]
    _, sl_all = O.slot_mapping(req, pos, bt, lens, dcp, bs, I, nb)
    caches = O.build_caches(rows, sl_all, dcp, nb, bs, -1)
    for b in range(2):
        for k in range(topk.shape[1]):
            if rank[b, k] >= 0:
                t = int(np.nonzero((req == b) & (pos == topk[b, k]))[0][0])
                assert (caches[rank[b, k], slot[b, k]] == rows[t]).all()
    # sharded sparse attention + sink equals the unsharded sparse attention with the sink key
    q, K, V = rnd(rng, 12), rnd(rng, 200, 12), rnd(rng, 200, 5)
    o, lse, _, _ = O.sfa_sharded(q, K, V, 0.4, topk[0], 200, dcp, bs, I, sink=None)
    o2, lse2 = O.sparse_attention(q, K, V, 0.4, topk[0])
    np.testing.assert_allclose(o, o2, rtol=1e-12)
    assert lse == pytest.approx(lse2, rel=1e-13)


def test_replicated_window_contributes_once():
    """'Replicated SWA contributes on one rank' (TokenSpeed page, "Decode
    computation"): merging the per-rank partials of the sharded keys with
    ONE partial of the replicated window keys (and the sink) equals attention
    over the union of both key sets plus the sink key; adding the window
    partial once per rank does not."""
    rng = np.random.default_rng(8)
    L, W, dcp, bs, I = 300, 40, 4, 8, 2
    q, K, V = rnd(rng, 16), rnd(rng, L, 16), rnd(rng, L, 12)
    Kw, Vw = rnd(rng, W, 16), rnd(rng, W, 12)
    sigma, scale = 0.9, 0.3
    _, _, po, pl = O.sharded_attention(q, K, V, scale, L, dcp, bs, I)
    ow, lw = O.attention(q, Kw, Vw, scale)
    o, lse = O.lse_merge(np.vstack([po, ow]), list(pl) + [lw], sink=sigma)
    k_star = q * sigma / (scale * float(np.dot(q, q)))
    o2, lse2 = O.attention(q, np.vstack([K, Kw, k_star]), np.vstack([V, Vw, np.zeros(12)]), scale)
    np.testing.assert_allclose(o, o2, rtol=1e-11, atol=1e-13)
    assert lse == pytest.approx(lse2, rel=1e-13)
    o3, lse3 = O.lse_merge(np.vstack([po] + [ow] * dcp), list(pl) + [lw] * dcp, sink=sigma)
    assert abs(lse3 - lse) > 1e-6


def test_distributed_topk_is_exact_and_follows_the_tie_rule():
    import heapq
    rng = np.random.default_rng(12)
    for dcp, bs, I, L, k in [(4, 8, 2, 500, 37), (8, 64, 64, 3000, 256), (3, 16, 1, 50, 64),
                             (2, 4, 4, 9, 9)]:
        # coarse scores: many ties
        g_scores = np.round(rng.standard_normal(L) * 2) / 2
        g_scores[rng.random(L) < 0.02] = np.nan
        ids = np.arange(L)
        # brute force: pick k times the best remaining (max score, then min id)
        pool = [(-(-np.inf if np.isnan(s) else s), int(i)) for s, i in zip(g_scores, ids)]
        want = [i for _, i in heapq.nsmallest(k, pool)]
        got_ids, got_scores = O.topk_exact(g_scores, ids, k)
        assert list(got_ids) == want
        # the same selection from per-rank local scores
        local = [[] for _ in range(dcp)]
        for x in range(L):
            local[O.target_rank(x, bs, dcp, I)].append(g_scores[x])
        lens = [len(v) for v in local]
        d_ids, d_scores = O.topk_distributed(local, lens, k, dcp, bs, I)
        assert list(d_ids) == want
        np.testing.assert_array_equal(d_scores, g_scores[want])
    # -0 and +0 are one score, and NaN ties with -inf; ties go by the smaller id
    z_ids, _ = O.topk_exact(np.array([0.0, -0.0, np.nan, -np.inf, 0.0]), np.array([4, 1, 0, 2, 3]), 5)
    assert list(z_ids) == [1, 3, 4, 0, 2]


def test_sfa_compaction_keeps_exactly_the_referenced_rows():
    import workloads as W
    dcp, bs, I = 4, 8, 8
    lens = np.array([500, 90])
    bt, nb = W.make_block_tables(lens, dcp, bs, "random", seed=4)
    req = np.concatenate([np.full(L, b) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    rows = np.arange(len(req) * 2).reshape(len(req), 2) + 1
    _, slot = O.slot_mapping(req, pos, bt, lens, dcp, bs, I, nb)
    caches = O.build_caches(rows, slot, dcp, nb, bs, -1)
    rng = np.random.default_rng(5)
    q_req = np.array([0, 0, 1, 0, 1])
    topk = np.stack([rng.choice(int(lens[b]), 20, replace=False) for b in q_req])
    topk[1, 3] = -1
    topk[2, 0] = 90
    blocks, ids, counts, index = O.sfa_compact_blocks(topk, q_req, lens, bt, caches, dcp, bs, I,
                                                      nb)
    flat = blocks.reshape(-1, 2)
    for qi in range(len(q_req)):
        for k in range(20):
            g = int(topk[qi, k])
            if g < 0 or g >= lens[q_req[qi]]:
                assert index[qi, k] == -1
                continue
            t = int(np.nonzero((req == q_req[qi]) & (pos == g))[0][0])
            assert (flat[index[qi, k]] == rows[t]).all()   # the selected token's own row
    # exactly the referenced blocks: brute-force set of (rank, block) over entries
    want = set()
    for qi in range(len(q_req)):
        for g in topk[qi]:
            if 0 <= g < lens[q_req[qi]]:
                r = O.target_rank(int(g), bs, dcp, I)
                want.add((r, int(bt[r, q_req[qi], O.virtual_block_index(int(g), bs, dcp)])))
    assert counts.sum() == len(want) == len(ids)
    start = 0
    for r in range(dcp):
        got = list(ids[start:start + counts[r]])
        assert got == sorted(p for rr, p in want if rr == r)
        start += counts[r]


def test_gather_context_inverts_the_cache_write():
    import workloads as W
    for dcp, bs, I in [(2, 4, 2), (4, 16, 1), (3, 8, 8)]:
        lens = np.array([1, 50, 3 * bs * dcp + 7])
        bt, nb = W.make_block_tables(lens, dcp, bs, "random", seed=dcp)
        req = np.concatenate([np.full(L, b) for b, L in enumerate(lens)])
        pos = np.concatenate([np.arange(L) for L in lens])
        rows = np.arange(len(req) * 3).reshape(len(req), 3) + 7
        _, slot = O.slot_mapping(req, pos, bt, lens, dcp, bs, I, nb)
        caches = O.build_caches(rows, slot, dcp, nb, bs, -1)
        # request-contiguous order is the write order: the gather returns the rows
        out, bad = O.gather_context(req, pos, caches, bt, dcp, bs, I, nb)
        assert bad == 0 and (out == rows).all()
        # any other order of tokens gives the same rows permuted
        perm = np.random.default_rng(1).permutation(len(req))
        out, _ = O.gather_context(req[perm], pos[perm], caches, bt, dcp, bs, I, nb)
        assert (out == rows[perm]).all()
        # unresolvable tokens give zero rows
        out, bad = O.gather_context([0, 5], [10 ** 6, 0], caches, bt, dcp, bs, I, nb)
        assert bad == 2 and (out == 0).all()


# ---------------------------------------------------------------------------
# several query heads over one key set (the full-size parity checks use
# these): pinned against scipy per head and the procedural dealing, not
# against the single-head oracle functions
# ---------------------------------------------------------------------------

def scipy_attention(q, K, V, scale):
    s = scale * np.einsum("d,nd->n", q, K)
    return scipy.special.softmax(s) @ V, scipy.special.logsumexp(s)


def test_attention_heads_against_library_routines():
    rng = np.random.default_rng(21)
    for nh, n, dk, dv in [(1, 1, 4, 4), (4, 300, 64, 64), (3, 33, 576, 512), (5, 2, 8, 3)]:
        Q, K, V = rnd(rng, nh, dk), rnd(rng, n, dk), rnd(rng, n, dv)
        o, lse = O.attention_heads(Q, K, V, 0.41)
        assert o.shape == (nh, dv) and lse.shape == (nh,)
        for h in range(nh):
            o_ref, l_ref = scipy_attention(Q[h], K, V, 0.41)
            np.testing.assert_allclose(o[h], o_ref, rtol=1e-12, atol=1e-13)
            assert lse[h] == pytest.approx(l_ref, rel=1e-13, abs=1e-13)
    # one key: every head gets v and its own score
    Q, k, v = rnd(rng, 3, 8), rnd(rng, 8), rnd(rng, 5)
    o, lse = O.attention_heads(Q, k[None], v[None], 0.5)
    for h in range(3):
        np.testing.assert_allclose(o[h], v, rtol=1e-14)
        assert lse[h] == pytest.approx(0.5 * float(Q[h] @ k), rel=1e-14)
    # no keys
    o, lse = O.attention_heads(Q, np.zeros((0, 8)), np.zeros((0, 5)), 1.0)
    assert (o == 0).all() and (lse == -math.inf).all()


@pytest.mark.parametrize("dcp,bs,I", [(1, 16, 1), (8, 16, 1), (3, 8, 4), (8, 64, 64), (4, 4, 2)])
def test_sharded_attention_heads_against_dealing_and_scipy(dcp, bs, I):
    """Per-rank partials equal scipy attention over the tokens the procedural
    dealing gives each rank; the merged result equals scipy attention over
    all keys plus, with a sink, one extra key of logit sigma_h and zero value."""
    rng = np.random.default_rng(dcp * 7 + bs + I)
    nh, dk, dv, scale = 4, 16, 12, 0.3
    for L in [1, dcp, bs * dcp + 1, 500]:
        Q, K, V = rnd(rng, nh, dk), rnd(rng, L, dk), rnd(rng, L, dv)
        sinks = rnd(rng, nh)
        local = deal_tokens(L, dcp, bs, I)
        for with_sink in (False, True):
            o, lse, po, pl = O.sharded_attention_heads(Q, K, V, scale, L, dcp, bs, I,
                                                       sinks=sinks if with_sink else None)
            for h in range(nh):
                for r in range(dcp):
                    if not local[r]:
                        assert pl[r, h] == -math.inf and (po[r, h] == 0).all()
                        continue
                    o_r, l_r = scipy_attention(Q[h], K[local[r]], V[local[r]], scale)
                    np.testing.assert_allclose(po[r, h], o_r, rtol=1e-12, atol=1e-13)
                    assert pl[r, h] == pytest.approx(l_r, rel=1e-13, abs=1e-13)
                s = scale * (K @ Q[h])
                if with_sink:
                    s = np.r_[s, sinks[h]]
                w = scipy.special.softmax(s)[:L]
                np.testing.assert_allclose(o[h], w @ V, rtol=1e-11, atol=1e-13)
                assert lse[h] == pytest.approx(scipy.special.logsumexp(s), rel=1e-13, abs=1e-13)


def test_sfa_sharded_heads_against_dealing_and_scipy():
    """Only the selected rows are given; entries outside [0, L) are dropped;
    each valid entry (duplicates included) is attended once, by the rank the
    procedural dealing gives its token; the merge applies each head's sink once."""
    rng = np.random.default_rng(33)
    dcp, bs, I, L = 4, 8, 8, 700
    nh, dk, dv, scale = 3, 20, 16, 0.25
    owner = np.empty(L, dtype=np.int64)
    for r, toks in enumerate(deal_tokens(L, dcp, bs, I)):
        owner[toks] = r
    sel = np.r_[rng.choice(L, 60, replace=False), [-1, L, 5, 5]]
    Ksel, Vsel = rnd(rng, len(sel), dk), rnd(rng, len(sel), dv)
    Ksel[-1], Vsel[-1] = Ksel[-2], Vsel[-2]         # the duplicate carries the same row
    Q, sinks = rnd(rng, nh, dk), rnd(rng, nh)
    o, lse, po, pl = O.sfa_sharded_heads(Q, sel, Ksel, Vsel, scale, L, dcp, bs, I, sinks=sinks)
    valid = (sel >= 0) & (sel < L)
    for h in range(nh):
        for r in range(dcp):
            m = valid & (owner[np.clip(sel, 0, L - 1)] == r)
            if not m.any():
                assert pl[r, h] == -math.inf
                continue
            o_r, l_r = scipy_attention(Q[h], Ksel[m], Vsel[m], scale)
            np.testing.assert_allclose(po[r, h], o_r, rtol=1e-12, atol=1e-13)
            assert pl[r, h] == pytest.approx(l_r, rel=1e-13)
        s = np.r_[scale * (Ksel[valid] @ Q[h]), sinks[h]]
        w = scipy.special.softmax(s)[:-1]
        np.testing.assert_allclose(o[h], w @ Vsel[valid], rtol=1e-11, atol=1e-13)
        assert lse[h] == pytest.approx(scipy.special.logsumexp(s), rel=1e-13)

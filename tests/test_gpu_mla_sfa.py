"""MLA and SFA decode vs the fp64 oracle (small cases; full size: every request)."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from workloads import device as D
from tests import ref

pytestmark = pytest.mark.gpu

MLA = W.CONFIGS["mla_bf16_b64"]
SFA = W.CONFIGS["sfa_bf16_b32"]

MLA_SMALL = [
    dataclasses.replace(MLA, B=2, lengths=[100, 37], dcp=2, bs=64, I=1),
    dataclasses.replace(MLA, B=3, lengths=[1, 640, 2049], dcp=4, bs=64, I=1),
    dataclasses.replace(MLA, B=2, lengths=[777, 64], dcp=3, bs=64, I=16),
    dataclasses.replace(MLA, B=2, Hq=16, lengths=[300, 5], dcp=2, bs=16, I=1),
    dataclasses.replace(MLA, B=2, Hq=4, dtype="f32", lengths=[90, 7], dcp=2, bs=16, I=2),
    # a request with an empty context: output 0, LSE -inf
    dataclasses.replace(MLA, B=3, lengths=[0, 300, 65], dcp=2, bs=64, I=1),
    # one rank: plain paged attention
    dataclasses.replace(MLA, B=2, lengths=[200, 64], dcp=1, bs=64, I=1),
]


def cid(c):
    return f"{c.kind}-{c.dtype}-B{c.B}-H{c.Hq}-dcp{c.dcp}-bs{c.bs}-I{c.I}"


def check(cfg, *a):
    (ref.check_f32 if cfg.dtype == "f32" else ref.check_bf16)(*a)


@pytest.mark.parametrize("cfg", MLA_SMALL, ids=cid)
def test_mla_small(lib, cfg):
    wl = D.build(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    po, pl = lib.decode_partial_mla(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, cfg.dv,
                                    err=err)
    out, lse = lib.decode_mla(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, cfg.dv,
                              out_dtype=torch.float32, err=err)
    po, pl, out, lse = (t.cpu().numpy() for t in (po, pl, out, lse))
    assert err.item() == 0
    # every head when the contexts are tiny (the full tiny MLA case: B=2,
    # L={100, 37}, all 128 heads), else both ends of each half of the heads
    heads = range(cfg.Hq) if cfg.Hq <= 16 or sum(cfg.lengths) <= 256 else [0, 1, 63, 64, 127]
    for b in range(cfg.B):
        exp = ref.mla_expected(cfg, wl.seq_lens_host, b, heads)
        for h in heads:
            o_ref, lse_ref, po_ref, pl_ref = exp[h]
            check(cfg, out[b, h], lse[b, h], o_ref, lse_ref, f"fused b{b} h{h}")
            for r in range(cfg.dcp):
                check(cfg, po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"r{r} b{b} h{h}")


SFA_SMALL = [
    dataclasses.replace(SFA, B=2, lengths=[3000, 70], topk=64),
    dataclasses.replace(SFA, B=3, lengths=[5000, 900, 2048], topk=256, dcp=4, bs=64, I=1),
    dataclasses.replace(SFA, B=2, Hq=8, dtype="f32", lengths=[400, 64], topk=32, dcp=2, bs=16,
                        I=16),
    dataclasses.replace(SFA, B=2, Hq=128, lengths=[9000, 300], topk=200, dcp=4, bs=64, I=64),
    dataclasses.replace(SFA, B=3, Hq=16, lengths=[3000, 17, 640], topk=16, dcp=2, bs=16, I=4),
    # one rank: plain sparse attention
    dataclasses.replace(SFA, B=2, lengths=[3000, 200], topk=128, dcp=1, bs=64, I=64),
    # six ranks (the fused call merges in clusters of six)
    dataclasses.replace(SFA, B=2, lengths=[9000, 1100], topk=300, dcp=6, bs=64, I=16),
    # more selected tokens than the tcgen05 kernel lists (2048): the other path
    dataclasses.replace(SFA, B=2, lengths=[20000, 5000], topk=3000, dcp=4, bs=64, I=64),
]


@pytest.mark.parametrize("cfg", SFA_SMALL, ids=cid)
def test_sfa_small(lib, cfg):
    wl = D.build(cfg)
    topk = wl.topk_host.copy()
    topk[0, 0] = -1                          # padding entries are skipped
    topk[-1, 1] = wl.seq_lens_host[-1]
    topk_d = torch.from_numpy(topk).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rk, sl = lib.sfa_remap(wl.layout, topk_d, wl.seq_lens, wl.block_table, wl.num_blocks, err=err)
    po, pl = lib.sfa_decode_partial(wl.layout, wl.q, wl.kv, rk, sl, cfg.scale, cfg.dv, err=err)
    out, lse = lib.sfa_decode(wl.layout, wl.q, wl.kv, topk_d, wl.seq_lens, cfg.scale, cfg.dv,
                              sink=wl.sink, out_dtype=torch.float32, err=err)
    mo, ml = lib.lse_merge(po, pl, wl.sink)
    assert err.item() == 0
    po, pl, out, lse, mo, ml = (t.cpu().numpy() for t in (po, pl, out, lse, mo, ml))
    sink = wl.sink.cpu().numpy()
    for b in range(cfg.B):
        heads = range(cfg.Hq) if cfg.Hq <= 8 else [0, 5, cfg.Hq - 1]
        exp = ref.sfa_expected(cfg, wl.seq_lens_host, topk, b, heads, sink=sink)
        for h in heads:
            o_ref, lse_ref, po_ref, pl_ref = exp[h]
            check(cfg, out[b, h], lse[b, h], o_ref, lse_ref, f"fused b{b} h{h}")
            check(cfg, mo[b, h], ml[b, h], o_ref, lse_ref, f"merge b{b} h{h}")
            for r in range(cfg.dcp):
                check(cfg, po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"r{r} b{b} h{h}")


def test_sfa_full_size_all_heads(lib):
    """Every request and every head of the SFA workload: the fused output and
    LSE (sink applied once) and every rank's partial, against the oracle."""
    wl = D.build(SFA)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.sfa_decode(wl.layout, wl.q, wl.kv, wl.topk, wl.seq_lens, SFA.scale, SFA.dv,
                              sink=wl.sink, err=err)
    rk, sl = lib.sfa_remap(wl.layout, wl.topk, wl.seq_lens, wl.block_table, wl.num_blocks,
                           err=err)
    po, pl = lib.sfa_decode_partial(wl.layout, wl.q, wl.kv, rk, sl, SFA.scale, SFA.dv, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    sink = wl.sink.cpu().numpy()
    worst = ref.WorstError()
    heads = range(SFA.Hq)
    for b, exp in ref.expected_for_requests(
            lambda b: ref.sfa_expected(SFA, wl.seq_lens_host, wl.topk_host, b, heads, sink=sink),
            range(SFA.B)):
        for h in heads:
            o_ref, lse_ref, po_ref, pl_ref = exp[h]
            ref.check_bf16(out[b, h], lse[b, h], o_ref, lse_ref, f"b{b} h{h}")
            worst.add(out[b, h], o_ref)
            for r in range(SFA.dcp):
                ref.check_bf16(po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"r{r} b{b} h{h}")
                worst.add(po[r, b, h], po_ref[r], partial=True)
    print(SFA.name, worst)


# The fused call on shapes the small cases miss: long per-rank selections
# (16 stages of 64 tokens per rank), a whole context selected (exactly 8 stages
# per rank) next to a request whose ranks 2 and 3 select nothing, 128 heads
# (two CTAs per (rank, request)), and more (rank, request) problems than SMs.
SFA_FUSED = [
    dataclasses.replace(SFA, B=2, lengths=[60000, 9000], topk=2048, dcp=2),
    dataclasses.replace(SFA, B=2, lengths=[2048, 100000], topk=2048, dcp=4),
    dataclasses.replace(SFA, B=2, Hq=128, lengths=[20000, 4000], topk=1000, dcp=2),
    dataclasses.replace(SFA, B=40, lengths=[600 + 97 * i for i in range(40)], topk=128, dcp=8),
]


@pytest.mark.parametrize("cfg", SFA_FUSED, ids=lambda c: f"B{c.B}-H{c.Hq}-dcp{c.dcp}-k{c.topk}")
def test_sfa_fused_shapes(lib, cfg):
    wl = D.build(cfg)
    topk = wl.topk_host.copy()
    if cfg.dcp == 4:
        rank = (topk[1] % (cfg.bs * cfg.dcp)) // cfg.I % cfg.dcp
        topk[1][rank >= 2] = -1
    topk_d = torch.from_numpy(topk).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.sfa_decode(wl.layout, wl.q, wl.kv, topk_d, wl.seq_lens, cfg.scale, cfg.dv,
                              sink=wl.sink, out_dtype=torch.float32, err=err)
    out2, lse2 = lib.sfa_decode(wl.layout, wl.q, wl.kv, topk_d, wl.seq_lens, cfg.scale, cfg.dv,
                                sink=wl.sink, out_dtype=torch.float32, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out, out2) and torch.equal(lse, lse2), "not bitwise repeatable"
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    sink = wl.sink.cpu().numpy()
    reqs = range(cfg.B) if cfg.B <= 2 else [0, 17, cfg.B - 1]
    for b in reqs:
        heads = [0, 17, cfg.Hq - 1]
        exp = ref.sfa_expected(cfg, wl.seq_lens_host, topk, b, heads, sink=sink)
        for h in heads:
            check(cfg, out[b, h], lse[b, h], exp[h][0], exp[h][1], f"b{b} h{h}")


@pytest.mark.parametrize("k_kind", ["no_entries", "padding_only"])
@pytest.mark.parametrize("with_sink", [False, True])
def test_sfa_empty_selection(lib, k_kind, with_sink):
    """No selected token on any rank: the fused call (tensor-core path) and the
    partial path give o = 0 with lse = the sink (or -inf without one), as the
    oracle does."""
    cfg = dataclasses.replace(SFA, B=2, lengths=[3000, 700], topk=64, dcp=4)
    wl = D.build(cfg)
    K = 0 if k_kind == "no_entries" else 64
    topk = torch.full((cfg.B, K), -1, dtype=torch.int32, device="cuda")
    sink = wl.sink if with_sink else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.sfa_decode(wl.layout, wl.q, wl.kv, topk, wl.seq_lens, cfg.scale, cfg.dv,
                              sink=sink, out_dtype=torch.float32, err=err)
    rk, sl = lib.sfa_remap(wl.layout, topk, wl.seq_lens, wl.block_table, wl.num_blocks, err=err)
    po, pl = lib.sfa_decode_partial(wl.layout, wl.q, wl.kv, rk, sl, cfg.scale, cfg.dv, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    out, lse, po, pl = (t.cpu().numpy() for t in (out, lse, po, pl))
    sink_h = wl.sink.cpu().numpy() if with_sink else None
    exp = ref.sfa_expected(cfg, wl.seq_lens_host, np.full((cfg.B, K), -1, np.int32), 0, [0, 63],
                           sink=sink_h)
    for h in (0, 63):
        ref.check_bf16(out[0, h], lse[0, h], exp[h][0], exp[h][1], f"h{h}")
    assert not out.any()
    assert not po.any() and np.isneginf(pl).all()
    if with_sink:
        np.testing.assert_allclose(lse, np.broadcast_to(sink_h, lse.shape), rtol=0, atol=1e-6)
    else:
        assert np.isneginf(lse).all()


def test_sfa_duplicate_indices_are_attended_as_listed(lib):
    """The top-k list is taken literally: an index listed twice is attended
    twice, by the fused call and the partial path alike, as by the oracle."""
    cfg = dataclasses.replace(SFA, B=2, lengths=[5000, 900], topk=128, dcp=4)
    wl = D.build(cfg)
    topk = wl.topk_host.copy()
    topk[0, 64:96] = topk[0, 0:32]          # 32 duplicates in request 0
    topk[1, 1] = topk[1, 0]
    topk_d = torch.from_numpy(topk).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.sfa_decode(wl.layout, wl.q, wl.kv, topk_d, wl.seq_lens, cfg.scale, cfg.dv,
                              sink=wl.sink, out_dtype=torch.float32, err=err)
    rk, sl = lib.sfa_remap(wl.layout, topk_d, wl.seq_lens, wl.block_table, wl.num_blocks, err=err)
    po, pl = lib.sfa_decode_partial(wl.layout, wl.q, wl.kv, rk, sl, cfg.scale, cfg.dv, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    out, lse, po, pl = (t.cpu().numpy() for t in (out, lse, po, pl))
    sink = wl.sink.cpu().numpy()
    for b in range(cfg.B):
        exp = ref.sfa_expected(cfg, wl.seq_lens_host, topk, b, [0, 31, 63], sink=sink)
        for h in (0, 31, 63):
            o_ref, lse_ref, po_ref, pl_ref = exp[h]
            ref.check_bf16(out[b, h], lse[b, h], o_ref, lse_ref, f"fused b{b} h{h}")
            for r in range(cfg.dcp):
                ref.check_bf16(po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"r{r} b{b} h{h}")


def mla_full(lib, cfg, heads_per_req, seed):
    """Every request, with heads_per_req seeded heads each (an fp64 check of all
    128 heads of 6M tokens would take hours): the fused output and LSE and
    every rank's partial, against the oracle."""
    wl = D.build(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.decode_mla(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, cfg.dv, err=err)
    po, pl = lib.decode_partial_mla(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, cfg.dv,
                                    err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    lens = wl.seq_lens_host
    del wl
    rng = np.random.default_rng(seed)
    heads = {b: sorted(rng.choice(cfg.Hq, heads_per_req, replace=False).tolist())
             for b in range(cfg.B)}
    worst = ref.WorstError()
    for b, exp in ref.expected_for_requests(lambda b: ref.mla_expected(cfg, lens, b, heads[b]),
                                            range(cfg.B), workers=2):
        for h in heads[b]:
            o_ref, lse_ref, po_ref, pl_ref = exp[h]
            ref.check_bf16(out[b, h], lse[b, h], o_ref, lse_ref, f"b{b} h{h}")
            worst.add(out[b, h], o_ref)
            for r in range(cfg.dcp):
                ref.check_bf16(po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"r{r} b{b} h{h}")
                worst.add(po[r, b, h], po_ref[r], partial=True)
    print(cfg.name, worst)


def test_mla_bad_block_table_entries_are_counted(lib):
    """Unusable block-table entries are counted, their stages attend nothing,
    and requests that do not touch them still match the oracle."""
    cfg = dataclasses.replace(MLA, B=2, lengths=[700, 300], dcp=2, bs=64, I=1)
    wl = D.build(cfg)
    bt = wl.block_table.clone()
    bt[1, 0, 2] = wl.num_blocks + 5     # rank 1, request 0, virtual block 2
    bt[0, 0, 1] = -3                    # rank 0, request 0, virtual block 1
    import context_paged_decode_gb300 as dcp
    kv = dcp.PagedKV(wl.k_pools, None, bt, wl.num_blocks)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.decode_mla(wl.layout, wl.q, kv, wl.local_lens, cfg.scale, cfg.dv,
                              out_dtype=torch.float32, err=err)
    torch.cuda.synchronize()
    assert 0 < err.item() < (1 << 20)   # counted; no wait timed out
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    heads = [0, 77, 127]
    exp = ref.mla_expected(cfg, wl.seq_lens_host, 1, heads)
    for h in heads:
        check(cfg, out[1, h], lse[1, h], exp[h][0], exp[h][1], f"b1 h{h}")


def test_mla_bf16_b64_full_size_all_requests(lib):
    mla_full(lib, MLA, 4, seed=0)


def test_longtail_mla_full_size_all_requests(lib):
    mla_full(lib, W.CONFIGS["longtail_mla"], 4, seed=1)


@pytest.mark.parametrize("dcp_size", [1, 2])
def test_mla_online_softmax_rescale(lib, dcp_size):
    """Scores that keep growing along the sequence (and one dominant late
    token) force the output to be rescaled many times."""
    import context_paged_decode_gb300 as dcp
    import oracle as O
    cfg = dataclasses.replace(MLA, B=1, lengths=[3000], dcp=dcp_size, bs=64, I=1)
    rng = np.random.default_rng(11)
    L = 3000
    q = rng.standard_normal((1, 128, 576)).astype(np.float32)
    kv = rng.standard_normal((L, 576)).astype(np.float32)
    kv[:, :] *= (1.0 + 6.0 * np.arange(L) / L)[:, None]
    kv[2500] = q[0, 5] * 0.2                              # one token that dominates head 5
    qb = W.f32_to_bf16_bits(q)
    kvb = W.f32_to_bf16_bits(kv)
    wl = D.build(cfg, populate=False)
    wl.q.view(torch.int16).copy_(torch.from_numpy(qb.view(np.int16)))
    req = torch.zeros(L, dtype=torch.int32, device="cuda")
    pos = torch.arange(L, dtype=torch.int64, device="cuda")
    _, slot = dcp.slot_mapping(wl.layout, req, pos, wl.block_table, wl.num_blocks)
    kvd = torch.from_numpy(kvb.view(np.int16)).cuda().view(torch.bfloat16)
    dcp.cache_write_mla(wl.layout, kvd, slot, wl.k_pools, wl.num_blocks)
    out, lse = lib.decode_mla(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, 512,
                              out_dtype=torch.float32)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    K = W.as_float64(kvb, "bf16")
    for h in [0, 5, 77, 127]:
        qv = W.as_float64(qb[0, h], "bf16")
        o_ref, lse_ref = O.attention(qv, K, K[:, :512], cfg.scale)
        ref.check_bf16(out[0, h], lse[0, h], o_ref, lse_ref, f"h{h}")


@pytest.mark.parametrize("dcp_size", [1, 2])
def test_sfa_online_softmax_rescale(lib, dcp_size):
    """Selected tokens whose scores grow along the top-k order (and one
    dominant late token) force the sparse kernel to rescale its output.
    Only the 64 rope columns grow: the scores' spread rises more than
    four-fold along the selection (every head's running maximum grows by more
    than 8 in log2 one to three times), while the value columns stay N(0, 1),
    so the output keeps the O(1) scale the bf16 tolerance is stated for."""
    import context_paged_decode_gb300 as dcp
    import oracle as O
    L, K = 3000, 1024
    cfg = dataclasses.replace(SFA, B=1, lengths=[L], topk=K, dcp=dcp_size, bs=64, I=1)
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, cfg.Hq, 576)).astype(np.float32)
    kv = rng.standard_normal((L, 576)).astype(np.float32)
    sel = np.sort(rng.choice(L, K, replace=False)).astype(np.int32)
    kv[sel, 512:] *= (1.0 + 12.0 * np.arange(K) / K)[:, None]
    kv[sel[900]] = q[0, 5] * 0.8                          # dominates head 5
    qb = W.f32_to_bf16_bits(q)
    kvb = W.f32_to_bf16_bits(kv)
    wl = D.build(cfg, populate=False)
    wl.q.view(torch.int16).copy_(torch.from_numpy(qb.view(np.int16)))
    req = torch.zeros(L, dtype=torch.int32, device="cuda")
    pos = torch.arange(L, dtype=torch.int64, device="cuda")
    _, slot = dcp.slot_mapping(wl.layout, req, pos, wl.block_table, wl.num_blocks)
    kvd = torch.from_numpy(kvb.view(np.int16)).cuda().view(torch.bfloat16)
    dcp.cache_write_mla(wl.layout, kvd, slot, wl.k_pools, wl.num_blocks)
    topk = torch.from_numpy(sel[None, :].copy()).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.sfa_decode(wl.layout, wl.q, wl.kv, topk, wl.seq_lens, cfg.scale, 512,
                              out_dtype=torch.float32, err=err)
    assert err.item() == 0
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    Ksel = W.as_float64(kvb, "bf16")[sel]
    for h in [0, 5, 33, cfg.Hq - 1]:
        qv = W.as_float64(qb[0, h], "bf16")
        o_ref, lse_ref = O.attention(qv, Ksel, Ksel[:, :512], cfg.scale)
        ref.check_bf16(out[0, h], lse[0, h], o_ref, lse_ref, f"h{h}")


@pytest.mark.parametrize("hq", [64, 128])
def test_sfa_bad_slots_are_counted_and_masked(lib, hq):
    """(rank, slot) pairs whose slot lies outside the rank's cache are counted
    once each and attended as masked tokens: the partials equal the oracle's
    with those top-k entries dropped."""
    cfg = dataclasses.replace(SFA, B=2, Hq=hq, lengths=[5000, 900], topk=256, dcp=4, bs=64, I=1)
    wl = D.build(cfg)
    topk = wl.topk_host.copy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rk, sl = lib.sfa_remap(wl.layout, torch.from_numpy(topk).cuda(), wl.seq_lens, wl.block_table,
                           wl.num_blocks, err=err)
    assert err.item() == 0
    rk_h, sl_h = rk.cpu().numpy(), sl.cpu().numpy()
    bad = [(0, 3), (0, 100), (1, 7)]                      # (request, top-k index)
    for b, k in bad:
        assert rk_h[b, k] >= 0
        sl_h[b, k] = wl.num_blocks * cfg.bs + 5           # beyond the rank's slots
        topk[b, k] = -1                                   # the oracle drops it
    po, pl = lib.sfa_decode_partial(wl.layout, wl.q, wl.kv, rk, torch.from_numpy(sl_h).cuda(),
                                    cfg.scale, cfg.dv, err=err)
    torch.cuda.synchronize()
    assert err.item() == len(bad)
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    for b in range(cfg.B):
        heads = [0, 37, hq - 1]
        exp = ref.sfa_expected(cfg, wl.seq_lens_host, topk, b, heads)
        for h in heads:
            _, _, po_ref, pl_ref = exp[h]
            for r in range(cfg.dcp):
                check(cfg, po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"r{r} b{b} h{h}")


@pytest.mark.parametrize("hq", [64, 128])
def test_sfa_fused_bad_block_table_entries_are_counted_and_dropped(lib, hq):
    """A selected token whose block-table entry is unusable is dropped by the
    fused call and counted once, as dcp_sfa_remap drops and counts it for the
    same table, and the output equals the oracle's with those entries
    dropped."""
    import context_paged_decode_gb300 as dcp
    cfg = dataclasses.replace(SFA, B=2, Hq=hq, lengths=[5000, 900], topk=256, dcp=4, bs=64, I=1)
    wl = D.build(cfg)
    topk = wl.topk_host.copy()
    vbs = cfg.bs * cfg.dcp
    bt = wl.block_table.clone()
    rk_good, _ = lib.sfa_remap(wl.layout, wl.topk, wl.seq_lens, wl.block_table, wl.num_blocks)
    rk_good = rk_good.cpu().numpy()
    # unusable entries of three (rank, request, virtual block) that selected
    # tokens go through: past the pool, negative, and past the pool again
    picks = [(0, 3, wl.num_blocks + 5), (0, 100, -3), (1, 7, wl.num_blocks)]
    for b, k, val in picks:
        assert rk_good[b, k] >= 0
        bt[rk_good[b, k], b, int(topk[b, k]) // vbs] = val
    kv = dcp.PagedKV(wl.kv.k_pools, None, bt, wl.num_blocks)
    err_remap = torch.zeros(1, dtype=torch.int32, device="cuda")
    rk_bad, _ = lib.sfa_remap(wl.layout, wl.topk, wl.seq_lens, bt, wl.num_blocks, err=err_remap)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.sfa_decode(wl.layout, wl.q, kv, wl.topk, wl.seq_lens, cfg.scale, cfg.dv,
                              sink=wl.sink, out_dtype=torch.float32, err=err)
    torch.cuda.synchronize()
    rk_bad = rk_bad.cpu().numpy()
    dropped = (rk_bad < 0) & (rk_good >= 0)
    assert dropped.sum() >= len(picks)
    assert err_remap.item() == dropped.sum()
    assert err.item() == err_remap.item()
    topk[dropped] = -1                                    # the oracle drops them
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    sink = None if wl.sink is None else wl.sink.cpu().numpy()
    for b in range(cfg.B):
        heads = [0, 37, hq - 1]
        exp = ref.sfa_expected(cfg, wl.seq_lens_host, topk, b, heads, sink=sink)
        for h in heads:
            check(cfg, out[b, h], lse[b, h], exp[h][0], exp[h][1], f"b{b} h{h}")


# The fused call merges the per-rank partials inside the partials kernel (a
# cluster of the request's CTAs); its output must be bitwise that of the
# page-defined seam: dcp_sfa_decode_partial, then dcp_lse_merge with the sink.
SFA_SEAM = [
    SFA,                                                                   # clusters of 4
    dataclasses.replace(SFA, B=40, lengths=[600 + 97 * i for i in range(40)], topk=128),  # of 3
    dataclasses.replace(SFA, B=2, lengths=[60000, 9000], topk=2048),       # ranks one per CTA
    dataclasses.replace(SFA, B=3, Hq=128, lengths=[20000, 4000, 1700], topk=1000, dcp=4),
    # clusters of 6 and 7 CTAs (one rank each)
    dataclasses.replace(SFA, B=3, lengths=[30000, 7000, 2500], topk=700, dcp=6, bs=64, I=16),
    dataclasses.replace(SFA, B=2, lengths=[40000, 3000], topk=1500, dcp=7, bs=64, I=8),
]


@pytest.mark.parametrize("cfg", SFA_SEAM, ids=lambda c: f"B{c.B}-H{c.Hq}-dcp{c.dcp}-k{c.topk}")
def test_sfa_fused_equals_partials_then_merge(lib, cfg):
    wl = D.build(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for out_dtype in (torch.float32, torch.bfloat16):
        out, lse = lib.sfa_decode(wl.layout, wl.q, wl.kv, wl.topk, wl.seq_lens, cfg.scale, cfg.dv,
                                  sink=wl.sink, out_dtype=out_dtype, err=err)
        rk, sl = lib.sfa_remap(wl.layout, wl.topk, wl.seq_lens, wl.block_table, wl.num_blocks,
                               err=err)
        po, pl = lib.sfa_decode_partial(wl.layout, wl.q, wl.kv, rk, sl, cfg.scale, cfg.dv, err=err)
        mo, ml = lib.lse_merge(po, pl, wl.sink, out_dtype=out_dtype)
        torch.cuda.synchronize()
        assert err.item() == 0
        bits = torch.int32 if out_dtype == torch.float32 else torch.int16
        assert torch.equal(out.view(bits), mo.view(bits)), "fused output differs from partials + merge"
        assert torch.equal(lse.view(torch.int32), ml.view(torch.int32))


# 16 ranks: one rank per CTA gives groups of 16, above the portable cluster
# size, so the fused call keeps the separate merge kernel; the partials and
# the merged output still match the oracle
def test_sfa_sixteen_ranks_separate_merge(lib):
    cfg = dataclasses.replace(SFA, B=2, lengths=[40000, 9000], topk=512, dcp=16)
    wl = D.build(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.sfa_decode(wl.layout, wl.q, wl.kv, wl.topk, wl.seq_lens, cfg.scale, cfg.dv,
                              sink=wl.sink, out_dtype=torch.float32, err=err)
    rk, sl = lib.sfa_remap(wl.layout, wl.topk, wl.seq_lens, wl.block_table, wl.num_blocks, err=err)
    po, pl = lib.sfa_decode_partial(wl.layout, wl.q, wl.kv, rk, sl, cfg.scale, cfg.dv, err=err)
    mo, ml = lib.lse_merge(po, pl, wl.sink)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out.view(torch.int32), mo.view(torch.int32))
    out, lse, po, pl = (t.cpu().numpy() for t in (out, lse, po, pl))
    sink = wl.sink.cpu().numpy()
    for b in range(cfg.B):
        heads = [0, 21, 63]
        exp = ref.sfa_expected(cfg, wl.seq_lens_host, wl.topk_host, b, heads, sink=sink)
        for h in heads:
            o_ref, lse_ref, po_ref, pl_ref = exp[h]
            check(cfg, out[b, h], lse[b, h], o_ref, lse_ref, f"fused b{b} h{h}")
            for r in range(cfg.dcp):
                check(cfg, po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"r{r} b{b} h{h}")


def test_mla_sixteen_ranks(lib):
    cfg = dataclasses.replace(MLA, B=2, lengths=[30000, 5000], dcp=16, bs=64, I=1)
    wl = D.build(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.decode_mla(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, cfg.dv,
                              out_dtype=torch.float32, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(cfg.B):
        exp = ref.mla_expected(cfg, wl.seq_lens_host, b, [0, 64, 127])
        for h in (0, 64, 127):
            check(cfg, out[b, h], lse[b, h], exp[h][0], exp[h][1], f"b{b} h{h}")

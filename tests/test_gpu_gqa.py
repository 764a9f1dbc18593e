"""GQA decode partials and the fused decode step vs the fp64 oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from workloads import device as D
from tests import ref

pytestmark = pytest.mark.gpu

BASE = W.CONFIGS["gqa_bf16_b32"]

SMALL = [
    W.CONFIGS["tiny_gqa_f32"],
    dataclasses.replace(W.CONFIGS["tiny_gqa_f32"], perm="identity"),
    dataclasses.replace(W.CONFIGS["tiny_gqa_f32"], lengths=[1, 2, 33], B=3, dcp=4, I=2),
    dataclasses.replace(BASE, B=4, lengths=[1, 17, 1000, 4099], dcp=4, bs=16, I=1),
    dataclasses.replace(BASE, B=3, lengths=[5, 300, 2500], dcp=8, bs=16, I=16),
    dataclasses.replace(BASE, B=3, lengths=[64, 1, 3001], dcp=3, bs=64, I=4),
    dataclasses.replace(BASE, B=2, Hq=16, Hkv=2, lengths=[700, 33], dcp=2, bs=32, I=8),
    dataclasses.replace(BASE, B=2, Hq=16, Hkv=1, lengths=[513, 2048], dcp=2, bs=16, I=1),
    dataclasses.replace(BASE, B=2, Hq=8, Hkv=8, lengths=[100, 1], dcp=2, bs=16, I=1),
    dataclasses.replace(BASE, B=2, Hq=8, Hkv=2, dk=64, dv=64, lengths=[100, 900], dcp=2, bs=16),
    dataclasses.replace(BASE, B=2, lengths=[40, 333], dcp=2, bs=8, I=2),
    # a request with an empty context: output 0, LSE -inf (the sink's logit with a sink)
    dataclasses.replace(BASE, B=3, lengths=[0, 100, 37], dcp=2, bs=16, I=1),
    dataclasses.replace(W.CONFIGS["tiny_gqa_f32"], B=2, lengths=[37, 0]),
    # one rank: plain paged attention
    dataclasses.replace(BASE, B=2, lengths=[500, 33], dcp=1, bs=16, I=1),
]


def cid(c):
    return f"{c.dtype}-B{c.B}-H{c.Hq}/{c.Hkv}-d{c.dk}-dcp{c.dcp}-bs{c.bs}-I{c.I}-{c.perm}"


def check(cfg, o, lse, o_ref, lse_ref, what):
    (ref.check_f32 if cfg.dtype == "f32" else ref.check_bf16)(o, lse, o_ref, lse_ref, what)


@pytest.mark.parametrize("cfg", SMALL, ids=cid)
def test_small_partials_and_fused(lib, cfg):
    wl = D.build(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    po, pl = lib.decode_partial_gqa(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, err=err)
    sink = torch.from_numpy(np.linspace(-1, 1, cfg.Hq).astype(np.float32)).cuda()
    out, lse = lib.decode_gqa(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, err=err,
                              out_dtype=torch.float32)
    outs, lses = lib.decode_gqa(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, sink=sink,
                                err=err)
    # the page-defined seam: per-rank partials merged by dcp_lse_merge
    mo, ml = lib.lse_merge(po, pl, sink)
    po, pl, out, lse = po.cpu().numpy(), pl.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()
    outs, lses = outs.float().cpu().numpy(), lses.cpu().numpy()
    mo, ml = mo.cpu().numpy(), ml.cpu().numpy()
    assert err.item() == 0
    s_host = sink.cpu().numpy()
    for b in range(cfg.B):
        exp = ref.gqa_expected(cfg, wl.seq_lens_host, b, range(cfg.Hq))
        exps = ref.gqa_expected(cfg, wl.seq_lens_host, b, range(cfg.Hq), sink=s_host)
        for h in range(cfg.Hq):
            o_ref, lse_ref, po_ref, pl_ref = exp[h]
            for r in range(cfg.dcp):
                check(cfg, po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"partial r{r} b{b} h{h}")
            check(cfg, out[b, h], lse[b, h], o_ref, lse_ref, f"fused b{b} h{h}")
            so_ref, slse_ref = exps[h][0], exps[h][1]
            check(cfg, outs[b, h], lses[b, h], so_ref, slse_ref, f"sink b{b} h{h}")
            check(cfg, mo[b, h], ml[b, h], so_ref, slse_ref, f"merge b{b} h{h}")


def test_bad_block_table_entries_are_counted(lib):
    cfg = dataclasses.replace(BASE, B=2, lengths=[300, 50], dcp=2, bs=16)
    wl = D.build(cfg)
    bt = wl.block_table.clone()
    bt[1, 0, 2] = wl.num_blocks + 5     # rank 1, request 0, virtual block 2
    bt[0, 1, 0] = -3
    import context_paged_decode_gb300 as dcp
    kv = dcp.PagedKV(wl.k_pools, wl.v_pools, bt, wl.num_blocks)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.decode_gqa(wl.layout, wl.q, kv, wl.local_lens, cfg.scale, err=err)
    torch.cuda.synchronize()
    assert err.item() > 0
    assert torch.isfinite(out[0].float()).all()


def full_check(lib, cfg):
    """Every request and every query head: the fused output and LSE, and every
    rank's partial output and LSE, against the oracle."""
    wl = D.build(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.decode_gqa(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, err=err)
    po, pl = lib.decode_partial_gqa(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    lens = wl.seq_lens_host
    del wl
    worst = ref.WorstError()
    heads = range(cfg.Hq)
    for b, exp in ref.expected_for_requests(lambda b: ref.gqa_expected(cfg, lens, b, heads),
                                            range(cfg.B)):
        for h in heads:
            o_ref, lse_ref, po_ref, pl_ref = exp[h]
            ref.check_bf16(out[b, h], lse[b, h], o_ref, lse_ref, f"b{b} h{h}")
            worst.add(out[b, h], o_ref)
            for r in range(cfg.dcp):
                ref.check_bf16(po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"r{r} b{b} h{h}")
                worst.add(po[r, b, h], po_ref[r], partial=True)
    print(cfg.name, worst)


def test_gqa_bf16_b32_full_size_all_heads(lib):
    full_check(lib, BASE)


def test_longtail_gqa_full_size_all_heads(lib):
    full_check(lib, W.CONFIGS["longtail_gqa"])


def test_sixteen_ranks(lib):
    cfg = dataclasses.replace(BASE, B=3, lengths=[70000, 3000, 17], dcp=16, bs=16, I=1)
    wl = D.build(cfg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.decode_gqa(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, err=err)
    po, pl = lib.decode_partial_gqa(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    for b in range(cfg.B):
        exp = ref.gqa_expected(cfg, wl.seq_lens_host, b, range(cfg.Hq))
        for h in range(cfg.Hq):
            o_ref, lse_ref, po_ref, pl_ref = exp[h]
            ref.check_bf16(out[b, h], lse[b, h], o_ref, lse_ref, f"b{b} h{h}")
            for r in range(cfg.dcp):
                ref.check_bf16(po[r, b, h], pl[r, b, h], po_ref[r], pl_ref[r], f"r{r} b{b} h{h}")

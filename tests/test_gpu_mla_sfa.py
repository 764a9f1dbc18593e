"""MLA and SFA decode vs the fp64 oracle (small cases; full-size sampled)."""
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
    heads = range(cfg.Hq) if cfg.Hq <= 16 else [0, 1, 63, 64, 127]
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


def test_sfa_full_size_sampled(lib):
    wl = D.build(SFA)
    out, lse = lib.sfa_decode(wl.layout, wl.q, wl.kv, wl.topk, wl.seq_lens, SFA.scale, SFA.dv,
                              sink=wl.sink)
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    sink = wl.sink.cpu().numpy()
    rng = np.random.default_rng(4)
    for b in rng.choice(SFA.B, 4, replace=False):
        heads = sorted(rng.choice(SFA.Hq, 3, replace=False).tolist())
        exp = ref.sfa_expected(SFA, wl.seq_lens_host, wl.topk_host, int(b), heads, sink=sink)
        for h in heads:
            ref.check_bf16(out[b, h], lse[b, h], exp[h][0], exp[h][1], f"b{b} h{h}")

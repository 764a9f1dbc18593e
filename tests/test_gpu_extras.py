"""Context gather (MLA chunked prefill) and CUDA-graph replay of the decode
step with changing context lengths."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from workloads import device as D
from tests import ref

pytestmark = pytest.mark.gpu

MLA = W.CONFIGS["mla_bf16_b64"]


@pytest.mark.parametrize("dcp_size,bs,I", [(4, 64, 1), (3, 64, 16), (2, 16, 16), (8, 64, 64)])
def test_gather_context_restores_request_order(lib, dcp_size, bs, I):
    cfg = dataclasses.replace(MLA, B=3, lengths=[1, 700, 2049], dcp=dcp_size, bs=bs, I=I)
    wl = D.build(cfg)
    for b, L in enumerate(wl.seq_lens_host):
        L = int(L)
        req = torch.full((L,), b, dtype=torch.int32, device="cuda")
        pos = torch.arange(L, dtype=torch.int64, device="cuda")
        out = lib.gather_context_mla(wl.layout, wl.kv, req, pos)
        want = W.token_rows(cfg, W.T_LATENT, b, 0, L).view(np.int16)
        assert (out.view(torch.int16).cpu().numpy() == want).all()
    # any order, plus tokens that do not resolve (zero rows, counted)
    rng = np.random.default_rng(0)
    req = np.array([2, 1, 0, 2, 5, 1, -1], dtype=np.int32)
    pos = np.array([2048, 0, 0, 77, 0, 10 ** 9, 3], dtype=np.int64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lib.gather_context_mla(wl.layout, wl.kv, torch.from_numpy(req).cuda(),
                                 torch.from_numpy(pos).cuda(), err=err)
    out = out.view(torch.int16).cpu().numpy()
    for t in range(len(req)):
        if t in (4, 5, 6):
            assert (out[t] == 0).all()
        else:
            want = W.token_rows(cfg, W.T_LATENT, int(req[t]), int(pos[t]), int(pos[t]) + 1)
            assert (out[t] == want[0].view(np.int16)).all()
    assert err.item() == 3


def test_gather_context_full_size_longest_request(lib):
    wl = D.build(MLA)
    b = int(np.argmax(wl.seq_lens_host))
    L = int(wl.seq_lens_host[b])
    req = torch.full((L,), b, dtype=torch.int32, device="cuda")
    pos = torch.arange(L, dtype=torch.int64, device="cuda")
    out = lib.gather_context_mla(wl.layout, wl.kv, req, pos)
    want = W.token_rows(MLA, W.T_LATENT, b, 0, L).view(np.int16)
    assert (out.view(torch.int16).cpu().numpy() == want).all()


# ---------------------------------------------------------------------------
# graph capture: static launch parameters, lengths read from device memory
# ---------------------------------------------------------------------------

def _graph_case(lib, cfg, run, lengths_list):
    """Capture run() once at the largest lengths, replay with others; every
    replay must equal an eager call with the same lengths bit for bit."""
    wl = D.build(cfg)  # caches hold the longest contexts; shorter ones are prefixes
    out = run(wl)      # warm-up outside capture (per-process set-up)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = run(wl)
    for lens in lengths_list:
        wl.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in out]
        eager = run(wl)
        torch.cuda.synchronize()
        for a, e in zip(got, eager):
            assert torch.equal(a.view(torch.uint8), e.view(torch.uint8))
    return wl, out


def test_graph_replay_gqa_changing_lengths(lib):
    cfg = dataclasses.replace(W.CONFIGS["gqa_bf16_b32"], B=3, lengths=[5000, 3000, 900], dcp=4)
    lay = lib.Layout(cfg.dcp, cfg.bs, cfg.I)
    local = torch.empty((cfg.B, cfg.dcp), dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.decode_workspace_size(lay, lib.KIND_GQA, cfg.B, cfg.Hq, cfg.Hkv, cfg.dv),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty((cfg.B, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((cfg.B, cfg.Hq), dtype=torch.float32, device="cuda")

    def run(wl):
        lib.local_seq_lens(lay, wl.seq_lens, out=local)
        lib.decode_gqa(lay, wl.q, wl.kv, local, cfg.scale, out=o, out_lse=lse, workspace=ws)
        return [o, lse]

    lengths = [[5000, 3000, 900], [1, 2999, 17], [4096, 64, 900], [5000, 1, 1]]
    wl, _ = _graph_case(lib, cfg, run, lengths)
    # the last replayed lengths also match the oracle
    lens = lengths[-1]
    oh, lh = o.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(cfg.B):
        exp = ref.gqa_expected(cfg, lens, b, [0, 31])
        for h in (0, 31):
            ref.check_bf16(oh[b, h], lh[b, h], exp[h][0], exp[h][1], f"b{b} h{h}")


def test_graph_replay_mla_changing_lengths(lib):
    cfg = dataclasses.replace(MLA, B=2, lengths=[4000, 1500], dcp=4)
    lay = lib.Layout(cfg.dcp, cfg.bs, cfg.I)
    local = torch.empty((cfg.B, cfg.dcp), dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.decode_workspace_size(lay, lib.KIND_MLA, cfg.B, cfg.Hq, 1, cfg.dv),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty((cfg.B, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((cfg.B, cfg.Hq), dtype=torch.float32, device="cuda")

    def run(wl):
        lib.local_seq_lens(lay, wl.seq_lens, out=local)
        lib.decode_mla(lay, wl.q, wl.kv, local, cfg.scale, cfg.dv, out=o, out_lse=lse, workspace=ws)
        return [o, lse]

    lengths = [[4000, 1500], [33, 1499], [2048, 1]]
    _graph_case(lib, cfg, run, lengths)
    lens = lengths[-1]
    oh, lh = o.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(cfg.B):
        exp = ref.mla_expected(cfg, lens, b, [3])
        ref.check_bf16(oh[b, 3], lh[b, 3], exp[3][0], exp[3][1], f"b{b}")


def test_graph_replay_sfa_changing_lengths(lib):
    cfg = dataclasses.replace(W.CONFIGS["sfa_bf16_b32"], B=2, lengths=[6000, 3000], topk=256)
    lay = lib.Layout(cfg.dcp, cfg.bs, cfg.I)
    ws = torch.empty(lib.decode_workspace_size(lay, lib.KIND_SFA, cfg.B, cfg.Hq, 1, cfg.dv),
                     dtype=torch.uint8, device="cuda")
    o = torch.empty((cfg.B, cfg.Hq, cfg.dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((cfg.B, cfg.Hq), dtype=torch.float32, device="cuda")

    def run(wl):
        lib.sfa_decode(lay, wl.q, wl.kv, wl.topk, wl.seq_lens, cfg.scale, cfg.dv, sink=wl.sink,
                       out=o, out_lse=lse, workspace=ws)
        return [o, lse]

    # shorter contexts drop the selected indices beyond them
    _graph_case(lib, cfg, run, [[6000, 3000], [2000, 2999], [1, 100]])

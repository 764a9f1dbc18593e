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


@pytest.mark.parametrize("dcp_size,bs,I,cap", [(8, 64, 64, None), (4, 16, 1, None), (3, 8, 8, 5)])
def test_sfa_compaction_matches_oracle(lib, dcp_size, bs, I, cap):
    import oracle as O
    cfg = dataclasses.replace(W.CONFIGS["sfa_bf16_b32"], B=2, lengths=[5000, 700], dcp=dcp_size, topk=64,
                              bs=bs, I=I)
    wl = D.build(cfg)
    rng = np.random.default_rng(dcp_size)
    q_req = np.array([0, 1, 0, 0, 1], dtype=np.int32)
    topk = np.stack([rng.choice(int(wl.seq_lens_host[b]), 64, replace=False) for b in q_req])
    topk = topk.astype(np.int32)
    topk[1, :2] = [-1, 700]                      # padding entries
    # reference caches from the generator rows (bit patterns)
    lens = wl.seq_lens_host
    req = np.concatenate([np.full(int(L), b) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(int(L)) for L in lens])
    rows = np.concatenate([W.token_rows(cfg, W.T_LATENT, b, 0, int(L)) for b, L in enumerate(lens)])
    _, slot = O.slot_mapping(req, pos, wl.bt_host, lens, cfg.dcp, cfg.bs, cfg.I, wl.num_blocks)
    caches = O.build_caches(rows.view(np.int16), slot, cfg.dcp, wl.num_blocks, cfg.bs, -1)
    eb, eids, ecounts, eindex = O.sfa_compact_blocks(topk, q_req, lens, wl.bt_host, caches,
                                                     cfg.dcp, cfg.bs, cfg.I, wl.num_blocks)
    max_blocks = len(eids) if cap is None else cap
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    blocks, ids, counts, index = lib.sfa_compact_blocks(
        wl.layout, wl.kv, torch.from_numpy(topk).cuda(), torch.from_numpy(q_req).cuda(),
        wl.seq_lens, max_blocks, err=err)
    counts = counts.cpu().numpy()
    assert (counts == ecounts).all()
    n = min(max_blocks, len(eids))
    assert (ids.cpu().numpy()[:n] == eids[:n]).all()
    got_blocks = blocks.view(torch.int16).cpu().numpy()[:n]
    assert (got_blocks == eb[:n]).all()
    idx = index.cpu().numpy()
    want = np.where(eindex < n * cfg.bs, eindex, -1)
    assert (idx == want).all()
    assert err.item() == int(((eindex >= n * cfg.bs)).sum())


def test_replicated_window_merged_once(lib):
    """Sharded global KV (dcp=4) + a sliding window every rank holds in full
    (computed once, as a dcp=1 partial) + sink, merged by dcp_lse_merge_swa."""
    import oracle as O
    glob = dataclasses.replace(W.CONFIGS["gqa_bf16_b32"], B=3, lengths=[3000, 40, 900], dcp=4)
    win = dataclasses.replace(glob, lengths=[128, 7, 128], dcp=1, bs=16, I=1, seed=77)
    wg, ww = D.build(glob), D.build(win)
    ww.q.copy_(wg.q)  # the same query attends both key sets
    po, pl = lib.decode_partial_gqa(wg.layout, wg.q, wg.kv, wg.local_lens, glob.scale)
    so, sl = lib.decode_partial_gqa(ww.layout, ww.q, ww.kv, ww.local_lens, win.scale)
    sink = torch.from_numpy(np.linspace(-1, 2, glob.Hq).astype(np.float32)).cuda()
    out, lse = lib.lse_merge_swa(po, pl, so[0].contiguous(), sl[0].contiguous(), sink)
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    s_host = sink.cpu().numpy()
    G = glob.Hq // glob.Hkv
    for b in range(glob.B):
        for h in (0, 9, 31):
            exp = ref.gqa_expected(glob, wg.seq_lens_host, b, [h])[h]
            Kw, Vw = ref.gqa_kv(win, b, h // G, int(ww.seq_lens_host[b]))
            ow, lw = O.attention(ref.q_vec(glob, b, h), Kw, Vw, glob.scale)
            o_ref, lse_ref = O.lse_merge(np.vstack([exp[2], ow]), list(exp[3]) + [lw],
                                         sink=float(s_host[h]))
            ref.check_bf16(out[b, h], lse[b, h], o_ref, lse_ref, f"b{b} h{h}")


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

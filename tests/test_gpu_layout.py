"""Integer steps on the GPU vs the oracle, bit for bit: per-rank context
lengths, slot mapping with owner masking, and the SFA global->local remap."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

LAYOUTS = [(1, 16, 1), (2, 16, 1), (2, 4, 2), (3, 16, 4), (8, 16, 1), (8, 64, 64), (8, 64, 1),
           (4, 8, 8), (16, 16, 16), (5, 12, 3)]


def cu(a, dt):
    return torch.from_numpy(np.ascontiguousarray(a).astype(dt)).cuda()


@pytest.mark.parametrize("dcp_size,bs,I", LAYOUTS)
def test_local_seq_lens(lib, dcp_size, bs, I):
    lens = [0, 1, 2, I, bs, bs * dcp_size - 1, bs * dcp_size, bs * dcp_size + 1, 977, 262144,
            1048576, 3 * bs * dcp_size + I + 1]
    L = lib.Layout(dcp_size, bs, I)
    out = lib.local_seq_lens(L, cu(lens, np.int32)).cpu().numpy()
    assert (out == O.local_seq_lens(lens, dcp_size, bs, I)).all()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lib.local_seq_lens(L, cu([-5, 3], np.int32), err=err).cpu().numpy()
    assert out[0].sum() == 0 and err.item() == 1


@pytest.mark.parametrize("dcp_size,bs,I", LAYOUTS)
def test_slot_mapping(lib, dcp_size, bs, I):
    rng = np.random.default_rng(dcp_size * 1000 + bs + I)
    lens = np.array([1, 2, bs * dcp_size, 5 * bs * dcp_size + 3, int(rng.integers(1, 3000))])
    bt, nb = W.make_block_tables(lens, dcp_size, bs, "random", seed=dcp_size + bs)
    req = np.concatenate([np.full(n, b) for b, n in enumerate(lens)])
    pos = np.concatenate([np.arange(n) for n in lens])
    perm = rng.permutation(len(req))
    req, pos = req[perm], pos[perm]
    L = lib.Layout(dcp_size, bs, I)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rk, sl = lib.slot_mapping(L, cu(req, np.int32), cu(pos, np.int64), cu(bt, np.int32), nb,
                              err=err)
    erk, esl = O.slot_mapping(req, pos, bt, lens, dcp_size, bs, I, nb)
    assert (rk.cpu().numpy() == erk).all()
    assert (sl.cpu().numpy() == esl).all()
    assert err.item() == 0
    # invalid tokens: bad request, negative position, beyond the table, bad table entry
    bt2 = bt.copy()
    bt2[0, 0, 0] = nb + 7
    bad_req = np.array([-1, len(lens), 0, 0, 0])
    bad_pos = np.array([0, 0, -3, 10 ** 12, 0])
    rk, sl = lib.slot_mapping(L, cu(bad_req, np.int32), cu(bad_pos, np.int64), cu(bt2, np.int32),
                              nb, err=err)
    erk, esl = O.slot_mapping(bad_req, bad_pos, bt2, lens, dcp_size, bs, I, nb)
    assert (rk.cpu().numpy() == erk).all() and (sl.cpu().numpy() == esl).all()
    assert err.item() == int((erk < 0).sum())


def test_slot_mapping_shared_table(lib):
    lens = np.array([300, 77])
    bt, nb = W.make_block_tables(lens, 4, 16, "random", seed=1)
    shared = bt[0]
    req = np.concatenate([np.full(n, b) for b, n in enumerate(lens)])
    pos = np.concatenate([np.arange(n) for n in lens])
    L = lib.Layout(4, 16, 2)
    rk, sl = lib.slot_mapping(L, cu(req, np.int32), cu(pos, np.int64), cu(shared, np.int32), nb)
    erk, esl = O.slot_mapping(req, pos, np.broadcast_to(shared, (4,) + shared.shape), lens, 4, 16,
                              2, nb)
    assert (rk.cpu().numpy() == erk).all() and (sl.cpu().numpy() == esl).all()


@pytest.mark.parametrize("dcp_size,bs,I", [(8, 64, 64), (4, 16, 1), (3, 8, 4)])
def test_sfa_remap(lib, dcp_size, bs, I):
    rng = np.random.default_rng(7)
    lens = np.array([5000, 1, 700, 64])
    bt, nb = W.make_block_tables(lens, dcp_size, bs, "random", seed=3)
    K = 64
    topk = np.stack([rng.choice(max(n, K), K, replace=False) for n in lens]).astype(np.int32)
    topk[1, :3] = [-1, 0, 1]   # padding and out-of-range entries
    topk[2, 5] = 700
    L = lib.Layout(dcp_size, bs, I)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rk, sl = lib.sfa_remap(L, cu(topk, np.int32), cu(lens, np.int32), cu(bt, np.int32), nb,
                           err=err)
    erk, esl = O.sfa_remap(topk, lens, bt, dcp_size, bs, I, nb)
    assert (rk.cpu().numpy() == erk).all() and (sl.cpu().numpy() == esl).all()
    assert err.item() == 0


def test_sfa_remap_full_config(lib):
    cfg = W.CONFIGS["sfa_bf16_b32"]
    lens = W.make_seq_lens(cfg)
    topk = W.make_topk(cfg, lens)
    bt, nb = W.make_block_tables(lens, cfg.dcp, cfg.bs, "random", seed=cfg.seed)
    L = lib.Layout(cfg.dcp, cfg.bs, cfg.I)
    rk, sl = lib.sfa_remap(L, cu(topk, np.int32), cu(lens, np.int32), cu(bt, np.int32), nb)
    erk, esl = O.sfa_remap(topk[:4], lens[:4], bt, cfg.dcp, cfg.bs, cfg.I, nb)
    assert (rk.cpu().numpy()[:4] == erk).all() and (sl.cpu().numpy()[:4] == esl).all()
    assert (rk.cpu().numpy() >= 0).all()

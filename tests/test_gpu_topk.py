"""Exact distributed top-k (local candidates per rank + merge) vs the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu


def make_scores(lens, dcp, bs, I, seed, nan_frac=0.01, coarse=False):
    """Global scores per request (quantised N(0,1): many ties), and the
    per-rank local score array [dcp, B, max_local] built from them."""
    rng = np.random.default_rng(seed)
    glob = []
    for b, L in enumerate(lens):
        s = W.stream_values(seed, W.T_Q, 1000 + b, 0, int(L), "f32").copy()
        if coarse:
            s = np.round(s * 4) / 4
        s[rng.random(int(L)) < nan_frac] = np.nan
        glob.append(s.astype(np.float32))
    local_lens = O.local_seq_lens(lens, dcp, bs, I)
    max_local = max(1, int(local_lens.max()))
    loc = np.full((dcp, len(lens), max_local), np.inf, dtype=np.float32)  # never read
    for b in range(len(lens)):
        for r in range(dcp):
            n = int(local_lens[b, r])
            x = O.global_token(np.arange(n), r, bs, dcp, I)
            loc[r, b, :n] = glob[b][x]
    return glob, loc, local_lens.astype(np.int32)


def decode_keys(keys):
    keys = keys.astype(np.uint64)
    ids = np.where(keys != 0, (np.uint64(0xFFFFFFFF) - (keys & np.uint64(0xFFFFFFFF))), 0)
    return np.where(keys != 0, ids.astype(np.int64), -1)


@pytest.mark.parametrize("dcp_size,bs,I,lens,k,coarse", [
    (8, 64, 64, [40000, 3000, 100], 2048, False),
    (4, 16, 1, [5000, 17, 800], 256, True),
    (3, 8, 4, [999, 1000], 999, True),
    (2, 16, 16, [70000], 4096, False),
])
def test_topk_matches_oracle(lib, dcp_size, bs, I, lens, k, coarse):
    glob, loc, local_lens = make_scores(lens, dcp_size, bs, I, seed=k + dcp_size, coarse=coarse)
    layout = lib.Layout(dcp_size, bs, I)
    loc_d = torch.from_numpy(loc).cuda()
    ll_d = torch.from_numpy(local_lens).cuda()
    ids, scores = lib.topk(layout, loc_d, ll_d, k)
    cand = lib.topk_local(layout, loc_d, ll_d, k)
    ids2, scores2 = lib.topk_merge(cand)
    ids, scores = ids.cpu().numpy(), scores.cpu().numpy()
    assert (ids == ids2.cpu().numpy()).all()
    cand = cand.cpu().numpy().view(np.uint64)
    for b, L in enumerate(lens):
        want_ids, want_scores = O.topk_exact(glob[b], np.arange(L), k)
        n = len(want_ids)
        assert (ids[b, :n] == want_ids).all()
        assert (ids[b, n:] == -1).all()
        # NaN is reported as -inf and -0 as +0 (equal scores)
        ws = np.where(np.isnan(want_scores), -np.inf, want_scores).astype(np.float32) + 0.0
        assert (scores[b, :n].view(np.uint32) == ws.view(np.uint32)).all()
        # each rank's candidates are its own exact local top-k
        for r in range(dcp_size):
            li, _ = O.topk_local(loc[r, b], local_lens[b, r], r, k, dcp_size, bs, I)
            got = decode_keys(cand[r, b])
            assert (got[:len(li)] == li).all() and (got[len(li):] == -1).all()

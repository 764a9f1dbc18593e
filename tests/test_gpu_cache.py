"""Owner-masked cache writes vs the oracle's caches, byte for byte."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from workloads import device as D

pytestmark = pytest.mark.gpu


def token_major(pool, kind):
    """GPU pool -> [num_blocks*bs, row] (HND pools are transposed to token-major)."""
    if kind == "gqa":
        nb, H, bs, d = pool.shape
        return pool.permute(0, 2, 1, 3).reshape(nb * bs, H * d)
    nb, bs, d = pool.shape
    return pool.reshape(nb * bs, d)


def bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32).cpu().numpy()


def expected_caches(cfg, wl):
    lens = wl.seq_lens_host
    tensors = [W.T_K, W.T_V] if cfg.kind == "gqa" else [W.T_LATENT]
    req = np.concatenate([np.full(n, b) for b, n in enumerate(lens)])
    pos = np.concatenate([np.arange(n) for n in lens])
    _, slot = O.slot_mapping(req, pos, wl.bt_host, lens, cfg.dcp, cfg.bs, cfg.I, wl.num_blocks)
    out = []
    for t in tensors:
        rows = np.concatenate([W.token_rows(cfg, t, b, 0, int(n)) for b, n in enumerate(lens)])
        rows = rows.view(np.int16 if cfg.dtype == "bf16" else np.int32)
        out.append(O.build_caches(rows, slot, cfg.dcp, wl.num_blocks, cfg.bs, -1))
    return out


CASES = [
    W.CONFIGS["tiny_gqa_f32"],
    dataclasses.replace(W.CONFIGS["tiny_gqa_f32"], perm="identity"),
    dataclasses.replace(W.CONFIGS["gqa_bf16_b32"], B=3, lengths=[1, 515, 2000], dcp=4, bs=16, I=4),
    dataclasses.replace(W.CONFIGS["mla_bf16_b64"], B=3, lengths=[3, 130, 700], dcp=3, bs=64, I=8),
    dataclasses.replace(W.CONFIGS["sfa_bf16_b32"], B=2, lengths=[1000, 64], topk=16),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"{c.name}-{c.dcp}-{c.bs}-{c.I}-{c.perm}")
def test_cache_bytes_match_oracle(lib, cfg):
    wl = D.build(cfg)
    torch.cuda.synchronize()
    exp = expected_caches(cfg, wl)
    pools = [wl.k_pools, wl.v_pools] if cfg.kind == "gqa" else [wl.k_pools]
    for e, plist in zip(exp, pools):
        for r in range(cfg.dcp):
            got = bits(token_major(plist[r], cfg.kind))
            assert (got == e[r]).all(), f"rank {r} differs"


def test_cache_full_size_sampled_rows(lib):
    cfg = W.CONFIGS["gqa_bf16_b32"]
    wl = D.build(cfg)
    torch.cuda.synchronize()
    lens = wl.seq_lens_host
    rng = np.random.default_rng(0)
    local = wl.local_lens.cpu().numpy()
    for r in range(cfg.dcp):
        # every owned (slot, head) row written exactly once, nothing else touched
        for pools in (wl.k_pools, wl.v_pools):
            written = (pools[r].view(torch.int16) != -1).any(dim=-1).sum().item()
            assert written == cfg.Hkv * int(local[:, r].sum())
    for _ in range(300):
        b = int(rng.integers(0, cfg.B))
        x = int(rng.integers(0, lens[b]))
        rk, sl = O.slot_mapping([b], [x], wl.bt_host, lens, cfg.dcp, cfg.bs, cfg.I, wl.num_blocks)
        r, s = int(rk[0]), int(sl[rk[0], 0])
        for t, pools in ((W.T_K, wl.k_pools), (W.T_V, wl.v_pools)):
            blk, off = divmod(s, cfg.bs)
            got = pools[r][blk, :, off, :].reshape(-1).view(torch.int16).cpu().numpy()
            want = W.token_rows(cfg, t, b, x, x + 1)[0].view(np.int16)
            assert (got == want).all()


def test_synth_generator_matches_numpy(lib):
    for dt in ("bf16", "f32"):
        out = torch.empty(100003, dtype=D.torch_dtype(dt), device="cuda")
        D.fill(out, 11, W.T_V, 5, 123456789, dt)
        want = W.stream_values(11, W.T_V, 5, 123456789, 100003, dt)
        got = out.view(torch.int16 if dt == "bf16" else torch.float32).cpu().numpy()
        if dt == "bf16":
            assert (got.view(np.uint16) == want).all()
        else:
            assert (got == want).all()

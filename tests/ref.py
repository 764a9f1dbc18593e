"""Expected values from the CPU oracle for the parity tests (CPU side only).

Inputs are regenerated from the seeded numpy generator of ``workloads``;
nothing here reads a GPU result.
"""
from __future__ import annotations

import numpy as np

import oracle as O
import workloads as W


def q_vec(cfg, b, h):
    return W.as_float64(W.query(cfg, b)[h], cfg.dtype)


def gqa_kv(cfg, b, g, L):
    K = W.as_float64(W.head_rows(cfg, W.T_K, b, g, 0, L), cfg.dtype)
    V = W.as_float64(W.head_rows(cfg, W.T_V, b, g, 0, L), cfg.dtype)
    return K, V


def latent_kv(cfg, b, L):
    rows = W.as_float64(W.token_rows(cfg, W.T_LATENT, b, 0, L), cfg.dtype)
    return rows, rows[:, :cfg.dv]


def gqa_expected(cfg, lens, b, heads, sink=None):
    """{h: (o, lse, per_rank_o, per_rank_lse)} for request b (fp64)."""
    L = int(lens[b])
    G = cfg.Hq // cfg.Hkv
    out = {}
    cache = {}
    for h in heads:
        g = h // G
        if g not in cache:
            cache[g] = gqa_kv(cfg, b, g, L)
        K, V = cache[g]
        s = None if sink is None else float(sink[h])
        out[h] = O.sharded_attention(q_vec(cfg, b, h), K, V, cfg.scale, L, cfg.dcp, cfg.bs, cfg.I,
                                     sink=s)
    return out


def mla_expected(cfg, lens, b, heads, sink=None):
    L = int(lens[b])
    K, V = latent_kv(cfg, b, L)
    out = {}
    for h in heads:
        s = None if sink is None else float(sink[h])
        out[h] = O.sharded_attention(q_vec(cfg, b, h), K, V, cfg.scale, L, cfg.dcp, cfg.bs, cfg.I,
                                     sink=s)
    return out


def sfa_expected(cfg, lens, topk, b, heads, sink=None):
    L = int(lens[b])
    K, V = latent_kv(cfg, b, L)
    out = {}
    for h in heads:
        s = None if sink is None else float(sink[h])
        out[h] = O.sfa_sharded(q_vec(cfg, b, h), K, V, cfg.scale, topk[b], L, cfg.dcp, cfg.bs,
                               cfg.I, sink=s)
    return out


# tolerances (stated by the workload spec): fp32 1e-5 relative; bf16 2e-2 abs on
# the output and 1e-3 abs on the LSE
def check_f32(o, lse, o_ref, lse_ref, what=""):
    o = np.asarray(o, dtype=np.float64)
    scale = max(float(np.abs(o_ref).max()), 1e-30)
    err = float(np.abs(o - o_ref).max())
    assert err <= 1e-5 * scale, f"{what}: max|do| {err:.3e} > 1e-5 * {scale:.3e}"
    if np.isneginf(lse_ref):
        assert np.isneginf(lse), f"{what}: lse {lse} != -inf"
    else:
        assert abs(float(lse) - lse_ref) <= 1e-5 * max(abs(lse_ref), 1.0), \
            f"{what}: lse {lse} vs {lse_ref}"


def check_bf16(o, lse, o_ref, lse_ref, what=""):
    o = np.asarray(o, dtype=np.float64)
    err = float(np.abs(o - o_ref).max())
    assert err <= 2e-2, f"{what}: max|do| {err:.3e} > 2e-2"
    if np.isneginf(lse_ref):
        assert np.isneginf(lse), f"{what}: lse {lse} != -inf"
    else:
        assert abs(float(lse) - lse_ref) <= 1e-3, f"{what}: lse {lse} vs {lse_ref}"

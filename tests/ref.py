"""Expected values from the CPU oracle for the parity tests (CPU side only),
and the checks that compare a GPU result with them.

Inputs are regenerated from the seeded numpy generator of ``workloads``;
nothing here reads a GPU result.
"""
from __future__ import annotations

import numpy as np

import oracle as O
import workloads as W


def q_vec(cfg, b, h):
    return W.as_float64(W.query(cfg, b)[h], cfg.dtype)


def q_rows(cfg, b, heads):
    return W.as_float64(W.query(cfg, b)[list(heads)], cfg.dtype)


def gqa_kv(cfg, b, g, L):
    K = W.as_float64(W.head_rows(cfg, W.T_K, b, g, 0, L), cfg.dtype)
    V = W.as_float64(W.head_rows(cfg, W.T_V, b, g, 0, L), cfg.dtype)
    return K, V


def latent_kv(cfg, b, L):
    rows = W.as_float64(W.token_rows(cfg, W.T_LATENT, b, 0, L), cfg.dtype)
    return rows, rows[:, :cfg.dv]


def _unpack(heads, res):
    o, lse, po, pl = res
    return {h: (o[i], float(lse[i]), po[:, i], pl[:, i]) for i, h in enumerate(heads)}


def gqa_expected(cfg, lens, b, heads, sink=None):
    """{h: (o, lse, per_rank_o[dcp, dv], per_rank_lse[dcp])} for request b (fp64)."""
    L = int(lens[b])
    G = cfg.Hq // cfg.Hkv
    heads = sorted(set(int(h) for h in heads))
    out = {}
    for g in sorted(set(h // G for h in heads)):
        hs = [h for h in heads if h // G == g]
        K, V = gqa_kv(cfg, b, g, L)
        sinks = None if sink is None else [float(sink[h]) for h in hs]
        out.update(_unpack(hs, O.sharded_attention_heads(q_rows(cfg, b, hs), K, V, cfg.scale, L,
                                                         cfg.dcp, cfg.bs, cfg.I, sinks=sinks)))
    return out


def mla_expected(cfg, lens, b, heads, sink=None):
    L = int(lens[b])
    heads = sorted(set(int(h) for h in heads))
    K, V = latent_kv(cfg, b, L)
    sinks = None if sink is None else [float(sink[h]) for h in heads]
    return _unpack(heads, O.sharded_attention_heads(q_rows(cfg, b, heads), K, V, cfg.scale, L,
                                                    cfg.dcp, cfg.bs, cfg.I, sinks=sinks))


def sfa_expected(cfg, lens, topk, b, heads, sink=None):
    """Only the selected tokens' rows are generated (invalid entries get a
    placeholder row that the oracle drops)."""
    L = int(lens[b])
    heads = sorted(set(int(h) for h in heads))
    sel = np.asarray(topk[b], dtype=np.int64)
    rows = W.as_float64(W.token_rows_at(cfg, W.T_LATENT, b, np.clip(sel, 0, None)), cfg.dtype)
    sinks = None if sink is None else [float(sink[h]) for h in heads]
    return _unpack(heads, O.sfa_sharded_heads(q_rows(cfg, b, heads), sel, rows, rows[:, :cfg.dv],
                                              cfg.scale, L, cfg.dcp, cfg.bs, cfg.I, sinks=sinks))


# ---------------------------------------------------------------------------
# checks
# ---------------------------------------------------------------------------
# Stated bounds: fp32 1e-5 relative; bf16 2e-2 absolute on the output and
# 1e-3 absolute on the LSE.  The bf16 absolute output bound alone cannot fail
# on long contexts, where a head's whole output is below 2e-2 (the average of
# ~100k N(0,1) value rows), so every bf16 check also applies a bound relative
# to the output vector's own scale: max|o - o_ref| <= BF16_REL * max|o_ref|
# for each (request, head) vector.  The kernels' own rounding (bf16
# probabilities in P.V, bf16 rounding of the final output) stays below
# ~4e-3 of that scale; a dropped split, a wrong value page or KV head, or a
# zero output exceeds it.
BF16_ABS_O = 2e-2
BF16_ABS_LSE = 1e-3
BF16_REL = 1e-2
F32_REL = 1e-5


def rel_err(o, o_ref):
    """max|o - o_ref| / max|o_ref| (0 when both are all zero, inf when only o_ref is)."""
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    err = float(np.abs(o - o_ref).max())
    scale = float(np.abs(o_ref).max())
    if scale == 0.0:
        return 0.0 if err == 0.0 else float("inf")
    return err / scale


def _check_lse(lse, lse_ref, tol, what):
    if np.isneginf(lse_ref):
        assert np.isneginf(lse), f"{what}: lse {lse} != -inf"
    else:
        assert abs(float(lse) - lse_ref) <= tol, f"{what}: lse {lse} vs {lse_ref}"


def check_f32(o, lse, o_ref, lse_ref, what=""):
    o = np.asarray(o, dtype=np.float64)
    scale = max(float(np.abs(o_ref).max()), 1e-30)
    err = float(np.abs(o - o_ref).max())
    assert err <= F32_REL * scale, f"{what}: max|do| {err:.3e} > 1e-5 * {scale:.3e}"
    _check_lse(lse, lse_ref, F32_REL * max(abs(lse_ref), 1.0) if np.isfinite(lse_ref) else 0,
               what)


def check_bf16(o, lse, o_ref, lse_ref, what=""):
    o = np.asarray(o, dtype=np.float64)
    err = float(np.abs(o - o_ref).max())
    assert err <= BF16_ABS_O, f"{what}: max|do| {err:.3e} > 2e-2"
    r = rel_err(o, o_ref)
    assert r <= BF16_REL, (f"{what}: max|do| {err:.3e} is {r:.3e} of max|o_ref| "
                           f"{float(np.abs(o_ref).max()):.3e} (bound {BF16_REL})")
    _check_lse(lse, lse_ref, BF16_ABS_LSE, what)


def check(cfg, o, lse, o_ref, lse_ref, what=""):
    (check_f32 if cfg.dtype == "f32" else check_bf16)(o, lse, o_ref, lse_ref, what)


def expected_for_requests(fn, reqs, workers=4):
    """[(b, fn(b))] for every request b, computed by a few threads (numpy
    releases the GIL in the generator and the products)."""
    from concurrent.futures import ThreadPoolExecutor
    reqs = [int(b) for b in reqs]
    with ThreadPoolExecutor(max_workers=max(1, min(workers, len(reqs)))) as ex:
        return list(zip(reqs, ex.map(fn, reqs)))


class WorstError:
    """Largest relative output error seen (reported by the full-size tests)."""

    def __init__(self):
        self.fused = 0.0
        self.partial = 0.0

    def add(self, o, o_ref, partial=False):
        r = rel_err(o, o_ref)
        if partial:
            self.partial = max(self.partial, r)
        else:
            self.fused = max(self.fused, r)

    def __str__(self):
        return (f"worst max|do|/max|o_ref|: fused {self.fused:.2e}, per-rank partials "
                f"{self.partial:.2e} (bound {BF16_REL})")

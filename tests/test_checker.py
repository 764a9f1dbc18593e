"""The bf16 parity check can fail at full size.

On a long context every element of a head's output is far below the stated
2e-2 absolute output bound (the output averages ~100k N(0,1) value rows), so
that bound alone passes an all-zero output.  These CPU tests build a
full-size-like case with the oracle, plant the mistakes a decode kernel could
make (in the oracle's result, never on the GPU) and check that
``ref.check_bf16`` rejects each one, while a result carrying the kernels' own
rounding (bf16 probabilities in P.V, a bf16 output) passes.
"""
import numpy as np
import pytest

import oracle as O
from tests import ref

DCP, BS, I = 8, 16, 1
D, G = 128, 4
SCALE = 1.0 / np.sqrt(D)


def bf16(x):
    """Round to the nearest bf16 value (ties to even), returned as fp64."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


@pytest.fixture(scope="module")
def case():
    rng = np.random.default_rng(7)
    L = 200_000
    Q = bf16(rng.standard_normal((G, D)))
    K = bf16(rng.standard_normal((L, D)))
    V = bf16(rng.standard_normal((L, D)))
    V_other = bf16(rng.standard_normal((L, D)))      # another KV head's values
    o, lse, po, pl = O.sharded_attention_heads(Q, K, V, SCALE, L, DCP, BS, I)
    return dict(L=L, Q=Q, K=K, V=V, V_other=V_other, o=o, lse=lse, po=po, pl=pl)


def kernel_like(Q, K, V, L):
    """The decode kernels' rounding: fp32 scores, probabilities rounded to
    bf16 before P.V (the row sum taken on the unrounded fp32 values), fp32
    partials, merge in fp32, output rounded to bf16."""
    po = np.zeros((DCP, G, D))
    pl = np.full((DCP, G), -np.inf)
    for r in range(DCP):
        idx = O.shard_tokens(L, r, DCP, BS, I)
        s = (SCALE * (K[idx] @ Q.T)).astype(np.float32)
        m = s.max(axis=0)
        p = np.exp(s - m).astype(np.float32)
        ls = p.sum(axis=0, dtype=np.float32)
        po[r] = ((bf16(p).T @ V[idx]) / ls[:, None]).astype(np.float32)
        pl[r] = m + np.log(ls)
    o = np.zeros((G, D))
    lse = np.zeros(G)
    for h in range(G):
        o[h], lse[h] = O.lse_merge(po[:, h], pl[:, h])
    return bf16(o), lse.astype(np.float32), po, pl


def rejects(o, lse, o_ref, lse_ref):
    with pytest.raises(AssertionError):
        ref.check_bf16(o, lse, o_ref, lse_ref, "planted")


def test_output_scale_is_below_the_absolute_bound(case):
    """Why the relative bound is needed: zeros pass the absolute bounds alone."""
    o = case["o"]
    assert np.abs(o).max() < ref.BF16_ABS_O
    assert np.abs(np.zeros_like(o) - o).max() <= ref.BF16_ABS_O


def test_kernel_rounding_passes(case):
    o, lse, po, pl = kernel_like(case["Q"], case["K"], case["V"], case["L"])
    for h in range(G):
        ref.check_bf16(o[h], lse[h], case["o"][h], case["lse"][h], f"h{h}")
        assert ref.rel_err(o[h], case["o"][h]) < 0.5 * ref.BF16_REL
        for r in range(DCP):
            ref.check_bf16(po[r, h], pl[r, h], case["po"][r, h], case["pl"][r, h], f"r{r} h{h}")


def test_zero_output_is_rejected(case):
    for h in range(G):
        rejects(np.zeros(D), case["lse"][h], case["o"][h], case["lse"][h])


def test_wrong_kv_heads_values_are_rejected(case):
    o, lse, _, _ = O.sharded_attention_heads(case["Q"], case["K"], case["V_other"], SCALE,
                                             case["L"], DCP, BS, I)
    for h in range(G):
        assert abs(lse[h] - case["lse"][h]) == 0       # the LSE cannot see the values
        rejects(o[h], lse[h], case["o"][h], case["lse"][h])


def test_dropped_split_is_rejected(case):
    """One split of 1/16 of a rank's tokens (~1,560 of 200,000) missing from
    the merge, in the output only (the LSE left correct)."""
    L, r = case["L"], 3
    idx = O.shard_tokens(L, r, DCP, BS, I)
    keep = np.ones(L, dtype=bool)
    n = len(idx) // 16
    keep[idx[5 * n:6 * n]] = False
    o, _, _, _ = O.sharded_attention_heads(case["Q"], case["K"][keep], case["V"][keep], SCALE,
                                           int(keep.sum()), DCP, BS, I)
    for h in range(G):
        rejects(o[h], case["lse"][h], case["o"][h], case["lse"][h])


def test_dropped_rank_is_rejected(case):
    for h in range(G):
        o, lse = O.lse_merge(case["po"][1:, h], case["pl"][1:, h])
        rejects(o, case["lse"][h], case["o"][h], case["lse"][h])
        rejects(case["o"][h], lse, case["o"][h], case["lse"][h])


def test_wrong_value_page_is_rejected_on_a_short_context():
    """One 16-token value page read from the wrong block (L = 2,000)."""
    rng = np.random.default_rng(8)
    L = 2000
    Q, K, V = (bf16(rng.standard_normal(s)) for s in ((G, D), (L, D), (L, D)))
    o, lse, _, _ = O.sharded_attention_heads(Q, K, V, SCALE, L, DCP, BS, I)
    Vbad = V.copy()
    Vbad[160:176] = V[1600:1616]
    ob, lb, _, _ = O.sharded_attention_heads(Q, K, Vbad, SCALE, L, DCP, BS, I)
    for h in range(G):
        rejects(ob[h], lb[h], o[h], lse[h])


def test_sign_error_in_the_scores_is_rejected(case):
    o, lse, _, _ = O.sharded_attention_heads(-case["Q"], case["K"], case["V"], SCALE, case["L"],
                                             DCP, BS, I)
    for h in range(G):
        rejects(o[h], case["lse"][h], case["o"][h], case["lse"][h])

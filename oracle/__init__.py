"""CPU oracle for the DCP decode hot path.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never calls it.  It shares no code with the CUDA path:
both sides see only the seeded inputs from the ``workloads`` module.

Everything here is plain numpy, fp64 for floating point, written directly
from the definitions on the pages it cites:

* "Decode Context Parallel (DCP)" (docs.vllm.ai, vLLM Ascend design docs),
  section "KV-cache layout": the four token -> (virtual block, offset, local
  block, rank) formulas and the ``block_size % interleave == 0`` constraint;
  section "Backend structure": the per-rank context-length matrix and the
  partial-output / LSE merge; sections "Decode" and "GLM-5.2 SFA DCP
  replicated indexer": attention over the local shard, and the remap of
  global top-k indices to local KV indices.
* "DeepSeek V4.1 context parallelism" (lightseek.org TokenSpeed design),
  section "Cache ownership": writes translate virtual slots to local slots
  and mask non-owners; section "Decode computation": the attention sink is
  applied once when the partials are merged by log-sum-exp.

Readings where the pages are silent:

* local in-block offset of token x on its rank:
  ``loc = (local_block_index // dcp) * I + offset_in_virtual_block % I`` and
  local position ``vb * block_size + loc``; the slot is
  ``BT[rank][b][vb] * block_size + loc``;
* LSE is the natural log of the sum of exp of the *scaled* scores;
* an empty shard has ``lse = -inf`` and ``o = 0``;
* the sink is one logit per query head, in scaled-score units, with a zero
  value vector.

Parity status: every function below is pinned by ``tests/test_oracle_pins.py``
(brute-force enumeration, closed forms, library routines, invariants).
"""
from __future__ import annotations

import math

import numpy as np

NEG_INF = float("-inf")


# ---------------------------------------------------------------------------
# KV-cache layout ("Decode Context Parallel (DCP)", section "KV-cache layout")
# ---------------------------------------------------------------------------

def check_layout(dcp: int, bs: int, I: int) -> None:
    """The page requires block_size % cp_kv_cache_interleave_size == 0."""
    if dcp < 1 or bs < 1 or I < 1 or bs % I != 0:
        raise ValueError(f"invalid DCP layout dcp={dcp} block_size={bs} interleave={I}")


def virtual_block_index(x, bs, dcp):
    return x // (bs * dcp)


def offset_in_virtual_block(x, bs, dcp):
    return x % (bs * dcp)


def local_block_index(x, bs, dcp, I):
    return offset_in_virtual_block(x, bs, dcp) // I


def target_rank(x, bs, dcp, I):
    return local_block_index(x, bs, dcp, I) % dcp


def local_offset(x, bs, dcp, I):
    """Offset of token x inside its rank's physical block (reading, see module doc)."""
    return (local_block_index(x, bs, dcp, I) // dcp) * I + offset_in_virtual_block(x, bs, dcp) % I


def local_position(x, bs, dcp, I):
    """Position of token x in its rank's local sequence shard."""
    return virtual_block_index(x, bs, dcp) * bs + local_offset(x, bs, dcp, I)


def global_token(p, r, bs, dcp, I):
    """Inverse of (target_rank, local_position): local position p on rank r -> token x."""
    vb, loc = p // bs, p % bs
    lbi = (loc // I) * dcp + r
    return vb * bs * dcp + lbi * I + loc % I


def local_seq_lens(seq_lens, dcp, bs, I) -> np.ndarray:
    """Per-rank context-length matrix [B, dcp], counted by enumerating every token.

    ("Backend structure": the DCP metadata owns the per-rank context-length matrix.)
    """
    check_layout(dcp, bs, I)
    out = np.zeros((len(seq_lens), dcp), dtype=np.int64)
    for b, L in enumerate(seq_lens):
        x = np.arange(int(L), dtype=np.int64)
        out[b] = np.bincount(target_rank(x, bs, dcp, I), minlength=dcp)
    return out


def local_seq_len_closed_form(L, r, dcp, bs, I):
    """Closed form for the number of tokens x < L owned by rank r."""
    full, rem = L // (bs * dcp), L % (bs * dcp)
    c, p = rem // I, rem % I
    return full * bs + (c // dcp) * I + (I if c % dcp > r else 0) + (p if c % dcp == r else 0)


def slot_mapping(req, pos, block_table, seq_lens_unused, dcp, bs, I, num_blocks):
    """Token -> (owner rank, per-rank slot with -1 on non-owners).

    req[T], pos[T]: request index and global position of each token.
    block_table[dcp][B][max_vb]: physical block of virtual block vb on rank r.
    Invalid tokens (request out of range, pos < 0, virtual block beyond the
    table, or a table entry outside [0, num_blocks)) get rank -1 and no slot.
    ("KV-cache layout"; "Cache ownership": translate virtual slots to local
    slots and mask non-owners.)
    """
    check_layout(dcp, bs, I)
    req = np.asarray(req, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    T = len(req)
    B, max_vb = block_table.shape[1], block_table.shape[2]
    rank = np.full(T, -1, dtype=np.int64)
    slot = np.full((dcp, T), -1, dtype=np.int64)
    for t in range(T):
        b, x = int(req[t]), int(pos[t])
        if b < 0 or b >= B or x < 0:
            continue
        vb = virtual_block_index(x, bs, dcp)
        if vb >= max_vb:
            continue
        r = target_rank(x, bs, dcp, I)
        phys = int(block_table[r, b, vb])
        if phys < 0 or phys >= num_blocks:
            continue
        rank[t] = r
        slot[r, t] = phys * bs + local_offset(x, bs, dcp, I)
    return rank, slot


def sfa_remap(topk, seq_lens, block_table, dcp, bs, I, num_blocks):
    """Global top-k token indices -> (rank, local slot); invalid entries -> (-1, -1).

    ("GLM-5.2 SFA DCP replicated indexer": global indices from the replicated
    indexer view are remapped to local KV indices before SFA runs.)
    """
    B, K = topk.shape
    rank = np.full((B, K), -1, dtype=np.int64)
    slot = np.full((B, K), -1, dtype=np.int64)
    for b in range(B):
        for k in range(K):
            g = int(topk[b, k])
            if g < 0 or g >= int(seq_lens[b]):
                continue
            vb = virtual_block_index(g, bs, dcp)
            if vb >= block_table.shape[2]:
                continue
            r = target_rank(g, bs, dcp, I)
            phys = int(block_table[r, b, vb])
            if phys < 0 or phys >= num_blocks:
                continue
            rank[b, k] = r
            slot[b, k] = phys * bs + local_offset(g, bs, dcp, I)
    return rank, slot


# ---------------------------------------------------------------------------
# owner-masked paged cache ("Cache ownership")
# ---------------------------------------------------------------------------

def build_caches(rows, slot, dcp, num_blocks, bs, sentinel):
    """Per-rank paged caches with token-major layout [num_blocks*bs, width].

    rows[T, width]: one row per token (any dtype; copied bit for bit).
    slot[dcp, T]: slot of token t on rank r or -1 (non-owner: not written).
    Bytes never written keep ``sentinel``.
    """
    T, width = rows.shape
    caches = np.full((dcp, num_blocks * bs, width), sentinel, dtype=rows.dtype)
    for r in range(dcp):
        for t in range(T):
            s = int(slot[r, t])
            if s >= 0:
                caches[r, s] = rows[t]
    return caches


# ---------------------------------------------------------------------------
# attention (fp64) and the exact LSE merge
# ---------------------------------------------------------------------------

def attention(q, K, V, scale):
    """Softmax attention of one query over a set of keys, fp64.

    q[dk], K[n, dk], V[n, dv] -> (o[dv], lse) with s_j = scale * q.k_j,
    lse = ln sum_j exp(s_j), o = sum_j exp(s_j - lse) v_j.  n == 0 gives
    (0, -inf).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64), NEG_INF
    s = scale * (K @ q)
    m = s.max()
    lse = m + math.log(np.exp(s - m).sum())
    o = np.exp(s - lse) @ V
    return o, lse


def attention_heads(Q, K, V, scale):
    """Softmax attention of several queries over one key set, fp64.

    The definition of ``attention`` applied to every row of Q[h, dk] (the
    query heads that share one KV head, or every head of an MLA latent):
    S[j, h] = scale * q_h.k_j, lse_h = ln sum_j exp(S[j, h]),
    o_h = sum_j exp(S[j, h] - lse_h) v_j.  Returns (O[h, dv], lse[h]); an
    empty key set gives zeros and -inf for every head.
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    nh = Q.shape[0]
    if K.shape[0] == 0:
        return np.zeros((nh, V.shape[1]), dtype=np.float64), np.full(nh, NEG_INF)
    S = scale * (K @ Q.T)
    m = S.max(axis=0)
    lse = m + np.log(np.exp(S - m).sum(axis=0))
    O = np.exp(S - lse).T @ V
    return O, lse


def shard_tokens(L, r, dcp, bs, I):
    """Global token ids owned by rank r among [0, L), in local-position order."""
    n = local_seq_len_closed_form(L, r, dcp, bs, I)
    return global_token(np.arange(n, dtype=np.int64), r, bs, dcp, I)


def lse_merge(parts_o, parts_lse, sink=None):
    """Exact merge of partial attention results by log-sum-exp.

    parts_o[n, dv], parts_lse[n]; sink: optional logit added once to the
    denominator with a zero value vector ("Decode computation" on the
    TokenSpeed page).  Returns (o[dv], lse); all parts empty and no sink
    gives (0, -inf).
    """
    parts_o = np.asarray(parts_o, dtype=np.float64)
    lses = [float(x) for x in parts_lse]
    if sink is not None:
        lses_all = lses + [float(sink)]
    else:
        lses_all = lses
    finite = [x for x in lses_all if x != NEG_INF]
    if not finite:
        return np.zeros(parts_o.shape[1], dtype=np.float64), NEG_INF
    m = max(finite)
    lse = m + math.log(sum(math.exp(x - m) for x in finite))
    o = np.zeros(parts_o.shape[1], dtype=np.float64)
    for i, x in enumerate(lses):
        if x != NEG_INF:
            o += math.exp(x - lse) * parts_o[i]
    return o, lse


def sharded_attention(q, K_all, V_all, scale, L, dcp, bs, I, sink=None):
    """DCP decode for one (request, head): per-rank partials, then the merge.

    K_all/V_all hold the request's keys/values in global token order.
    Returns (o, lse, per_rank_o[dcp, dv], per_rank_lse[dcp]).
    """
    dv = V_all.shape[1]
    po = np.zeros((dcp, dv))
    pl = np.full(dcp, NEG_INF)
    for r in range(dcp):
        idx = shard_tokens(L, r, dcp, bs, I)
        po[r], pl[r] = attention(q, K_all[idx], V_all[idx], scale)
    o, lse = lse_merge(po, pl, sink)
    return o, lse, po, pl


def sharded_attention_heads(Q, K_all, V_all, scale, L, dcp, bs, I, sinks=None):
    """``sharded_attention`` for several query heads over the same keys.

    Q[h, dk]; K_all/V_all hold the request's keys/values in global token
    order; sinks: None or one logit per row of Q.  Each rank attends its own
    shard ("Decode": attention over the local KV), then each head's partials
    are merged by log-sum-exp with its sink applied once.  Returns
    (o[h, dv], lse[h], per_rank_o[dcp, h, dv], per_rank_lse[dcp, h]).
    """
    Q = np.asarray(Q, dtype=np.float64)
    nh, dv = Q.shape[0], V_all.shape[1]
    po = np.zeros((dcp, nh, dv))
    pl = np.full((dcp, nh), NEG_INF)
    for r in range(dcp):
        idx = shard_tokens(L, r, dcp, bs, I)
        po[r], pl[r] = attention_heads(Q, K_all[idx], V_all[idx], scale)
    o = np.zeros((nh, dv))
    lse = np.full(nh, NEG_INF)
    for h in range(nh):
        s = None if sinks is None else float(sinks[h])
        o[h], lse[h] = lse_merge(po[:, h], pl[:, h], s)
    return o, lse, po, pl


def sparse_attention(q, K_all, V_all, scale, sel):
    """Attention restricted to the selected global token ids (SFA, unsharded)."""
    sel = np.asarray([g for g in sel if g >= 0 and g < K_all.shape[0]], dtype=np.int64)
    return attention(q, K_all[sel], V_all[sel], scale)


def sfa_sharded(q, K_all, V_all, scale, sel, L, dcp, bs, I, sink=None):
    """SFA under DCP: each rank attends its owned selected tokens; merge with sink once."""
    dv = V_all.shape[1]
    po = np.zeros((dcp, dv))
    pl = np.full(dcp, NEG_INF)
    sel = np.asarray([g for g in sel if 0 <= g < L], dtype=np.int64)
    owners = target_rank(sel, bs, dcp, I)
    for r in range(dcp):
        mine = sel[owners == r]
        po[r], pl[r] = attention(q, K_all[mine], V_all[mine], scale)
    o, lse = lse_merge(po, pl, sink)
    return o, lse, po, pl


def sfa_sharded_heads(Q, sel, K_sel, V_sel, scale, L, dcp, bs, I, sinks=None):
    """``sfa_sharded`` for several query heads, given only the selected rows.

    sel[k] are the global top-k token ids of the request and K_sel[k] /
    V_sel[k] the key / value rows of token sel[k] (so a long context need
    not be materialised).  Entries outside [0, L) are dropped; every other
    entry is attended as listed by the rank that owns it ("GLM-5.2 SFA DCP
    replicated indexer": each rank attends the selected tokens it holds);
    the partials are merged per head with its sink applied once.  Returns
    (o[h, dv], lse[h], per_rank_o[dcp, h, dv], per_rank_lse[dcp, h]).
    """
    Q = np.asarray(Q, dtype=np.float64)
    sel = np.asarray(sel, dtype=np.int64)
    keep = (sel >= 0) & (sel < L)
    sel = sel[keep]
    K_sel = np.asarray(K_sel)[keep]
    V_sel = np.asarray(V_sel)[keep]
    owners = target_rank(sel, bs, dcp, I)
    nh, dv = Q.shape[0], V_sel.shape[1]
    po = np.zeros((dcp, nh, dv))
    pl = np.full((dcp, nh), NEG_INF)
    for r in range(dcp):
        mine = owners == r
        po[r], pl[r] = attention_heads(Q, K_sel[mine], V_sel[mine], scale)
    o = np.zeros((nh, dv))
    lse = np.full(nh, NEG_INF)
    for h in range(nh):
        s = None if sinks is None else float(sinks[h])
        o[h], lse[h] = lse_merge(po[:, h], pl[:, h], s)
    return o, lse, po, pl


# ---------------------------------------------------------------------------
# exact distributed top-k ("DeepSeek V4.1 context parallelism", section
# "Decode computation": each rank computes local top-k candidates and the
# scores and logical ids are merged across ranks -- exact top-k selection
# under the kernel's score/tie rule)
# ---------------------------------------------------------------------------
# Rule (this library's, the page names none): a higher score ranks first; equal
# scores rank the smaller logical (global) token id first; NaN counts as -inf.

def _rank_order(scores, ids):
    """Indices of (score, id) in rule order: higher score first, ties by
    smaller id; NaN counts as -inf, and -0 and +0 are the same score."""
    s = np.where(np.isnan(scores), -np.inf, np.asarray(scores, dtype=np.float64))
    return np.lexsort((np.asarray(ids), -s))


def topk_exact(scores, ids, k):
    """Top-k of (score, id) pairs by the rule; returns (ids, scores) sorted."""
    order = _rank_order(scores, ids)[:k]
    return np.asarray(ids)[order], np.asarray(scores)[order]


def topk_local(local_scores, local_len, r, k, dcp, bs, I):
    """Rank r's candidates: the top-k of the scores of its local positions
    (local position p holds global token global_token(p, r))."""
    p = np.arange(int(local_len), dtype=np.int64)
    ids = global_token(p, r, bs, dcp, I)
    return topk_exact(np.asarray(local_scores)[:int(local_len)], ids, k)


def topk_distributed(local_scores, local_lens, k, dcp, bs, I):
    """Local top-k on every rank, then the top-k of all candidates."""
    cand_ids, cand_scores = [], []
    for r in range(dcp):
        i, s = topk_local(local_scores[r], local_lens[r], r, k, dcp, bs, I)
        cand_ids.append(i)
        cand_scores.append(s)
    return topk_exact(np.concatenate(cand_scores), np.concatenate(cand_ids), k)


# ---------------------------------------------------------------------------
# SFA prefill compaction ("Decode Context Parallel (DCP)", section "GLM-5.2
# SFA DCP replicated indexer": during prefill or a mixed batch, only the KV
# blocks referenced by the sparse block table are compacted, then gathered)
# ---------------------------------------------------------------------------

def sfa_compact_blocks(topk, q_req, seq_lens, block_table, caches, dcp, bs, I, num_blocks):
    """Reference compaction.

    topk[Q, K] global token ids of each query, q_req[Q] its request.
    Returns (blocks [n, bs, width] copied from the per-rank caches -- ranks
    in order, each rank's referenced physical blocks in increasing id
    order --, ids [n] physical id of each, counts [dcp], index [Q, K] row of
    each selected token in blocks viewed as [n*bs, width], -1 when invalid).
    caches[r] is rank r's token-major pool [num_blocks*bs, width].
    """
    Q, K = topk.shape
    refs = [set() for _ in range(dcp)]
    where = np.full((Q, K, 2), -1, dtype=np.int64)  # (rank, phys*bs + loc) per entry
    for qi in range(Q):
        b = int(q_req[qi])
        for k in range(K):
            g = int(topk[qi, k])
            if b < 0 or b >= len(seq_lens) or g < 0 or g >= int(seq_lens[b]):
                continue
            vb = virtual_block_index(g, bs, dcp)
            if vb >= block_table.shape[2]:
                continue
            r = target_rank(g, bs, dcp, I)
            phys = int(block_table[r, b, vb])
            if phys < 0 or phys >= num_blocks:
                continue
            refs[r].add(phys)
            where[qi, k] = (r, phys * bs + local_offset(g, bs, dcp, I))
    ids, counts, first = [], [], {}
    for r in range(dcp):
        srt = sorted(refs[r])
        counts.append(len(srt))
        for p in srt:
            first[(r, p)] = len(ids)
            ids.append(p)
    width = caches[0].shape[1]
    blocks = np.zeros((len(ids), bs, width), dtype=caches[0].dtype)
    for r in range(dcp):
        for p in sorted(refs[r]):
            blocks[first[(r, p)]] = caches[r][p * bs:(p + 1) * bs]
    index = np.full((Q, K), -1, dtype=np.int64)
    for qi in range(Q):
        for k in range(K):
            r, s = where[qi, k]
            if r >= 0:
                index[qi, k] = first[(int(r), int(s) // bs)] * bs + int(s) % bs
    return blocks, np.asarray(ids, dtype=np.int64), np.asarray(counts, dtype=np.int64), index


# ---------------------------------------------------------------------------
# chunked-prefill context gather ("Decode Context Parallel (DCP)", section
# "Prefill and chunked prefill": MLA gathers the context KV cache and
# restores request-contiguous order)
# ---------------------------------------------------------------------------

def gather_context(req, pos, caches, block_table, dcp, bs, I, num_blocks):
    """Rows of tokens (req[t], pos[t]) read back from the per-rank caches.

    caches[r]: token-major pool [num_blocks*bs, width] of rank r.  A token
    whose slot cannot be resolved gives a zero row (and is reported in the
    returned `bad` count).
    """
    rank, slot = slot_mapping(req, pos, block_table, None, dcp, bs, I, num_blocks)
    width = caches[0].shape[1]
    out = np.zeros((len(req), width), dtype=caches[0].dtype)
    bad = 0
    for t in range(len(req)):
        r = int(rank[t])
        if r < 0:
            bad += 1
            continue
        out[t] = caches[r][int(slot[r, t])]
    return out, bad

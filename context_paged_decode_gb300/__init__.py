"""Python binding of libdcp.so, the GB300 hot path of Decode Context Parallelism.

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  The functions carry
the C names without the ``dcp_`` prefix; see ``include/dcp.h`` for the
meaning, layout and error behaviour of every argument.

If the shared library is missing or fails to load, every call raises: there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdcp.so")
MAX_RANKS = 16

F32, BF16 = 0, 1
KIND_GQA, KIND_MLA, KIND_SFA = 0, 1, 2
_DT = {torch.float32: F32, torch.bfloat16: BF16}


class DcpError(RuntimeError):
    pass


class Layout(C.Structure):
    _fields_ = [("dcp_size", C.c_int32), ("block_size", C.c_int32), ("interleave", C.c_int32)]

    def __init__(self, dcp_size, block_size, interleave=1):
        super().__init__(int(dcp_size), int(block_size), int(interleave))

    def __repr__(self):
        return f"Layout(dcp={self.dcp_size}, bs={self.block_size}, I={self.interleave})"


class RankPtrs(C.Structure):
    _fields_ = [("ptr", C.c_void_p * MAX_RANKS)]


class PagedKVStruct(C.Structure):
    _fields_ = [("k", RankPtrs), ("v", RankPtrs), ("num_blocks", C.c_int64),
                ("block_table", C.c_void_p), ("max_vblocks", C.c_int32),
                ("bt_rank_stride", C.c_int64)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libdcp.so (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise DcpError(f"{path} not found: build it with __graft_entry__.build()")
    lib = C.CDLL(path)
    i32, i64, vp, f32 = C.c_int32, C.c_int64, C.c_void_p, C.c_float
    L, RP, PK = Layout, RankPtrs, PagedKVStruct
    sig = {
        "dcp_strerror": (C.c_char_p, [C.c_int]),
        "dcp_version": (C.c_int, []),
        "dcp_local_seq_lens": (C.c_int, [L, vp, i32, vp, vp, vp]),
        "dcp_slot_mapping": (C.c_int, [L, vp, vp, i64, vp, i32, i32, i64, i64, vp, vp, vp, vp]),
        "dcp_cache_write_gqa": (C.c_int, [L, vp, vp, i64, i32, i32, C.c_int, vp, i64, RP, RP, vp,
                                          vp]),
        "dcp_cache_write_mla": (C.c_int, [L, vp, i64, i32, C.c_int, vp, i64, RP, vp, vp]),
        "dcp_gather_context_mla": (C.c_int, [L, PK, i32, i32, C.c_int, vp, vp, i64, vp, vp, vp]),
        "dcp_decode_workspace_size": (C.c_int, [L, C.c_int, i32, i32, i32, i32,
                                                C.POINTER(C.c_size_t)]),
        "dcp_decode_partial_gqa": (C.c_int, [L, vp, i32, i32, i32, i32, f32, C.c_int, PK, vp, vp,
                                             vp, vp, C.c_size_t, vp, vp]),
        "dcp_lse_merge": (C.c_int, [i32, vp, vp, i32, i32, i32, vp, vp, C.c_int, vp, vp]),
        "dcp_lse_merge_swa": (C.c_int, [i32, vp, vp, vp, vp, i32, i32, i32, vp, vp, C.c_int, vp,
                                        vp]),
        "dcp_decode_gqa": (C.c_int, [L, vp, i32, i32, i32, i32, f32, C.c_int, PK, vp, vp, vp,
                                     C.c_int, vp, vp, C.c_size_t, vp, vp]),
        "dcp_decode_gqa_noalloc": (C.c_int, [L, vp, i32, i32, i32, i32, f32, C.c_int, PK, vp, vp,
                                             vp, C.c_int, vp, vp, vp]),
        "dcp_decode_partial_mla": (C.c_int, [L, vp, i32, i32, i32, i32, f32, C.c_int, PK, vp, vp,
                                             vp, vp, C.c_size_t, vp, vp]),
        "dcp_decode_mla": (C.c_int, [L, vp, i32, i32, i32, i32, f32, C.c_int, PK, vp, vp, vp,
                                     C.c_int, vp, vp, C.c_size_t, vp, vp]),
        "dcp_sfa_remap": (C.c_int, [L, vp, i32, i32, vp, vp, i32, i64, i64, vp, vp, vp, vp]),
        "dcp_topk_workspace_size": (C.c_int, [L, i32, i32, C.POINTER(C.c_size_t)]),
        "dcp_topk_local": (C.c_int, [L, vp, i32, i32, vp, i32, vp, vp]),
        "dcp_topk_merge": (C.c_int, [i32, vp, i32, i32, vp, C.c_size_t, vp, vp, vp]),
        "dcp_topk": (C.c_int, [L, vp, i32, i32, vp, i32, vp, vp, vp, C.c_size_t, vp]),
        "dcp_sfa_compact_workspace_size": (C.c_int, [L, i64, C.POINTER(C.c_size_t)]),
        "dcp_sfa_compact_blocks": (C.c_int, [L, vp, vp, i32, i32, vp, i32, PK, i32, C.c_int, i64,
                                             vp, vp, vp, vp, vp, C.c_size_t, vp, vp]),
        "dcp_sfa_decode_partial": (C.c_int, [L, vp, i32, i32, i32, i32, f32, C.c_int, PK, vp, vp,
                                             i32, vp, vp, vp, vp]),
        "dcp_sfa_decode": (C.c_int, [L, vp, i32, i32, i32, i32, f32, C.c_int, PK, vp, i32, vp, vp,
                                     vp, C.c_int, vp, vp, C.c_size_t, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def exported_symbols():
    """Names of the C entry points this binding expects the library to export."""
    return ["dcp_strerror", "dcp_version", "dcp_local_seq_lens", "dcp_slot_mapping",
            "dcp_cache_write_gqa", "dcp_cache_write_mla", "dcp_gather_context_mla",
            "dcp_decode_workspace_size",
            "dcp_decode_partial_gqa", "dcp_lse_merge", "dcp_lse_merge_swa", "dcp_decode_gqa",
            "dcp_decode_gqa_noalloc",
            "dcp_decode_partial_mla",
            "dcp_decode_mla", "dcp_sfa_remap", "dcp_topk_workspace_size", "dcp_topk_local", "dcp_topk_merge",
            "dcp_topk", "dcp_sfa_compact_workspace_size", "dcp_sfa_compact_blocks",
            "dcp_sfa_decode_partial", "dcp_sfa_decode"]


def _check(rc):
    if rc != 0:
        msg = load().dcp_strerror(rc).decode()
        raise DcpError(f"libdcp error {rc}: {msg}")


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _dtype(t):
    try:
        return _DT[t.dtype]
    except KeyError:
        raise DcpError(f"unsupported dtype {t.dtype}") from None


def _cuda_contig(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise DcpError("tensors must be contiguous CUDA tensors")


def rank_ptrs(tensors) -> RankPtrs:
    rp = RankPtrs()
    for i, t in enumerate(tensors or []):
        rp.ptr[i] = t.data_ptr()
    return rp


class PagedKV:
    """Per-rank paged pools plus the block table, as the decode calls read them.

    k_pools / v_pools: one tensor per rank (GQA: [num_blocks, Hkv, bs, d];
    latent: [num_blocks, bs, kv_dim], v_pools None).  block_table:
    [dcp, B, max_vb] int32 (one table per rank) or [B, max_vb] (shared).
    """

    def __init__(self, k_pools, v_pools, block_table, num_blocks):
        self.k_pools = list(k_pools)
        self.v_pools = list(v_pools) if v_pools is not None else None
        self.block_table = block_table
        self.num_blocks = int(num_blocks)
        _cuda_contig(block_table, *self.k_pools, *(self.v_pools or []))
        if block_table.dtype != torch.int32:
            raise DcpError("block_table must be int32")
        if block_table.dim() == 3:
            self.max_vb = block_table.shape[2]
            self.bt_rank_stride = block_table.shape[1] * block_table.shape[2]
        else:
            self.max_vb = block_table.shape[1]
            self.bt_rank_stride = 0

    def struct(self) -> PagedKVStruct:
        s = PagedKVStruct()
        s.k = rank_ptrs(self.k_pools)
        s.v = rank_ptrs(self.v_pools)
        s.num_blocks = self.num_blocks
        s.block_table = self.block_table.data_ptr()
        s.max_vblocks = self.max_vb
        s.bt_rank_stride = self.bt_rank_stride
        return s


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def local_seq_lens(layout, seq_lens, out=None, err=None, stream=None):
    lib = load()
    _cuda_contig(seq_lens)
    B = seq_lens.shape[0]
    if out is None:
        out = torch.empty((B, layout.dcp_size), dtype=torch.int32, device=seq_lens.device)
    _check(lib.dcp_local_seq_lens(layout, _p(seq_lens), B, _p(out), _p(err), _stream(stream)))
    return out


def slot_mapping(layout, req_idx, positions, block_table, num_blocks, out_rank=None,
                 out_slot=None, err=None, stream=None):
    lib = load()
    _cuda_contig(req_idx, positions, block_table)
    T = req_idx.shape[0]
    if block_table.dim() == 3:
        B, max_vb, stride = block_table.shape[1], block_table.shape[2], \
            block_table.shape[1] * block_table.shape[2]
    else:
        B, max_vb, stride = block_table.shape[0], block_table.shape[1], 0
    dev = req_idx.device
    if out_rank is None:
        out_rank = torch.empty(T, dtype=torch.int32, device=dev)
    if out_slot is None:
        out_slot = torch.empty((layout.dcp_size, T), dtype=torch.int64, device=dev)
    _check(lib.dcp_slot_mapping(layout, _p(req_idx), _p(positions), T, _p(block_table), B, max_vb,
                                stride, int(num_blocks), _p(out_rank), _p(out_slot), _p(err),
                                _stream(stream)))
    return out_rank, out_slot


def cache_write_gqa(layout, k, v, slot, k_pools, v_pools, num_blocks, err=None, stream=None):
    lib = load()
    _cuda_contig(k, v, slot)
    T, Hkv, d = k.shape
    _check(lib.dcp_cache_write_gqa(layout, _p(k), _p(v), T, Hkv, d, _dtype(k), _p(slot),
                                   int(num_blocks), rank_ptrs(k_pools), rank_ptrs(v_pools),
                                   _p(err), _stream(stream)))


def cache_write_mla(layout, kv, slot, pools, num_blocks, err=None, stream=None):
    lib = load()
    _cuda_contig(kv, slot)
    T, dk = kv.shape
    _check(lib.dcp_cache_write_mla(layout, _p(kv), T, dk, _dtype(kv), _p(slot), int(num_blocks),
                                   rank_ptrs(pools), _p(err), _stream(stream)))


def gather_context_mla(layout, kv: PagedKV, req_idx, positions, out=None, err=None,
                       stream=None):
    """Rows of tokens (req_idx[t], positions[t]) from the sharded latent cache."""
    lib = load()
    _cuda_contig(req_idx, positions)
    T = req_idx.shape[0]
    pool = kv.k_pools[0]
    kv_dim = pool.shape[-1]
    B = kv.block_table.shape[-2]
    if out is None:
        out = torch.empty((T, kv_dim), dtype=pool.dtype, device=pool.device)
    _check(lib.dcp_gather_context_mla(layout, kv.struct(), B, kv_dim, _dtype(pool), _p(req_idx),
                                      _p(positions), T, _p(out), _p(err), _stream(stream)))
    return out


def decode_workspace_size(layout, kind, num_reqs, num_q_heads, num_kv_heads, head_dim_v):
    lib = load()
    n = C.c_size_t(0)
    _check(lib.dcp_decode_workspace_size(layout, kind, num_reqs, num_q_heads, num_kv_heads,
                                         head_dim_v, C.byref(n)))
    return n.value


def _workspace(layout, kind, B, Hq, Hkv, dv, device, workspace):
    need = decode_workspace_size(layout, kind, B, Hq, Hkv, dv)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    return workspace


def decode_partial_gqa(layout, q, kv: PagedKV, local_lens, scale, part_o=None, part_lse=None,
                       workspace=None, err=None, stream=None):
    lib = load()
    _cuda_contig(q, local_lens)
    B, Hq, d = q.shape
    Hkv = kv.k_pools[0].shape[1]
    dev = q.device
    if part_o is None:
        part_o = torch.empty((layout.dcp_size, B, Hq, d), dtype=torch.float32, device=dev)
    if part_lse is None:
        part_lse = torch.empty((layout.dcp_size, B, Hq), dtype=torch.float32, device=dev)
    ws = _workspace(layout, KIND_GQA, B, Hq, Hkv, d, dev, workspace)
    _check(lib.dcp_decode_partial_gqa(layout, _p(q), B, Hq, Hkv, d, float(scale), _dtype(q),
                                      kv.struct(), _p(local_lens), _p(part_o), _p(part_lse),
                                      _p(ws), ws.numel(), _p(err), _stream(stream)))
    return part_o, part_lse


def decode_gqa(layout, q, kv: PagedKV, local_lens, scale, sink=None, out_dtype=None, out=None,
               out_lse=None, workspace=None, err=None, stream=None):
    lib = load()
    _cuda_contig(q, local_lens, sink)
    B, Hq, d = q.shape
    Hkv = kv.k_pools[0].shape[1]
    dev = q.device
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, d), dtype=odt, device=dev)
    if out_lse is None:
        out_lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = _workspace(layout, KIND_GQA, B, Hq, Hkv, d, dev, workspace)
    _check(lib.dcp_decode_gqa(layout, _p(q), B, Hq, Hkv, d, float(scale), _dtype(q), kv.struct(),
                              _p(local_lens), _p(sink), _p(out), _dtype(out), _p(out_lse),
                              _p(ws), ws.numel(), _p(err), _stream(stream)))
    return out, out_lse


def decode_gqa_noalloc(layout, q, kv: PagedKV, local_lens, scale, sink=None, out_dtype=None,
                       out=None, out_lse=None, err=None, stream=None):
    """dcp_decode_gqa without a caller workspace: the library's fixed 16 MiB
    device array holds the split-KV scratch (for callers that cannot allocate;
    calls that overlap on the GPU race on that array)."""
    lib = load()
    _cuda_contig(q, local_lens, sink)
    B, Hq, d = q.shape
    Hkv = kv.k_pools[0].shape[1]
    dev = q.device
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, d), dtype=odt, device=dev)
    if out_lse is None:
        out_lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    _check(lib.dcp_decode_gqa_noalloc(layout, _p(q), B, Hq, Hkv, d, float(scale), _dtype(q),
                                      kv.struct(), _p(local_lens), _p(sink), _p(out),
                                      _dtype(out), _p(out_lse), _p(err), _stream(stream)))
    return out, out_lse


def lse_merge(part_o, part_lse, sink=None, out_dtype=torch.float32, out=None, out_lse=None,
              stream=None):
    lib = load()
    _cuda_contig(part_o, part_lse, sink)
    n, B, H, dv = part_o.shape
    dev = part_o.device
    if out is None:
        out = torch.empty((B, H, dv), dtype=out_dtype, device=dev)
    if out_lse is None:
        out_lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    _check(lib.dcp_lse_merge(n, _p(part_o), _p(part_lse), B, H, dv, _p(sink), _p(out),
                             _dtype(out), _p(out_lse), _stream(stream)))
    return out, out_lse


def lse_merge_swa(part_o, part_lse, swa_o, swa_lse, sink=None, out_dtype=torch.float32, out=None,
                  out_lse=None, stream=None):
    """Merge the per-rank partials with ONE replicated-window partial (+ sink)."""
    lib = load()
    _cuda_contig(part_o, part_lse, swa_o, swa_lse, sink)
    n, B, H, dv = part_o.shape
    dev = part_o.device
    if out is None:
        out = torch.empty((B, H, dv), dtype=out_dtype, device=dev)
    if out_lse is None:
        out_lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    _check(lib.dcp_lse_merge_swa(n, _p(part_o), _p(part_lse), _p(swa_o), _p(swa_lse), B, H, dv,
                                 _p(sink), _p(out), _dtype(out), _p(out_lse), _stream(stream)))
    return out, out_lse


def decode_partial_mla(layout, q, kv: PagedKV, local_lens, scale, v_dim=512, part_o=None,
                       part_lse=None, workspace=None, err=None, stream=None):
    lib = load()
    _cuda_contig(q, local_lens)
    B, Hq, dk = q.shape
    dev = q.device
    if part_o is None:
        part_o = torch.empty((layout.dcp_size, B, Hq, v_dim), dtype=torch.float32, device=dev)
    if part_lse is None:
        part_lse = torch.empty((layout.dcp_size, B, Hq), dtype=torch.float32, device=dev)
    ws = _workspace(layout, KIND_MLA, B, Hq, 1, v_dim, dev, workspace)
    _check(lib.dcp_decode_partial_mla(layout, _p(q), B, Hq, dk, v_dim, float(scale), _dtype(q),
                                      kv.struct(), _p(local_lens), _p(part_o), _p(part_lse),
                                      _p(ws), ws.numel(), _p(err), _stream(stream)))
    return part_o, part_lse


def decode_mla(layout, q, kv: PagedKV, local_lens, scale, v_dim=512, sink=None, out_dtype=None,
               out=None, out_lse=None, workspace=None, err=None, stream=None):
    lib = load()
    _cuda_contig(q, local_lens, sink)
    B, Hq, dk = q.shape
    dev = q.device
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, v_dim), dtype=odt, device=dev)
    if out_lse is None:
        out_lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = _workspace(layout, KIND_MLA, B, Hq, 1, v_dim, dev, workspace)
    _check(lib.dcp_decode_mla(layout, _p(q), B, Hq, dk, v_dim, float(scale), _dtype(q),
                              kv.struct(), _p(local_lens), _p(sink), _p(out), _dtype(out),
                              _p(out_lse), _p(ws), ws.numel(), _p(err), _stream(stream)))
    return out, out_lse


def sfa_remap(layout, topk, seq_lens, block_table, num_blocks, out_rank=None, out_slot=None,
              err=None, stream=None):
    lib = load()
    _cuda_contig(topk, seq_lens, block_table)
    B, K = topk.shape
    if block_table.dim() == 3:
        max_vb, stride = block_table.shape[2], block_table.shape[1] * block_table.shape[2]
    else:
        max_vb, stride = block_table.shape[1], 0
    if out_rank is None:
        out_rank = torch.empty((B, K), dtype=torch.int32, device=topk.device)
    if out_slot is None:
        out_slot = torch.empty((B, K), dtype=torch.int32, device=topk.device)
    _check(lib.dcp_sfa_remap(layout, _p(topk), B, K, _p(seq_lens), _p(block_table), max_vb,
                             stride, int(num_blocks), _p(out_rank), _p(out_slot), _p(err),
                             _stream(stream)))
    return out_rank, out_slot


def topk_local(layout, local_scores, local_lens, k, cand=None, stream=None):
    """Per-rank top-k candidate keys [dcp, B, k] (uint64 stored as int64)."""
    lib = load()
    _cuda_contig(local_scores, local_lens)
    dcp_, B, max_local = local_scores.shape
    if cand is None:
        cand = torch.empty((dcp_, B, k), dtype=torch.int64, device=local_scores.device)
    _check(lib.dcp_topk_local(layout, _p(local_scores), B, max_local, _p(local_lens), k, _p(cand),
                              _stream(stream)))
    return cand


def topk_merge(cand, stream=None):
    lib = load()
    _cuda_contig(cand)
    dcp_, B, k = cand.shape
    dev = cand.device
    ws = torch.empty(B * k * 8, dtype=torch.uint8, device=dev)
    ids = torch.empty((B, k), dtype=torch.int32, device=dev)
    scores = torch.empty((B, k), dtype=torch.float32, device=dev)
    _check(lib.dcp_topk_merge(dcp_, _p(cand), B, k, _p(ws), ws.numel(), _p(ids), _p(scores),
                              _stream(stream)))
    return ids, scores


def topk(layout, local_scores, local_lens, k, stream=None):
    """Exact global top-k ids and scores [B, k] from per-rank local scores."""
    lib = load()
    _cuda_contig(local_scores, local_lens)
    dcp_, B, max_local = local_scores.shape
    dev = local_scores.device
    n = C.c_size_t(0)
    _check(lib.dcp_topk_workspace_size(layout, B, k, C.byref(n)))
    ws = torch.empty(max(n.value, 1), dtype=torch.uint8, device=dev)
    ids = torch.empty((B, k), dtype=torch.int32, device=dev)
    scores = torch.empty((B, k), dtype=torch.float32, device=dev)
    _check(lib.dcp_topk(layout, _p(local_scores), B, max_local, _p(local_lens), k, _p(ids),
                        _p(scores), _p(ws), ws.numel(), _stream(stream)))
    return ids, scores


def sfa_compact_blocks(layout, kv: PagedKV, topk, q_req, seq_lens, max_blocks, err=None,
                       stream=None):
    """Compact the referenced latent blocks; returns (blocks, ids, counts, index)."""
    lib = load()
    _cuda_contig(topk, q_req, seq_lens)
    Q, K = topk.shape
    pool = kv.k_pools[0]
    kv_dim, bs = pool.shape[-1], pool.shape[-2]
    dev = pool.device
    n = C.c_size_t(0)
    _check(lib.dcp_sfa_compact_workspace_size(layout, kv.num_blocks, C.byref(n)))
    ws = torch.empty(max(n.value, 1), dtype=torch.uint8, device=dev)
    blocks = torch.empty((max(max_blocks, 1), bs, kv_dim), dtype=pool.dtype, device=dev)
    ids = torch.empty(max(max_blocks, 1), dtype=torch.int32, device=dev)
    counts = torch.empty(layout.dcp_size, dtype=torch.int32, device=dev)
    index = torch.empty((Q, K), dtype=torch.int64, device=dev)
    _check(lib.dcp_sfa_compact_blocks(layout, _p(topk), _p(q_req), Q, K, _p(seq_lens),
                                      kv.block_table.shape[-2], kv.struct(), kv_dim, _dtype(pool),
                                      int(max_blocks), _p(blocks), _p(ids), _p(counts),
                                      _p(index), _p(ws), ws.numel(), _p(err), _stream(stream)))
    return blocks, ids, counts, index


def sfa_decode_partial(layout, q, kv: PagedKV, sel_rank, sel_slot, scale, v_dim=512,
                       part_o=None, part_lse=None, err=None, stream=None):
    lib = load()
    _cuda_contig(q, sel_rank, sel_slot)
    B, Hq, dk = q.shape
    K = sel_rank.shape[1]
    dev = q.device
    if part_o is None:
        part_o = torch.empty((layout.dcp_size, B, Hq, v_dim), dtype=torch.float32, device=dev)
    if part_lse is None:
        part_lse = torch.empty((layout.dcp_size, B, Hq), dtype=torch.float32, device=dev)
    _check(lib.dcp_sfa_decode_partial(layout, _p(q), B, Hq, dk, v_dim, float(scale), _dtype(q),
                                      kv.struct(), _p(sel_rank), _p(sel_slot), K, _p(part_o),
                                      _p(part_lse), _p(err), _stream(stream)))
    return part_o, part_lse


def sfa_decode(layout, q, kv: PagedKV, topk, seq_lens, scale, v_dim=512, sink=None,
               out_dtype=None, out=None, out_lse=None, workspace=None, err=None, stream=None):
    lib = load()
    _cuda_contig(q, topk, seq_lens, sink)
    B, Hq, dk = q.shape
    K = topk.shape[1]
    dev = q.device
    odt = out_dtype or q.dtype
    if out is None:
        out = torch.empty((B, Hq, v_dim), dtype=odt, device=dev)
    if out_lse is None:
        out_lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = _workspace(layout, KIND_SFA, B, Hq, 1, v_dim, dev, workspace)
    _check(lib.dcp_sfa_decode(layout, _p(q), B, Hq, dk, v_dim, float(scale), _dtype(q),
                              kv.struct(), _p(topk), K, _p(seq_lens), _p(sink), _p(out),
                              _dtype(out), _p(out_lse), _p(ws), ws.numel(), _p(err),
                              _stream(stream)))
    return out, out_lse

"""Stage a synthetic DCP decode workload on the GPU (tests and bench only).

Values come from the GPU copy of the seeded generator (``synth.cu``), which
produces the same bits as the numpy generator in ``workloads/__init__.py``.
The per-rank paged caches are then filled through the library's own public
calls (``slot_mapping`` + ``cache_write_*``), exactly as a serving engine
would write them one chunk of tokens at a time.  Nothing here computes any
part of the method itself.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass, field

import numpy as np
import torch

import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
_synth = None


def synth_lib():
    global _synth
    if _synth is None:
        path = os.path.join(HERE, "libdcp_synth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} not built")
        lib = C.CDLL(path)
        lib.synth_fill.restype = C.c_int
        lib.synth_fill.argtypes = [C.c_uint64, C.c_int64, C.c_int64, C.c_void_p, C.c_int,
                                   C.c_void_p, C.c_void_p]
        _synth = lib
    return _synth


_tables = {}


def device_table(dtype: str, device):
    key = (dtype, str(device))
    if key not in _tables:
        t = W.value_table(dtype)
        if dtype == "bf16":
            _tables[key] = torch.from_numpy(t.view(np.int16).copy()).to(device)
        else:
            _tables[key] = torch.from_numpy(t.copy()).to(device)
    return _tables[key]


def torch_dtype(dtype: str):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def fill(out: torch.Tensor, seed: int, tensor: int, request: int, e0: int, dtype: str):
    """Fill a contiguous device tensor with stream elements [e0, e0 + numel)."""
    tab = device_table(dtype, out.device)
    key = W.stream_key(seed, tensor, request)
    rc = synth_lib().synth_fill(key, e0, out.numel(), tab.data_ptr(), tab.element_size(),
                                out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill failed ({rc})")


@dataclass
class DeviceWorkload:
    cfg: W.Config
    layout: object
    seq_lens_host: np.ndarray
    seq_lens: torch.Tensor
    local_lens: torch.Tensor
    bt_host: np.ndarray
    block_table: torch.Tensor
    num_blocks: int
    q: torch.Tensor
    kv: object                       # context_paged_decode_gb300.PagedKV
    k_pools: list
    v_pools: list
    sink: torch.Tensor | None = None
    topk_host: np.ndarray | None = None
    topk: torch.Tensor | None = None
    extra: dict = field(default_factory=dict)

    def kv_bytes(self) -> int:
        """Bytes of K/V (or latent rows) the decode step must read once."""
        tokens = int(self.seq_lens_host.astype(np.int64).sum())
        c = self.cfg
        if c.kind == "gqa":
            return tokens * c.Hkv * c.dk * 2 * (2 if c.dtype == "bf16" else 4)
        return tokens * c.dk * (2 if c.dtype == "bf16" else 4)


def build(cfg: W.Config, device="cuda", seq_lens=None, perm=None, populate=True,
          chunk_tokens=1 << 18, sentinel=True):
    """Allocate and populate the per-rank caches of one workload on the GPU."""
    import context_paged_decode_gb300 as dcp

    lens = np.asarray(seq_lens if seq_lens is not None else W.make_seq_lens(cfg), dtype=np.int32)
    layout = dcp.Layout(cfg.dcp, cfg.bs, cfg.I)
    bt_host, nb = W.make_block_tables(lens, cfg.dcp, cfg.bs, perm or cfg.perm, seed=cfg.seed)
    tdt = torch_dtype(cfg.dtype)
    B = len(lens)
    seq_lens_d = torch.from_numpy(lens).to(device)
    bt = torch.from_numpy(bt_host).to(device)
    q = torch.empty((B, cfg.Hq, cfg.dk), dtype=tdt, device=device)
    for b in range(B):
        fill(q[b], cfg.seed, W.T_Q, b, 0, cfg.dtype)
    if cfg.kind == "gqa":
        shape = (nb, cfg.Hkv, cfg.bs, cfg.dk)
        k_pools = [torch.empty(shape, dtype=tdt, device=device) for _ in range(cfg.dcp)]
        v_pools = [torch.empty(shape, dtype=tdt, device=device) for _ in range(cfg.dcp)]
    else:
        shape = (nb, cfg.bs, cfg.dk)
        k_pools = [torch.empty(shape, dtype=tdt, device=device) for _ in range(cfg.dcp)]
        v_pools = None
    if sentinel:  # all-ones bytes: NaN in bf16 and f32, so unwritten slots are visible
        for t in k_pools + (v_pools or []):
            t.view(torch.uint8).fill_(0xFF)
    local = dcp.local_seq_lens(layout, seq_lens_d)
    kv = dcp.PagedKV(k_pools, v_pools, bt, nb)
    wl = DeviceWorkload(cfg, layout, lens, seq_lens_d, local, bt_host, bt, nb, q, kv, k_pools,
                        v_pools or [])
    if cfg.sink:
        wl.sink = torch.from_numpy(W.sink_logits(cfg)).to(device)
    if cfg.topk:
        wl.topk_host = W.make_topk(cfg, lens)
        wl.topk = torch.from_numpy(wl.topk_host).to(device)
    if populate:
        populate_caches(wl, chunk_tokens)
    return wl


def populate_caches(wl: DeviceWorkload, chunk_tokens=1 << 18, tokens=None):
    """Write every token (or tokens[b] = (x0, x1) ranges) through slot_mapping + cache_write."""
    import context_paged_decode_gb300 as dcp

    cfg = wl.cfg
    dev = wl.q.device
    tdt = torch_dtype(cfg.dtype)
    row = cfg.Hkv * cfg.dk if cfg.kind == "gqa" else cfg.dk
    for b, L in enumerate(wl.seq_lens_host):
        x0_all, x1_all = (0, int(L)) if tokens is None else tokens[b]
        for x0 in range(x0_all, x1_all, chunk_tokens):
            x1 = min(x1_all, x0 + chunk_tokens)
            n = x1 - x0
            req = torch.full((n,), b, dtype=torch.int32, device=dev)
            pos = torch.arange(x0, x1, dtype=torch.int64, device=dev)
            _, slot = dcp.slot_mapping(wl.layout, req, pos, wl.block_table, wl.num_blocks)
            if cfg.kind == "gqa":
                k = torch.empty((n, cfg.Hkv, cfg.dk), dtype=tdt, device=dev)
                v = torch.empty_like(k)
                fill(k, cfg.seed, W.T_K, b, x0 * row, cfg.dtype)
                fill(v, cfg.seed, W.T_V, b, x0 * row, cfg.dtype)
                dcp.cache_write_gqa(wl.layout, k, v, slot, wl.k_pools, wl.v_pools, wl.num_blocks)
            else:
                kvr = torch.empty((n, cfg.dk), dtype=tdt, device=dev)
                fill(kvr, cfg.seed, W.T_LATENT, b, x0 * row, cfg.dtype)
                dcp.cache_write_mla(wl.layout, kvr, slot, wl.k_pools, wl.num_blocks)

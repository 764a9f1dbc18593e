"""Seeded synthetic inputs for the DCP decode workloads.

This module is shared by the CPU oracle (tests) and by the GPU path (tests,
bench).  It holds only input generation: context lengths, block tables,
top-k index sets and the q/k/v/latent/sink values.  None of the method's
arithmetic (layout, slot mapping, attention, merge) lives here.

Value generator (both the numpy version below and the CUDA version in
``synth.cu`` implement exactly this definition, bit for bit):

* a 64-bit stream key per (seed, tensor id, request)::

      key = mix64(seed*G1 + tensor*G2 + request*G3 + G4)   (mod 2**64)

* element ``e`` of that stream (row-major index inside the request's tensor)::

      u = mix64(key + (e + 1) * GAMMA)                     (mod 2**64)
      value = TABLE[u >> 48]

  ``mix64`` is the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014; the
  constants are Stafford's "Mix13").  ``TABLE[i]`` is the standard-normal
  quantile at ``(i + 0.5) / 65536`` (inverse-transform sampling with a 16-bit
  uniform), rounded to fp32, and to bf16 by round-to-nearest-even for bf16
  tensors.  So every value is an N(0, 1) draw quantised to 65536 levels,
  which is finer than bf16 except beyond |x| > 4.2 where the table ends.

Because any element can be regenerated from its index alone, the oracle can
rebuild one (request, head) slice of a multi-gigabyte cache without
generating the rest.
"""
from __future__ import annotations

import math
import os
import statistics
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB
_G1 = 0xD1B54A32D192ED03
_G2 = 0x8CB92BA72F3D8DD7
_G3 = 0xABC98388FB8FAC03
_G4 = 0x2545F4914F6CDD1D

# tensor ids of the value streams
T_Q, T_K, T_V, T_LATENT, T_SINK = 1, 2, 3, 4, 5


def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2**64)."""
    z &= M64
    z = ((z ^ (z >> 30)) * _C1) & M64
    z = ((z ^ (z >> 27)) * _C2) & M64
    return z ^ (z >> 31)


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_C1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_C2)
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor: int, request: int) -> int:
    return mix64_int(int(seed) * _G1 + int(tensor) * _G2 + int(request) * _G3 + _G4)


_TABLES: dict = {}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def value_table(dtype: str) -> np.ndarray:
    """65536-entry quantile table: fp32 values, or bf16 bit patterns (uint16)."""
    if dtype not in _TABLES:
        if "f32" not in _TABLES:
            nd = statistics.NormalDist()
            _TABLES["f32"] = np.array(
                [nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)], dtype=np.float32)
        if dtype == "bf16":
            _TABLES["bf16"] = f32_to_bf16_bits(_TABLES["f32"])
        elif dtype != "f32":
            raise ValueError(dtype)
    return _TABLES[dtype]


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1))
    return _POOL


def _fill_chunk(key: int, e0: int, n: int, table: np.ndarray, out: np.ndarray):
    e = np.arange(e0 + 1, e0 + 1 + n, dtype=np.uint64)
    u = _mix64_np(e * np.uint64(GAMMA) + np.uint64(key))
    out[:] = table[(u >> np.uint64(48)).astype(np.intp)]


def stream_values(seed: int, tensor: int, request: int, e0: int, n: int, dtype: str) -> np.ndarray:
    """Elements [e0, e0+n) of one value stream.

    Returns fp32 values for dtype 'f32' and bf16 bit patterns (uint16) for 'bf16'.
    """
    table = value_table(dtype)
    key = stream_key(seed, tensor, request)
    out = np.empty(n, dtype=table.dtype)
    chunk = 1 << 22
    if n <= chunk:
        _fill_chunk(key, e0, n, table, out)
        return out
    futs = [_pool().submit(_fill_chunk, key, e0 + s, min(chunk, n - s), table, out[s:s + chunk])
            for s in range(0, n, chunk)]
    for f in futs:
        f.result()
    return out


def as_float64(vals: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of generated elements (fp32 values or bf16 bits)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(vals).astype(np.float64)
    return np.asarray(vals, dtype=np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# workload configurations
# ---------------------------------------------------------------------------

@dataclass
class Config:
    name: str
    kind: str            # "gqa", "mla" or "sfa"
    B: int
    Hq: int
    Hkv: int             # 1 for the latent (MLA / SFA) caches
    dk: int              # key width (GQA head_dim; 576 for the latent)
    dv: int              # value width (GQA head_dim; 512 for the latent)
    dtype: str           # "f32" or "bf16"
    dcp: int
    bs: int
    I: int
    scale: float
    seed: int
    lengths: object      # list of ints, or a recipe name
    perm: str = "random"     # physical block permutation per rank: "random" or "identity"
    topk: int = 0
    sink: bool = False
    description: str = ""
    extra: dict = field(default_factory=dict)


CONFIGS = {
    "tiny_gqa_f32": Config(
        "tiny_gqa_f32", "gqa", B=2, Hq=8, Hkv=2, dk=64, dv=64, dtype="f32", dcp=2, bs=16, I=1,
        scale=1.0 / 8.0, seed=1, lengths=[100, 37],
        description="tiny GQA DCP decode, fp32: B=2, L={100,37}, Hq=8, Hkv=2, d=64, dcp=2, bs=16, I=1"),
    "gqa_bf16_b32": Config(
        "gqa_bf16_b32", "gqa", B=32, Hq=32, Hkv=8, dk=128, dv=128, dtype="bf16", dcp=8, bs=16, I=1,
        scale=1.0 / math.sqrt(128.0), seed=2, lengths="bimodal",
        description="GQA DCP decode, bf16: B=32, Hq=32, Hkv=8, d=128, bimodal 1k-256k contexts, "
                    "dcp=8, bs=16, I=1, random physical blocks per rank"),
    "mla_bf16_b64": Config(
        "mla_bf16_b64", "mla", B=64, Hq=128, Hkv=1, dk=576, dv=512, dtype="bf16", dcp=8, bs=64, I=1,
        scale=1.0 / math.sqrt(192.0), seed=3, lengths="bimodal",
        description="MLA DCP decode, bf16: B=64, Hq=128, latent 512+64, bimodal contexts, "
                    "dcp=8, bs=64, I=1"),
    "sfa_bf16_b32": Config(
        "sfa_bf16_b32", "sfa", B=32, Hq=64, Hkv=1, dk=576, dv=512, dtype="bf16", dcp=8, bs=64, I=64,
        scale=1.0 / math.sqrt(192.0), seed=4, lengths="uniform_32k_128k", topk=2048, sink=True,
        description="SFA sparse DCP decode, bf16 MLA-shaped KV, Hq=64: B=32, L~U[32k,128k], "
                    "dcp=8, bs=64, I=64, top-k 2048, per-head sink"),
    "longtail_gqa": Config(
        "longtail_gqa", "gqa", B=4, Hq=32, Hkv=8, dk=128, dv=128, dtype="bf16", dcp=8, bs=64, I=1,
        scale=1.0 / math.sqrt(128.0), seed=5, lengths=[1048576, 524288, 262144, 4096],
        description="long-tail GQA stress: B=4, L={1M,512k,256k,4k}, dcp=8, bs=64, I=1"),
    "longtail_mla": Config(
        "longtail_mla", "mla", B=4, Hq=128, Hkv=1, dk=576, dv=512, dtype="bf16", dcp=8, bs=64, I=1,
        scale=1.0 / math.sqrt(192.0), seed=5, lengths=[1048576, 524288, 262144, 4096],
        description="long-tail MLA stress: B=4, L={1M,512k,256k,4k}, dcp=8, bs=64, I=1"),
}


def make_seq_lens(cfg: Config) -> np.ndarray:
    """Context lengths (each counts the decode token itself)."""
    if isinstance(cfg.lengths, (list, tuple)):
        return np.asarray(cfg.lengths, dtype=np.int32)
    rng = np.random.default_rng(cfg.seed)
    out = np.empty(cfg.B, dtype=np.int64)
    if cfg.lengths == "bimodal":
        # 47% short-to-mid: uniform in [1024, 65536); 53% long: log-uniform in [65536, 262144]
        for b in range(cfg.B):
            if rng.random() < 0.47:
                out[b] = rng.integers(1024, 65536)
            else:
                out[b] = int(math.exp(rng.uniform(math.log(65536.0), math.log(262144.0))))
        out = np.clip(out, 1024, 262144)
    elif cfg.lengths == "uniform_32k_128k":
        out[:] = rng.integers(32768, 131072, size=cfg.B, endpoint=True)
    else:
        raise ValueError(cfg.lengths)
    return out.astype(np.int32)


def make_block_tables(seq_lens, dcp: int, bs: int, perm: str = "random", seed: int = 0,
                      max_vb: int | None = None):
    """Per-rank block tables BT[r][b][vb] -> physical block id, and the pool size.

    Every rank gets one physical block per virtual block vb < ceil(L_b / (bs*dcp)).
    Physical ids on rank r are a seeded random permutation (or the identity) of
    [0, num_blocks).  Unused entries are -1.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    nvb = (seq_lens + bs * dcp - 1) // (bs * dcp)
    if max_vb is None:
        max_vb = int(max(1, nvb.max()))
    num_blocks = int(nvb.sum())
    bt = np.full((dcp, len(seq_lens), max_vb), -1, dtype=np.int32)
    rng = np.random.default_rng(seed + 7919)
    for r in range(dcp):
        ids = np.arange(num_blocks, dtype=np.int32)
        if perm == "random":
            ids = rng.permutation(num_blocks).astype(np.int32)
        o = 0
        for b, n in enumerate(nvb):
            bt[r, b, :n] = ids[o:o + n]
            o += int(n)
    return bt, max(num_blocks, 1)


def make_topk(cfg: Config, seq_lens) -> np.ndarray:
    """Global top-k token indices per request, sampled without replacement from [0, L_b)."""
    out = np.empty((cfg.B, cfg.topk), dtype=np.int32)
    for b in range(cfg.B):
        rng = np.random.default_rng([cfg.seed, 104729, b])
        out[b] = rng.choice(int(seq_lens[b]), size=cfg.topk, replace=False).astype(np.int32)
    return out


def sink_logits(cfg: Config) -> np.ndarray:
    """One attention-sink logit per query head, N(0,1) from the value generator (fp32)."""
    return stream_values(cfg.seed, T_SINK, 0, 0, cfg.Hq, "f32").astype(np.float32)


# row widths of each value stream (elements per token / per request)
def row_elems(cfg: Config, tensor: int) -> int:
    if tensor == T_Q:
        return cfg.Hq * cfg.dk
    if tensor in (T_K, T_V):
        return cfg.Hkv * cfg.dk
    if tensor == T_LATENT:
        return cfg.dk
    raise ValueError(tensor)


def token_rows(cfg: Config, tensor: int, b: int, x0: int, x1: int) -> np.ndarray:
    """Rows of tokens [x0, x1) of request b: shape [x1-x0, row_elems] (fp32 or bf16 bits)."""
    w = row_elems(cfg, tensor)
    v = stream_values(cfg.seed, tensor, b, x0 * w, (x1 - x0) * w, cfg.dtype)
    return v.reshape(x1 - x0, w)


def query(cfg: Config, b: int) -> np.ndarray:
    """q of request b: [Hq, dk] (fp32 or bf16 bits)."""
    return stream_values(cfg.seed, T_Q, b, 0, cfg.Hq * cfg.dk, cfg.dtype).reshape(cfg.Hq, cfg.dk)


def _fill_at(key: int, idx: np.ndarray, table: np.ndarray, out: np.ndarray):
    u = _mix64_np((idx.astype(np.uint64) + np.uint64(1)) * np.uint64(GAMMA) + np.uint64(key))
    out[:] = table[(u >> np.uint64(48)).astype(np.intp)]


def head_rows(cfg: Config, tensor: int, b: int, h: int, x0: int, x1: int) -> np.ndarray:
    """GQA k or v of kv head h for tokens [x0, x1): [x1-x0, dk] (fp32 or bf16 bits).

    Generates only that head's elements (indices (x*Hkv + h)*dk + i of the stream).
    """
    table = value_table(cfg.dtype)
    key = stream_key(cfg.seed, tensor, b)
    n = x1 - x0
    out = np.empty((n, cfg.dk), dtype=table.dtype)
    step = max(1, (1 << 21) // cfg.dk)
    ar = np.arange(cfg.dk, dtype=np.int64)

    def work(s):
        e = min(n, s + step)
        x = np.arange(x0 + s, x0 + e, dtype=np.int64)
        idx = (x[:, None] * cfg.Hkv + h) * cfg.dk + ar[None, :]
        _fill_at(key, idx, table, out[s:e])

    futs = [_pool().submit(work, s) for s in range(0, n, step)]
    for f in futs:
        f.result()
    return out


def token_rows_at(cfg: Config, tensor: int, b: int, xs) -> np.ndarray:
    """Rows of the tokens xs (any order, any values >= 0) of request b:
    [len(xs), row_elems] (fp32 or bf16 bits), without generating the rest of
    the context (the sparse top-k checks need 2048 rows of a 128k context)."""
    table = value_table(cfg.dtype)
    key = stream_key(cfg.seed, tensor, b)
    w = row_elems(cfg, tensor)
    xs = np.asarray(xs, dtype=np.int64)
    out = np.empty((len(xs), w), dtype=table.dtype)
    if len(xs):
        idx = xs[:, None] * w + np.arange(w, dtype=np.int64)[None, :]
        _fill_at(key, idx, table, out)
    return out

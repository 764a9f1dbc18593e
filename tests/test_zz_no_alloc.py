"""dcp_decode_gqa_noalloc: the decode step for callers that cannot allocate.

Callers such as runtimes that own every byte of device memory, or C code
with no device allocator, call this entry point instead of dcp_decode_gqa;
its workspace lives in a fixed array inside the library.  These checks go
through the C ABI (the ctypes binding) and compare it bit for bit with
dcp_decode_gqa on calls in a row with different batches, so state left in
the shared array by one call cannot leak into the next.  Kept in its own file, named
to be collected last.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as W
from workloads import device as D

pytestmark = pytest.mark.gpu


def _compare(lib, wl, cfg, sink=None):
    out_ref, lse_ref = lib.decode_gqa(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale, sink=sink,
                                      out_dtype=torch.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = lib.decode_gqa_noalloc(wl.layout, wl.q, wl.kv, wl.local_lens, cfg.scale,
                                      sink=sink, out_dtype=torch.float32, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    # Both entry points run the same plan, split and merge kernels with the
    # same fixed merge order, so the results must be identical bit for bit:
    # any difference means the shared array fed stale state into the step.
    assert torch.isfinite(out).all()
    assert torch.equal(out.view(torch.int32), out_ref.view(torch.int32))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))


def test_noalloc_matches_decode_gqa_two_calls(lib):
    base = W.CONFIGS["gqa_bf16_b32"]
    lens = W.make_seq_lens(base)
    first = dataclasses.replace(base, B=6, lengths=[int(x) for x in lens[:6]])
    second = dataclasses.replace(base, B=3, lengths=[1, 700, 40000], dcp=4, bs=64, I=2, seed=9)
    wl1 = D.build(first)
    wl2 = D.build(second)
    sink = torch.from_numpy(np.linspace(-2, 2, second.Hq).astype(np.float32)).cuda()
    _compare(lib, wl1, first)
    _compare(lib, wl2, second, sink=sink)
    _compare(lib, wl1, first)


def test_noalloc_rejects_batches_beyond_the_fixed_scratch(lib):
    base = W.CONFIGS["gqa_bf16_b32"]
    B = 512
    layout = lib.Layout(base.dcp, base.bs, base.I)
    need = lib.decode_workspace_size(layout, lib.KIND_GQA, B, base.Hq, base.Hkv, base.dk)
    assert need > (16 << 20)
    q = torch.zeros((B, base.Hq, base.dk), dtype=torch.bfloat16, device="cuda")
    pools = [torch.zeros((1, base.Hkv, base.bs, base.dk), dtype=torch.bfloat16, device="cuda")
             for _ in range(base.dcp)]
    bt = torch.zeros((base.dcp, B, 1), dtype=torch.int32, device="cuda")
    kv = lib.PagedKV(pools, pools, bt, 1)
    local = torch.zeros((B, base.dcp), dtype=torch.int32, device="cuda")
    with pytest.raises(lib.DcpError, match="workspace"):
        lib.decode_gqa_noalloc(layout, q, kv, local, base.scale)

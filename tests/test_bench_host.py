"""Host-side helpers of bench.py (CPU only): the staged per-step buffers of the
end-to-end measurement, the BLAS thread count of the CPU baseline, and the
ncu traffic entries."""
import hashlib
import os

import pytest
import torch

import bench


def test_staged_views_hold_copies_at_aligned_offsets():
    q = torch.randn(3, 5, 7).to(torch.bfloat16)
    pos = torch.arange(11, dtype=torch.int64)
    lens = torch.tensor([4, 9, 2], dtype=torch.int32)
    buf, views = bench.staged([q, None, pos, lens], "cpu")
    vq, vnone, vpos, vlens = views
    assert vnone is None
    for v, t in ((vq, q), (vpos, pos), (vlens, lens)):
        assert v.shape == t.shape and v.dtype == t.dtype
        assert torch.equal(v, t)
        off = v.data_ptr() - buf.data_ptr()
        assert off % 256 == 0 and 0 <= off and off + v.numel() * v.element_size() <= buf.numel()
    # the views are the buffer: one copy into it refreshes every input
    host = buf.clone()
    host.view(torch.uint8).zero_()
    buf.copy_(host)
    assert not vq.float().any() and not vpos.any() and not vlens.any()


def test_staged_views_do_not_overlap():
    ts = [torch.ones(n, dtype=torch.float32) * (i + 1) for i, n in enumerate((1, 63, 64, 65, 300))]
    buf, views = bench.staged(ts, "cpu")
    spans = sorted((v.data_ptr(), v.data_ptr() + v.numel() * 4) for v in views)
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    for v, t in zip(views, ts):
        assert torch.equal(v, t)


def test_blas_threads_is_a_positive_count():
    n = bench.blas_threads()
    assert isinstance(n, int) and 1 <= n <= (os.cpu_count() or 1) * 4


@pytest.mark.parametrize("name", sorted(bench.NCU_TRAFFIC))
def test_traffic_entries_name_a_committed_capture(name):
    e = bench.NCU_TRAFFIC[name]
    root = os.path.dirname(os.path.abspath(bench.__file__))
    assert os.path.exists(os.path.join(root, e["source"]))
    assert os.path.exists(os.path.join(root, e["capture"]))
    assert e["dram_bytes"] > 0 and e["kv_bytes"] > 0
    # a kernel source changed since its capture reads as "no traffic", never as stale bytes
    with open(os.path.join(root, e["source"]), "rb") as f:
        current = hashlib.sha256(f.read()).hexdigest()[:16]
    t = bench.traffic_per_launch(name, e["kv_bytes"])
    if current == e["sha256_16"]:
        assert t == e["dram_bytes"]
    else:
        assert t is None


def test_cpu_baseline_reports_the_host_and_the_sample_share():
    import workloads as W
    cfg = W.CONFIGS["tiny_gqa_f32"]
    lens = W.make_seq_lens(cfg)
    cb = bench.cpu_baseline(cfg, lens, 0.01)
    assert cb["kind"] == "oracle" and cb["cores"] >= 1
    assert cb["nproc"] == os.cpu_count() and isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    assert cb["step_kv_bytes"] == bench.step_bytes(cfg, lens, cfg.B)[0]
    assert 0 < cb["sample_fraction_of_step"] <= 1.0
    assert cb["sample_kv_bytes"] == round(cb["sample_fraction_of_step"] * cb["step_kv_bytes"])


def test_both_arms_name_the_same_workload():
    import workloads as W
    cfg = W.CONFIGS["gqa_bf16_b32"]
    lens = W.make_seq_lens(cfg)
    c = bench.workload_config(cfg, lens, 1)
    assert c == bench.workload_config(cfg, lens.copy(), 1)
    assert c["kv_bytes_per_step"] == bench.step_bytes(cfg, lens, cfg.B)[0]
    assert set(c) == {"workload", "name", "batch", "context_tokens", "kv_bytes_per_step",
                      "parallelism"}
    sfa = W.CONFIGS["sfa_bf16_b32"]
    assert bench.workload_config(sfa, W.make_seq_lens(sfa), 1)["kv_bytes_per_step"] == 32 * 2048 * 1152

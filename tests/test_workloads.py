"""The seeded input generator: determinism, distribution, bf16 rounding."""
import numpy as np
import torch

import workloads as W


def test_table_is_normal_quantiles():
    t = W.value_table("f32").astype(np.float64)
    assert np.all(np.diff(t) > 0)
    np.testing.assert_allclose(t, -t[::-1], atol=1e-6)
    assert abs(t.mean()) < 1e-6 and abs(t.std() - 1.0) < 2e-3


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([1.00390625, 1.01171875, -3.0078125], np.float32)])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (ours == ref).all()
    assert (W.bf16_bits_to_f32(ours) == torch.from_numpy(x).to(torch.bfloat16).float().numpy()).all()


def test_streams_are_deterministic_and_sliceable():
    cfg = W.CONFIGS["gqa_bf16_b32"]
    a = W.stream_values(2, W.T_K, 3, 0, 5000, "bf16")
    b = W.stream_values(2, W.T_K, 3, 1000, 2000, "bf16")
    assert (a[1000:3000] == b).all()
    rows = W.token_rows(cfg, W.T_K, 3, 10, 20)
    for h in range(cfg.Hkv):
        assert (W.head_rows(cfg, W.T_K, 3, h, 10, 20) == rows[:, h * 128:(h + 1) * 128]).all()
    xs = np.array([17, 10, 19, 10])
    assert (W.token_rows_at(cfg, W.T_K, 3, xs) == rows[xs - 10]).all()
    sfa = W.CONFIGS["sfa_bf16_b32"]
    lat = W.token_rows(sfa, W.T_LATENT, 1, 0, 40)
    assert (W.token_rows_at(sfa, W.T_LATENT, 1, [39, 0, 7]) == lat[[39, 0, 7]]).all()
    other = W.stream_values(2, W.T_V, 3, 0, 5000, "bf16")
    assert (a != other).mean() > 0.9
    f = W.as_float64(W.stream_values(9, W.T_Q, 0, 0, 1 << 20, "bf16"), "bf16")
    assert abs(f.mean()) < 5e-3 and abs(f.std() - 1) < 5e-3


def test_config_lengths():
    L = W.make_seq_lens(W.CONFIGS["gqa_bf16_b32"])
    assert len(L) == 32 and L.min() >= 1024 and L.max() <= 262144
    L4 = W.make_seq_lens(W.CONFIGS["sfa_bf16_b32"])
    assert L4.min() >= 32768 and L4.max() <= 131072
    topk = W.make_topk(W.CONFIGS["sfa_bf16_b32"], L4)
    for b in range(32):
        assert len(set(topk[b].tolist())) == 2048 and topk[b].max() < L4[b]

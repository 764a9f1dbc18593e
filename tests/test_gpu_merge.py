"""dcp_lse_merge vs the oracle's merge, including empty parts and the sink."""
import math

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,B,H,dv", [(1, 1, 1, 4), (2, 3, 8, 64), (8, 32, 32, 128),
                                      (8, 4, 128, 512), (13, 2, 5, 1024),
                                      # more parts than a warp has lanes: LSEs in blocks of 32
                                      (33, 2, 4, 128), (70, 1, 3, 512)])
@pytest.mark.parametrize("with_sink", [False, True])
def test_merge_matches_oracle(lib, n, B, H, dv, with_sink):
    rng = np.random.default_rng(n * 31 + dv)
    po = rng.standard_normal((n, B, H, dv)).astype(np.float32)
    pl = (rng.standard_normal((n, B, H)) * 4).astype(np.float32)
    pl[rng.random((n, B, H)) < 0.2] = -np.inf
    if n > 1:
        pl[:, 0, 0] = -np.inf           # a row with every part empty
    po[np.isneginf(pl)] = np.nan        # an empty part adds nothing, whatever its o holds
    sink = rng.standard_normal(H).astype(np.float32) if with_sink else None
    out, lse = lib.lse_merge(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(),
                             None if sink is None else torch.from_numpy(sink).cuda())
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        for h in range(H):
            o_ref, l_ref = O.lse_merge(po[:, b, h].astype(np.float64), pl[:, b, h],
                                       None if sink is None else float(sink[h]))
            scale = max(1.0, float(np.abs(o_ref).max()))
            assert np.abs(out[b, h] - o_ref).max() <= 1e-5 * scale
            if math.isinf(l_ref):
                assert np.isneginf(lse[b, h])
            else:
                assert abs(lse[b, h] - l_ref) <= 1e-5 * max(1.0, abs(l_ref))


def test_merge_bf16_output_rounding(lib):
    rng = np.random.default_rng(3)
    po = rng.standard_normal((3, 2, 4, 128)).astype(np.float32)
    pl = rng.standard_normal((3, 2, 4)).astype(np.float32)
    o32, _ = lib.lse_merge(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda())
    o16, _ = lib.lse_merge(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(),
                           out_dtype=torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16))

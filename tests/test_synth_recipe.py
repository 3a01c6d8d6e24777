"""The synthetic workload recipe: shapes, byte counts and Zipf skew (CPU)."""
import numpy as np
import torch

from int4_routed_expert_06_b300 import synth
from oracle import oracle as O


def test_expert_bytes_match_layout_arithmetic():
    # 512x2048 int4 matrix, group 64, fp16 scale+bias: 524288 + 65536 bytes
    assert synth.bytes_per_qmatrix(512, 2048, 64, 2) == 589_824
    assert synth.expert_bytes(synth.DEC_80B) == 3 * 589_824
    assert synth.active_expert_bytes(synth.DEC_80B) == 19_464_192
    assert synth.active_expert_bytes(synth.DEC_35B) == 15_925_248
    # tiny: 32x64, group 32, fp32 scale+bias = 1024 + 512
    assert synth.bytes_per_qmatrix(32, 64, 32, 4) == 1536


def test_zipf_bias_gives_zipf_11_popularity():
    shp = synth.STACK_80B
    g = torch.Generator().manual_seed(3)
    wr = (torch.randn((shp.n_experts, shp.hidden), generator=g) * shp.router_std).to(torch.bfloat16)
    xs = torch.randn((800, shp.hidden), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    bias = synth.zipf_router_bias(shp, seed=4)
    lg, _ = O.router(xs, wr, bias)
    idx, _ = O.topk(lg, shp.top_k)
    freq = np.bincount(idx.ravel(), minlength=shp.n_experts) / len(xs)
    rank = np.argsort(np.argsort(-bias.numpy(), kind="stable"), kind="stable") + 1
    byrank = np.zeros(shp.n_experts)
    byrank[rank - 1] = freq
    r = np.arange(1, shp.n_experts + 1)
    m = (byrank < 0.9) & (byrank > 5.0 / len(xs))
    slope = np.polyfit(np.log(r[m]), np.log(byrank[m]), 1)[0]
    assert -1.3 < slope < -0.9, slope


def test_quantiser_codes_in_range_and_deterministic():
    shp = synth.TINY
    a = synth.make_layer(shp)
    b = synth.make_layer(shp)
    for k in a:
        if isinstance(a[k], torch.Tensor):
            assert torch.equal(a[k], b[k]), k
        else:
            assert a[k] == b[k], k
    q = a["q_gate"].view(torch.int32)
    assert q.dtype == torch.int32 and q.shape == (8, 32, 8)
    t = synth.shuffled_slots(512, 2)
    assert sorted(t.tolist()) == list(range(512))


def test_tiny_router_and_shared_gate_lie_on_the_affine4_grid():
    """The tiny workload quantises all its weights: its router and shared-gate
    rows, kept dense, hold at most 16 equally spaced values per group of 32
    (s * q + b with q in 0..15)."""
    shp = synth.TINY
    r = synth.make_router(shp)
    for wmat in (r["w_router"], r["w_shared_gate"][None]):
        g = wmat.double().reshape(-1, shp.group)
        lo = g.min(dim=1, keepdim=True).values
        step = (g.max(dim=1, keepdim=True).values - lo) / 15.0
        q = (g - lo) / step
        assert torch.allclose(q, q.round(), atol=1e-4)
        assert int(q.round().max()) <= 15 and int(q.round().min()) >= 0

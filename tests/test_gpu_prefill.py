"""GPU parity of the many-token path (tcgen05 grouped GEMMs) with the oracle.

Shapes: an 80B-shaped layer with 64 experts at ragged token counts (every
token checked), the same at T = 600 where the busiest expert spans several
256-token units (sampled tokens), and the full 80B prefill of 4096 tokens
with Zipf-skewed routing (sampled tokens, bucketing checked exactly).
"""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_util import assert_close, layer_forward, near_tie_tokens, workspace
from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth
from oracle import oracle as O

pytestmark = pytest.mark.gpu

SMALL = dataclasses.replace(synth.PREFILL_80B, name="prefill-64e", n_experts=64, top_k=8, tokens=96)


def _setup(shape, seed=7):
    w = synth.make_layer(shape, device="cuda")
    dl = B.DeviceLayer(shape, w, synth.shuffled_slots(shape.n_experts, seed))
    return w, dl, O.Layer(w, shape.group, shape.top_k)


@pytest.fixture(scope="module")
def small():
    return _setup(SMALL)


@pytest.mark.parametrize("T", [64, 96, 131])
def test_prefill_small_every_token(small, T):
    w, dl, L = small
    x = synth.make_x(SMALL, 70 + T, T, device="cuda")
    y, y32, idx, tw = layer_forward(dl, x)
    ref = L.forward(x)
    ok = ~near_tie_tokens(ref["logits"], SMALL.top_k)
    np.testing.assert_array_equal(idx.cpu().numpy()[ok], ref["idx"][ok])
    assert_close(y32.cpu().numpy()[ok], ref["y"][ok], "bf16", f"T={T} y_f32")
    assert_close(y.float().cpu().numpy()[ok], ref["y"][ok], "bf16", f"T={T} y")


def test_prefill_matches_generic_kernels(small):
    w, dl, L = small
    x = synth.make_x(SMALL, 5, 80, device="cuda")
    try:
        B.moe_set_kernel_path(0)
        a = layer_forward(dl, x)
        B.moe_set_kernel_path(1)
        b = layer_forward(dl, x)
    finally:
        B.moe_set_kernel_path(0)
    assert torch.equal(a[2], b[2])
    assert_close(a[1].cpu().numpy(), b[1].double().cpu().numpy(), "bf16", "grouped GEMM vs generic")


def _sampled_check(shape, w, L, dl, T, seed, n_sample):
    x = synth.make_x(shape, seed, T, device="cuda")
    y, y32, idx, tw = layer_forward(dl, x)
    idx_np = idx.cpu().numpy()
    # sample: seeded tokens plus tokens routed to the busiest expert
    rng = np.random.default_rng(seed)
    busiest = np.bincount(idx_np.ravel(), minlength=shape.n_experts).argmax()
    on_busiest = np.nonzero((idx_np == busiest).any(axis=1))[0]
    sample = sorted(set(rng.choice(T, n_sample, replace=False).tolist()) | set(on_busiest[-4:].tolist()))
    xs = x[sample]
    ref = L.forward(xs)
    ok = ~near_tie_tokens(ref["logits"], shape.top_k)
    np.testing.assert_array_equal(idx_np[sample][ok], ref["idx"][ok])
    assert_close(y32.cpu().numpy()[sample][ok], ref["y"][ok], "bf16", f"T={T} sampled")
    return idx_np


def test_prefill_multi_chunk_experts(small):
    w, dl, L = small
    idx = _sampled_check(SMALL, w, L, dl, 600, 11, 24)
    assert np.bincount(idx.ravel()).max() > 256          # the busiest expert spans several units


def test_prefill_80b_full_size_sampled():
    shape = synth.PREFILL_80B
    w, dl, L = _setup(shape, 2)
    idx = _sampled_check(shape, w, L, dl, shape.tokens, synth.PREFILL_X_SEED, 24)
    counts = np.bincount(idx.ravel(), minlength=shape.n_experts)
    assert counts.max() > 1000 and (counts == 0).sum() < shape.n_experts   # Zipf skew present
    # bucketing of this routing, exactly
    cfg = B.config_for(shape)
    d_idx = torch.from_numpy(idx).cuda()
    T, k, E = shape.tokens, shape.top_k, shape.n_experts
    c = torch.empty(E, dtype=torch.int32, device="cuda")
    o = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pt = torch.empty(T * k, dtype=torch.int32, device="cuda")
    pr = torch.empty(T * k, dtype=torch.int32, device="cuda")
    nb = B.moe_bucket_workspace_bytes(cfg, T)
    B.moe_bucket(cfg, d_idx, T, c, o, pt, pr, workspace(nb), nb)
    torch.cuda.synchronize()
    rc, ro, rt, rr = O.bucket(idx, E)
    assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(pt.cpu().numpy(), rt)
    assert np.array_equal(pr.cpu().numpy(), rr) and np.array_equal(o.cpu().numpy(), ro)

"""Parity of the affine int8 variant (8-bit codes, four a word, same groups,
scales and biases as int4) on the 35B- and 80B-shaped layers: the
single-token kernels and the generic ones at T = 1 against the oracle, a
ragged batch on the generic kernels, and one routed expert alone.

The Swiftlet README, "Relation to TurboFieldfare": MLX affine int4/int8 group
quantisation.
"""
import numpy as np
import pytest

from gpu_util import assert_close, device_layer, layer_forward, layer_of, near_tie_tokens, workspace
from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth
from oracle import oracle as O

pytestmark = pytest.mark.gpu

NAMES = ["35b-dec-int8", "80b-dec-int8"]


@pytest.fixture
def path():
    yield B.moe_set_kernel_path
    B.moe_set_kernel_path(0)


@pytest.mark.parametrize("kpath", [0, 1])
@pytest.mark.parametrize("name", NAMES)
def test_int8_decode_parity(name, kpath, path):
    """20 decode steps (the first 10 of the seeded sequence and 10 from the
    rest), each its own T = 1 call; near-tie steps counted, at most 1."""
    path(kpath)
    shape, w, L = layer_of(name)
    assert shape.bits == 8 and w["q_gate"].shape[-1] == shape.hidden // 4
    dl = device_layer(name)
    xs = synth.decode_xs(shape, 1000, device="cuda")
    rng = np.random.default_rng(8)
    steps = list(range(10)) + sorted(int(s) for s in rng.choice(np.arange(10, 1000), 10, replace=False))
    ties = 0
    for s in steps:
        x = xs[s:s + 1]
        y, y32, idx, tw = layer_forward(dl, x)
        ref = L.forward(x)
        if near_tie_tokens(ref["logits"], shape.top_k)[0]:
            ties += 1
            continue
        np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"], err_msg=f"{name} step {s}")
        np.testing.assert_allclose(tw.cpu().numpy(), ref["w"], rtol=2e-5, atol=1e-6)
        assert_close(y32.cpu().numpy(), ref["y"], shape.act, f"{name} step {s} y_f32")
        assert_close(y.float().cpu().numpy(), ref["y"], shape.act, f"{name} step {s} y")
    assert ties <= 1


@pytest.mark.parametrize("name,T", [("35b-dec-int8", 5), ("80b-dec-int8", 33), ("80b-dec-int8", 70)])
def test_int8_batched_tokens(name, T):
    """Several tokens in one call (generic kernels; T = 70 is past the
    many-token threshold, where the 8-bit codes also take the generic path)."""
    shape, w, L = layer_of(name)
    dl = device_layer(name)
    x = synth.make_x(shape, 321, T, device="cuda")
    y, y32, idx, tw = layer_forward(dl, x)
    ref = L.forward(x)
    ok = ~near_tie_tokens(ref["logits"], shape.top_k)
    assert ok.sum() >= T - 1
    np.testing.assert_array_equal(idx.cpu().numpy()[ok], ref["idx"][ok])
    assert_close(y32.cpu().numpy()[ok], ref["y"][ok], shape.act, f"{name} T={T}")


def test_int8_fast_and_generic_agree(path):
    name = "80b-dec-int8"
    shape, w, L = layer_of(name)
    dl = device_layer(name)
    xs = synth.decode_xs(shape, 4, device="cuda")
    for s in range(4):
        path(0)
        _, y0, i0, _ = layer_forward(dl, xs[s:s + 1])
        path(1)
        _, y1, i1, _ = layer_forward(dl, xs[s:s + 1])
        assert np.array_equal(i0.cpu().numpy(), i1.cpu().numpy())
        ref = L.forward(xs[s:s + 1])
        assert_close(y0.cpu().numpy(), y1.cpu().numpy().astype(np.float64), shape.act, "fast vs generic")
        assert_close(y0.cpu().numpy(), ref["y"], shape.act, "fast vs oracle")


def test_int8_expert_forward_parity():
    import torch
    name = "80b-dec-int8"
    shape, w, L = layer_of(name)
    T = 3
    x = synth.make_x(shape, 99, T, device="cuda")
    cfg = B.config_for(shape)
    assert cfg.bits == 8
    for e in (0, shape.n_experts - 1):
        ex = B.expert_struct(w, e)
        y = torch.empty((T, shape.hidden), dtype=torch.bfloat16, device="cuda")
        y32 = torch.empty((T, shape.hidden), device="cuda")
        nb = B.moe_expert_workspace_bytes(cfg, T)
        B.moe_expert_forward(cfg, ex, shape.inter, x, T, y, y32, workspace(nb), nb)
        torch.cuda.synchronize()
        view = O.ExpertView(w, e)
        assert view.bits == 8
        ref = np.stack([O.expert(view, shape.group, x[t]) for t in range(T)])
        assert_close(y32.cpu().numpy(), ref, shape.act, f"int8 expert {e}")

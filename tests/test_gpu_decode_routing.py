"""Routing on the single-token path (the selection every decode token of the
bench uses), driven into its corner cases through moe_layer_forward at T = 1
on the 80B-shaped layer: exact ties at the k-th place and at the top (the
lower expert id ranks first), all logits equal (every key a candidate), and
all of the top k inside one group of the selection's threshold step.

The router rows are edited in place on the device; the oracle sees the same
edited rows.  Identical rows give bit-identical fp32 logits on the GPU (each
row is computed by the same code on the same x) and identical fp64 logits in
the oracle, so these ties are exact on both sides and the indices must match
bit for bit.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_close, device_layer, layer_forward, layer_of
from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth
from oracle import oracle as O

pytestmark = pytest.mark.gpu

NAME = "80b-dec"


@pytest.fixture(scope="module")
def layer80():
    shape, w, _ = layer_of(NAME)
    dl = device_layer(NAME)
    orig = dl.replicas[0]["w_router"].clone()
    yield shape, w, dl
    dl.replicas[0]["w_router"].copy_(orig)
    torch.cuda.synchronize()


def _run(shape, w, dl, wr, x):
    """Forward x through dl with router rows wr (device bf16); the oracle on the
    same rows.  -> (gpu idx, gpu w, gpu y32, oracle result)."""
    dl.replicas[0]["w_router"].copy_(wr)
    torch.cuda.synchronize()
    B.moe_set_kernel_path(0)
    y, y32, idx, tw = layer_forward(dl, x)
    wo = dict(w)
    wo["w_router"] = wr
    ref = O.Layer(wo, shape.group, shape.top_k).forward(x)
    return idx.cpu().numpy()[0], tw.cpu().numpy()[0], y32.cpu().numpy(), ref


def test_exact_tie_at_the_kth_place_goes_to_the_lower_id(layer80):
    shape, w, dl = layer80
    k = shape.top_k
    x = synth.make_x(shape, 4242, 1, device="cuda")
    lg, _, ref_idx, _ = O.Layer(w, shape.group, k).route(x)
    order = np.argsort(-lg[0], kind="stable")
    top = set(order[:k].tolist())
    a = int(order[k - 1])
    outside = [e for e in range(shape.n_experts) if e not in top]
    above = min(e for e in outside if e > a)
    below = max(e for e in outside if e < a)
    for b, winner, loser in ((above, a, above), (below, below, a)):
        wr = w["w_router"].clone()
        wr[b] = wr[a]
        idx, tw, y32, ref = _run(shape, w, dl, wr, x)
        assert ref["idx"][0, k - 1] == winner and loser not in ref["idx"][0]
        np.testing.assert_array_equal(idx, ref["idx"][0])
        assert_close(y32, ref["y"], shape.act, f"tie at k-th place, copy {a} -> {b}")


def test_exact_tie_at_the_top_orders_by_id_with_equal_weights(layer80):
    shape, w, dl = layer80
    k = shape.top_k
    x = synth.make_x(shape, 4243, 1, device="cuda")
    lg, _, _, _ = O.Layer(w, shape.group, k).route(x)
    order = np.argsort(-lg[0], kind="stable")
    first = int(order[0])
    below = [e for e in range(first) if e not in set(order[:k].tolist())]
    assert below, "choose another x: the top expert has the lowest id"
    c = below[0]
    wr = w["w_router"].clone()
    wr[c] = wr[first]
    idx, tw, y32, ref = _run(shape, w, dl, wr, x)
    assert (idx[0], idx[1]) == (c, first)
    np.testing.assert_array_equal(idx, ref["idx"][0])
    assert tw[0] == tw[1]
    np.testing.assert_allclose(tw, ref["w"][0], rtol=1e-5, atol=1e-7)


def test_all_logits_equal_select_the_k_lowest_ids(layer80):
    """Every key is a candidate of the threshold step: the ranking runs over
    many candidates in batches of 32."""
    shape, w, dl = layer80
    k = shape.top_k
    x = synth.make_x(shape, 4244, 1, device="cuda")
    wr = w["w_router"][:1].expand(shape.n_experts, -1).contiguous()
    idx, tw, y32, ref = _run(shape, w, dl, wr, x)
    np.testing.assert_array_equal(idx, np.arange(k))
    np.testing.assert_array_equal(idx, ref["idx"][0])
    np.testing.assert_allclose(tw, np.full(k, 1.0 / k), rtol=1e-6)
    assert_close(y32, ref["y"], shape.act, "all logits equal")


@pytest.mark.parametrize("first", [16, 200, 502])
def test_top_k_inside_one_group(layer80, first):
    """The k largest logits belong to k consecutive experts (inside one group
    of the threshold step, or across the last ones); the other rows are
    small draws."""
    shape, w, dl = layer80
    k = shape.top_k
    x = synth.make_x(shape, 4245, 1, device="cuda")
    xf = x[0].float()
    wr = (w["w_router"].float() * 0.1)
    for j in range(k):
        wr[first + j] = xf * ((3.0 - 0.1 * j) / xf.norm())
    wr = wr.to(torch.bfloat16)
    idx, tw, y32, ref = _run(shape, w, dl, wr, x)
    np.testing.assert_array_equal(idx, np.arange(first, first + k))
    np.testing.assert_array_equal(idx, ref["idx"][0])
    assert_close(y32, ref["y"], shape.act, f"top k at {first}..")

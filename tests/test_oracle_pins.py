"""Pins of the CPU oracle against things other than itself (CPU only).

Each pin ties one oracle function to brute force, a closed form, an
independent library routine (numpy matmul, scipy softmax / expit, numpy stable
sort) or a hand-computed trace, chosen so that a plausible slip (a dropped
term, a wrong sign, a swapped nibble order, a transposed operand, a reversed
tie-break) fails at least one of them.
"""
import dataclasses
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special as sps
import torch

from int4_routed_expert_06_b300 import synth
from oracle import oracle as O
from oracle.slot_policy import PoolExhausted, SlotPolicy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- top-k

def _brute_topk(logits, k):
    """Best k-subset by logit sum (tie-free inputs), ordered by logit desc."""
    best = max(itertools.combinations(range(len(logits)), k), key=lambda c: sum(logits[list(c)]))
    return sorted(best, key=lambda e: -logits[e])


@pytest.mark.parametrize("E,k,seed", [(8, 2, s) for s in range(20)] + [(16, 3, s) for s in range(10)]
                         + [(12, 5, 3), (9, 1, 4)])
def test_topk_brute_force(E, k, seed):
    lg = np.random.default_rng(seed).normal(size=E)
    idx, w = O.topk(lg, k)
    assert list(idx) == _brute_topk(lg, k)


def test_topk_ties_lower_id_first():
    lg = np.array([1.0, 3.0, 3.0, 2.0, 3.0])
    assert list(O.topk(lg, 1)[0]) == [1]
    assert list(O.topk(lg, 2)[0]) == [1, 2]
    assert list(O.topk(lg, 4)[0]) == [1, 2, 4, 3]
    assert list(O.topk(np.zeros(6), 3)[0]) == [0, 1, 2]


@pytest.mark.parametrize("E,k", [(8, 2), (256, 8), (512, 10), (64, 64), (40, 1)])
def test_topk_weights_equal_softmax_then_renormalise(E, k):
    lg = np.random.default_rng(E * 7 + k).normal(scale=2.0, size=E)
    idx, w = O.topk(lg, k)
    full = sps.softmax(lg)                       # library softmax over all E
    ref = full[idx] / full[idx].sum()            # then renormalise over the k
    np.testing.assert_allclose(w, ref, rtol=1e-13, atol=0)
    assert abs(w.sum() - 1.0) < 1e-12
    assert np.all(np.diff(w) <= 0)               # descending score, descending weight
    if k == E:
        np.testing.assert_allclose(w, np.sort(full)[::-1], rtol=1e-13)
    if k == 1:
        assert w[0] == 1.0


# --------------------------------------------------------------- dequant

@pytest.mark.parametrize("sd,group,n_out,n_in", [("f32", 32, 24, 64), ("f16", 64, 16, 256),
                                                 ("f32", 128, 8, 512)])
def test_dequant_reproduces_quantised_draws(sd, group, n_out, n_in):
    """Affine grid round trip: dequant(quantise(w)) is within half a step of w.
    A swapped nibble order or transposed scale index would miss by up to 15 steps."""
    g = torch.Generator().manual_seed(11)
    w = torch.randn((n_out, n_in), generator=g) * 0.05
    q, s, b = synth.quantise_affine4(w, group, synth.torch_dtype(sd))
    W = O.dequant(q, s, b, group)
    step = np.repeat(O.f64(s), group, axis=1)
    err = np.abs(W - w.double().numpy())
    slack = 0.0 if sd == "f32" else 2.0 ** -10 * (np.abs(np.repeat(O.f64(b), group, 1)) + 15 * step)
    assert np.all(err <= step * (0.5 + 1e-5) + slack + 1e-12)
    assert err.max() > 0.1 * step.min()          # not accidentally exact


def test_dequant_closed_forms():
    n_out, n_in, G = 4, 64, 32
    rng = np.random.default_rng(0)
    s = rng.uniform(0.01, 0.1, size=(n_out, n_in // G))
    b = rng.normal(size=(n_out, n_in // G))
    zero = np.zeros((n_out, n_in // 8), np.uint32)
    np.testing.assert_array_equal(O.dequant(zero, s, b, G), np.repeat(b, G, axis=1))
    full = np.full((n_out, n_in // 8), 0xFFFFFFFF, np.uint32)
    np.testing.assert_allclose(O.dequant(full, s, b, G), np.repeat(15 * s + b, G, axis=1), rtol=1e-15)
    # one code in one known place: row 2, column 13 -> word 1, nibble 5
    one = zero.copy()
    one[2, 1] = 0x7 << 20
    D = O.dequant(one, s, b, G)
    expect = np.repeat(b, G, axis=1)
    expect[2, 13] += 7 * s[2, 0]
    np.testing.assert_allclose(D, expect, rtol=1e-15)


def test_qmatvec_matches_numpy_matmul_and_group_sum_identity():
    rng = np.random.default_rng(1)
    n_out, n_in, G = 12, 128, 64
    q = rng.integers(0, 2**32, size=(n_out, n_in // 8), dtype=np.uint32)
    s = rng.uniform(0.001, 0.02, size=(n_out, n_in // G))
    b = rng.normal(scale=0.02, size=(n_out, n_in // G))
    v = rng.normal(size=n_in)
    y = O.qmatvec(q, s, b, G, v)
    np.testing.assert_allclose(y, O.dequant(q, s, b, G) @ v, rtol=1e-12, atol=1e-14)
    # q = 0: y = sum_g bias_g * sum_{c in g} v_c
    z = O.qmatvec(np.zeros_like(q), s, b, G, v)
    np.testing.assert_allclose(z, b @ v.reshape(-1, G).sum(axis=1), rtol=1e-12, atol=1e-15)


def test_expert_matches_dense_numpy():
    shp = synth.TINY
    ex = synth.make_experts(shp, 2, shp.inter, seed=5)
    x = np.random.default_rng(2).normal(size=shp.hidden)
    for e in range(2):
        view = O.ExpertView(ex, e)
        Wg = O.dequant(ex["q_gate"][e], ex["s_gate"][e], ex["b_gate"][e], shp.group)
        Wu = O.dequant(ex["q_up"][e], ex["s_up"][e], ex["b_up"][e], shp.group)
        Wd = O.dequant(ex["q_down"][e], ex["s_down"][e], ex["b_down"][e], shp.group)
        assert Wg.shape == (shp.inter, shp.hidden) and Wd.shape == (shp.hidden, shp.inter)
        g, u = Wg @ x, Wu @ x
        ref = Wd @ (g * sps.expit(g) * u)        # silu(g) = g * logistic(g)
        np.testing.assert_allclose(O.expert(view, shp.group, x), ref, rtol=1e-12, atol=1e-14)


def test_dequant_int8_closed_forms_and_byte_placement():
    """8-bit codes: four a word, the lowest column in the lowest byte."""
    n_out, n_in, G = 4, 64, 32
    rng = np.random.default_rng(3)
    s = rng.uniform(0.001, 0.01, size=(n_out, n_in // G))
    b = rng.normal(size=(n_out, n_in // G))
    zero = np.zeros((n_out, n_in // 4), np.uint32)
    np.testing.assert_array_equal(O.dequant(zero, s, b, G, bits=8), np.repeat(b, G, axis=1))
    full = np.full((n_out, n_in // 4), 0xFFFFFFFF, np.uint32)
    np.testing.assert_allclose(O.dequant(full, s, b, G, bits=8), np.repeat(255 * s + b, G, axis=1), rtol=1e-15)
    # one code in one known place: row 1, column 45 -> word 11, byte 1; group 1
    one = zero.copy()
    one[1, 11] = 0xC8 << 8
    D = O.dequant(one, s, b, G, bits=8)
    expect = np.repeat(b, G, axis=1)
    expect[1, 45] += 200 * s[1, 1]
    np.testing.assert_allclose(D, expect, rtol=1e-15)
    # the same word read as 4-bit codes is a different matrix
    assert not np.allclose(O.dequant(one, s, b, G, bits=4)[:, :64], D)


@pytest.mark.parametrize("sd,group", [("f32", 64), ("f16", 64), ("f32", 32)])
def test_dequant_int8_round_trip_within_half_step(sd, group):
    g = torch.Generator().manual_seed(12)
    w = torch.randn((16, 256), generator=g) * 0.05
    q, s, b = synth.quantise_affine4(w, group, synth.torch_dtype(sd), bits=8)
    assert q.shape == (16, 64)
    W = O.dequant(q, s, b, group, bits=8)
    step = np.repeat(O.f64(s), group, axis=1)
    err = np.abs(W - w.double().numpy())
    slack = 0.0 if sd == "f32" else 2.0 ** -10 * (np.abs(np.repeat(O.f64(b), group, 1)) + 255 * step)
    assert np.all(err <= step * (0.5 + 1e-5) + slack + 1e-12)
    # 255 levels: the step is about 1/17 of the 4-bit step of the same rows
    _, s4, _ = synth.quantise_affine4(w, group, synth.torch_dtype(sd), bits=4)
    np.testing.assert_allclose(O.f64(s4) / O.f64(s), 17.0, rtol=2e-3)


def test_qmatvec_int8_matches_numpy_matmul():
    rng = np.random.default_rng(4)
    n_out, n_in, G = 10, 256, 64
    q = rng.integers(0, 2**32, size=(n_out, n_in // 4), dtype=np.uint32)
    s = rng.uniform(0.0001, 0.002, size=(n_out, n_in // G))
    b = rng.normal(scale=0.02, size=(n_out, n_in // G))
    v = rng.normal(size=n_in)
    codes = np.stack([(q >> (8 * j)) & 0xFF for j in range(4)], axis=2).reshape(n_out, n_in)
    W = codes * np.repeat(s, G, axis=1) + np.repeat(b, G, axis=1)   # built here, not by the oracle
    np.testing.assert_allclose(O.qmatvec(q, s, b, G, v, bits=8), W @ v, rtol=1e-12, atol=1e-14)


def test_expert_int8_matches_dense_numpy():
    shp = dataclasses.replace(synth.TINY, bits=8)
    ex = synth.make_experts(shp, 2, shp.inter, seed=6)
    ex["bits"] = 8
    assert ex["q_gate"].shape[-1] == shp.hidden // 4
    x = np.random.default_rng(5).normal(size=shp.hidden)
    for e in range(2):
        view = O.ExpertView(ex, e)
        assert view.bits == 8 and view.hidden == shp.hidden
        Wg, Wu, Wd = (O.dequant(ex["q_" + m][e], ex["s_" + m][e], ex["b_" + m][e], shp.group, bits=8)
                      for m in ("gate", "up", "down"))
        g, u = Wg @ x, Wu @ x
        ref = Wd @ (g * sps.expit(g) * u)
        np.testing.assert_allclose(O.expert(view, shp.group, x), ref, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------- layer

def _tiny_layer():
    shp = synth.TINY
    return shp, synth.make_layer(shp), synth.make_x(shp, synth.TINY_X_SEED)


def test_tiny_router_is_tie_free():
    shp, layer, x = _tiny_layer()
    logits, _ = O.router(x, layer["w_router"])
    srt = np.sort(logits, axis=1)[:, ::-1]
    gap = srt[:, shp.top_k - 1] - srt[:, shp.top_k]
    assert gap.min() >= 1e-3, gap


def test_router_matches_numpy_and_bias_shifts():
    shp, layer, x = _tiny_layer()
    xd, wr = O.f64(x), O.f64(layer["w_router"])
    bias = np.linspace(-1, 1, shp.n_experts)
    lg, s = O.router(x, wr, bias, layer["w_shared_gate"])
    np.testing.assert_allclose(lg, xd @ wr.T + bias, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(s, xd @ O.f64(layer["w_shared_gate"]), rtol=1e-13)


def test_layer_matches_independent_composition():
    shp, layer, x = _tiny_layer()
    L = O.Layer(layer, shp.group, shp.top_k)
    out = L.forward(x)
    xd = O.f64(x)
    lg = xd @ O.f64(layer["w_router"]).T
    s = xd @ O.f64(layer["w_shared_gate"])

    def dense(pfx, e):
        return [O.dequant(layer[pfx + "q_" + m][e], layer[pfx + "s_" + m][e], layer[pfx + "b_" + m][e],
                          shp.group) for m in ("gate", "up", "down")]

    for t in range(shp.tokens):
        order = np.argsort(-lg[t], kind="stable")[: shp.top_k]
        p = sps.softmax(lg[t])[order]
        p = p / p.sum()
        y = np.zeros(shp.hidden)
        for e, pe in zip(order, p):
            Wg, Wu, Wd = dense("", e)
            y += pe * (Wd @ (Wg @ xd[t] * sps.expit(Wg @ xd[t]) * (Wu @ xd[t])))
        Wg, Wu, Wd = dense("shared_", 0)
        y += sps.expit(s[t]) * (Wd @ (Wg @ xd[t] * sps.expit(Wg @ xd[t]) * (Wu @ xd[t])))
        assert list(out["idx"][t]) == list(order)
        np.testing.assert_allclose(out["y"][t], y, rtol=1e-11, atol=1e-13)


def test_layer_batch_permutation_and_token_independence():
    shp, layer, x = _tiny_layer()
    L = O.Layer(layer, shp.group, shp.top_k)
    y = L.forward(x)["y"]
    perm = [2, 0, 3, 1]
    yp = L.forward(x[perm])["y"]
    np.testing.assert_array_equal(yp, y[perm])            # bit-exact
    for t in range(shp.tokens):
        np.testing.assert_array_equal(L.forward(x[t:t + 1])["y"][0], y[t])


def test_layer_identical_experts_closed_form():
    """All routed experts equal => the renormalised weights sum to one and
    y = E(x) + sigmoid(s) * E_shared(x)."""
    shp, layer, x = _tiny_layer()
    same = dict(layer)
    for m in ("gate", "up", "down"):
        for p in ("q_", "s_", "b_"):
            same[p + m] = layer[p + m][:1].expand_as(layer[p + m]).contiguous()
    L = O.Layer(same, shp.group, shp.top_k)
    out = L.forward(x)
    ev = O.ExpertView(same, 0)
    for t in range(shp.tokens):
        ref = O.expert(ev, shp.group, x[t]) + O.sigmoid(out["s"][t]) * O.expert(L.shared, shp.group, x[t])
        np.testing.assert_allclose(out["y"][t], ref, rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------- bucketing

@pytest.mark.parametrize("T,k,E,seed", [(1, 10, 512, 0), (4, 2, 8, 1), (97, 8, 256, 2), (300, 10, 64, 3)])
def test_bucket_matches_stable_sort(T, k, E, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, pt, pr = O.bucket(idx, E)
    np.testing.assert_array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    order = np.argsort(idx.ravel(), kind="stable")         # pairs in (expert, token, rank) order
    np.testing.assert_array_equal(pt, order // k)
    np.testing.assert_array_equal(pr, order % k)


# --------------------------------------------------------------- slot policy

def test_slot_policy_golden_traces():
    with open(os.path.join(GOLDEN, "slot_policy_traces.json")) as f:
        traces = json.load(f)["traces"]
    for tr in traces:
        pol = SlotPolicy(1, tr["n_experts"], tr["n_slots"], tr.get("rule", "lfu_recency"))
        for st in tr["steps"]:
            before = list(pol.table[0])
            slots, fills = pol.lookup(0, st["need"])
            assert [list(f) for f in fills] == st["fills"], (tr["name"], st)
            evicted = [e for e in range(tr["n_experts"]) if before[e] >= 0 and pol.table[0][e] < 0]
            assert sorted(evicted) == sorted(st["evicted"]), (tr["name"], st)
            assert pol.table[0] == st["table"], (tr["name"], st)
            assert slots == [st["table"][e] for e in st["need"]]
        assert (pol.hits, pol.misses, pol.evictions) == (tr["hits"], tr["misses"], tr["evictions"])


def test_slot_policy_exhaustion_and_layers_independent():
    pol = SlotPolicy(2, 8, 2)
    with pytest.raises(PoolExhausted):
        pol.lookup(0, [0, 1, 2])
    pol.lookup(0, [0, 1])
    pol.lookup(1, [2, 3])
    assert pol.table[0][:4] == [0, 1, -1, -1] and pol.table[1][:4] == [-1, -1, 0, 1]


def test_openmp_build_gives_the_same_doubles():
    """The all-cores build of the oracle (OpenMP over output rows, used only
    to time the CPU baseline) computes every output exactly as the plain build."""
    for shp, x in ((synth.TINY, synth.make_x(synth.TINY, synth.TINY_X_SEED)),
                   (synth.DEC_35B, synth.make_x(synth.DEC_35B, 1234, 1))):
        w = synth.make_layer(shp)
        ref = O.Layer(w, shp.group, shp.top_k).forward(x)
        O.set_threads(4)
        try:
            got = O.Layer(w, shp.group, shp.top_k).forward(x)
        finally:
            O.set_threads(1)
        assert np.array_equal(got["y"], ref["y"]) and np.array_equal(got["idx"], ref["idx"])
        assert np.array_equal(got["logits"], ref["logits"])

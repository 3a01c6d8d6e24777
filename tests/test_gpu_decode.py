"""GPU parity of the decode path against the CPU oracle, through the C-ABI.

Routing indices are compared bit-exactly, outputs within the stated
tolerance; workloads are the tiny layer and the 35B- and 80B-shaped layers at
their full sizes, in the launch configuration the bench times (T = 1).
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, assert_close, device_layer, layer_forward, layer_of, near_tie_tokens, workspace
from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth
from oracle import oracle as O

pytestmark = pytest.mark.gpu

NAMES = ["tiny", "35b-dec", "80b-dec"]


def _xs(name, n):
    shape = synth.SHAPES[name]
    if name == "tiny":
        return synth.make_x(shape, synth.TINY_X_SEED, device="cuda")
    return synth.decode_xs(shape, n, device="cuda")


def _route(dl, x, w):
    shape = dl.shape
    T = x.shape[0]
    idx = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
    tw = torch.empty((T, shape.top_k), dtype=torch.float32, device="cuda")
    sg = torch.empty((T,), dtype=torch.float32, device="cuda")
    lg = torch.empty((T, shape.n_experts), dtype=torch.float32, device="cuda")
    rep = dl.replicas[0]
    B.moe_route(dl.cfg, x, T, rep["w_router"], rep["router_bias"], rep["w_shared_gate"], idx, tw, sg, lg)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), tw.cpu().numpy(), sg.cpu().numpy(), lg.cpu().numpy()


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("T", [1, 13, 64])
def test_route_parity(name, T):
    shape, w, L = layer_of(name)
    dl = device_layer(name)
    x = _xs(name, 64)[:T] if name != "tiny" else _xs(name, 4)[: min(T, 4)]
    idx, tw, sg, lg = _route(dl, x, w)
    ref_lg, ref_s, ref_idx, ref_w = L.route(x)
    scale = np.abs(ref_lg).max()
    np.testing.assert_allclose(lg, ref_lg, rtol=0, atol=2e-5 * scale)
    np.testing.assert_allclose(sg, ref_s, rtol=0, atol=2e-5 * max(1.0, np.abs(ref_s).max()))
    tie = near_tie_tokens(ref_lg, shape.top_k)
    assert tie.sum() <= max(1, len(x) // 50), "too many near-ties for a seeded workload"
    np.testing.assert_array_equal(idx[~tie], ref_idx[~tie])
    # selection and weights on the GPU's own fp32 logits: exact selection
    own_idx, own_w = O.topk(lg.astype(np.float64), shape.top_k)
    np.testing.assert_array_equal(idx, own_idx)
    np.testing.assert_allclose(tw, own_w, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(tw.sum(axis=1), 1.0, rtol=1e-5)


def test_topk_ties_and_k_equals_e_on_device():
    """Exact ties pick the lower expert id; k = E gives a full softmax order."""
    cfg = B.config_for(synth.TINY)
    cfg.top_k = 8
    H, E = 64, 8
    x = torch.zeros((2, H), device="cuda")
    x[:, 0] = 1.0
    wr = torch.zeros((E, H), device="cuda")
    wr[:, 0] = torch.tensor([1.0, 3.0, 3.0, 2.0, 3.0, -1.0, 0.5, 3.0])
    wsg = torch.zeros(H, device="cuda")
    idx = torch.empty((2, 8), dtype=torch.int32, device="cuda")
    tw = torch.empty((2, 8), device="cuda")
    sg = torch.empty(2, device="cuda")
    lg = torch.empty((2, E), device="cuda")
    B.moe_route(cfg, x, 2, wr, None, wsg, idx, tw, sg, lg)
    torch.cuda.synchronize()
    assert idx[0].tolist() == [1, 2, 4, 7, 3, 0, 6, 5]
    ref_idx, ref_w = O.topk(wr[:, 0].double().cpu().numpy(), 8)
    np.testing.assert_allclose(tw[0].cpu().numpy(), ref_w, rtol=1e-6)
    cfg.top_k = 1
    B.moe_route(cfg, x, 2, wr, None, wsg, idx, tw, sg, lg)
    torch.cuda.synchronize()
    assert idx[0, 0].item() == 1 and tw[0, 0].item() == 1.0


@pytest.fixture
def kernel_path():
    """Select the single-token fast kernels (0) or the generic ones (1)."""
    def set_path(p):
        B.moe_set_kernel_path(p)
    yield set_path
    B.moe_set_kernel_path(0)


def _decode_sample(n_first=50, n_random=50, steps=1000, seed=77):
    """Decode steps checked: the first n_first of the seeded sequence and
    n_random more drawn (seeded) from the rest."""
    rng = np.random.default_rng(seed)
    rest = rng.choice(np.arange(n_first, steps), size=n_random, replace=False)
    return list(range(n_first)) + sorted(int(s) for s in rest)


@pytest.mark.parametrize("path", [0, 1])
@pytest.mark.parametrize("name", NAMES)
def test_layer_decode_parity(name, path, kernel_path):
    """T = 1 decode steps, each its own call (the bench's configuration), on
    the fast single-token kernels and on the generic ones: the tiny layer's
    tokens, and for the 35B- and 80B-shaped layers the first 50 steps of the
    seeded decode sequence plus 50 seeded random ones from the rest of its
    1000.  Routing must match the oracle exactly except on near-tie steps
    (gap between the k-th and (k+1)-th oracle logit within 1e-4 max(1, |l_k|)),
    which are counted: at most 2 of 100."""
    kernel_path(path)
    shape, w, L = layer_of(name)
    dl = device_layer(name)
    if name == "tiny":
        xs = _xs(name, 4)
        steps = list(range(len(xs)))
    else:
        xs = synth.decode_xs(shape, 1000, device="cuda")
        steps = _decode_sample()
    ties = 0
    for s in steps:
        x = xs[s:s + 1]
        y, y32, idx, tw = layer_forward(dl, x)
        ref = L.forward(x)
        if near_tie_tokens(ref["logits"], shape.top_k)[0]:
            ties += 1
            continue
        np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"], err_msg=f"{name} step {s}")
        assert_close(y32.cpu().numpy(), ref["y"], shape.act, f"{name} step {s} y_f32")
        assert_close(y.float().cpu().numpy(), ref["y"], shape.act, f"{name} step {s} y")
    assert ties <= 2, f"{ties} near-tie steps of {len(steps)}"


@pytest.mark.parametrize("name,T", [("tiny", 4), ("35b-dec", 5), ("80b-dec", 3), ("80b-dec", 12), ("80b-dec", 13)])
def test_layer_batched_tokens(name, T):
    """Several tokens in one call (ragged, not a multiple of any tile); on the
    80B layer T = 3 and 12 run the single-token kernels once a token, T = 13
    the generic kernels."""
    shape, w, L = layer_of(name)
    dl = device_layer(name)
    x = _xs(name, max(T, 8))[:T]
    y, y32, idx, tw = layer_forward(dl, x)
    ref = L.forward(x)
    ok = ~near_tie_tokens(ref["logits"], shape.top_k)
    np.testing.assert_array_equal(idx.cpu().numpy()[ok], ref["idx"][ok])
    assert_close(y32.cpu().numpy()[ok], ref["y"][ok], shape.act, f"{name} T={T}")


@pytest.mark.parametrize("name", ["tiny", "80b-dec"])
def test_expert_forward_parity(name):
    shape, w, L = layer_of(name)
    T = 3
    x = _xs(name, 4)[:T] if name != "tiny" else _xs(name, 4)[:T]
    for e in (0, shape.n_experts - 1):
        ex = B.expert_struct(w, e)
        y = torch.empty((T, shape.hidden), dtype=synth.torch_dtype(shape.act), device="cuda")
        y32 = torch.empty((T, shape.hidden), device="cuda")
        cfg = B.config_for(shape)
        nb = B.moe_expert_workspace_bytes(cfg, T)
        B.moe_expert_forward(cfg, ex, shape.inter, x, T, y, y32, workspace(nb), nb)
        torch.cuda.synchronize()
        view = O.ExpertView(w, e)
        ref = np.stack([O.expert(view, shape.group, x[t]) for t in range(T)])
        assert_close(y32.cpu().numpy(), ref, shape.act, f"expert {e}")


@pytest.mark.parametrize("name", ["35b-dec", "80b-dec"])
def test_route_then_experts_parity(name):
    """moe_route followed by moe_experts_forward (routing passed in) at T = 1."""
    shape, w, L = layer_of(name)
    dl = device_layer(name)
    xs = _xs(name, 4)
    rep = dl.replicas[0]
    nb = B.moe_layer_workspace_bytes(dl.cfg, 1)
    ws = workspace(nb)
    for s in range(4):
        x = xs[s:s + 1]
        idx = torch.empty((1, shape.top_k), dtype=torch.int32, device="cuda")
        tw = torch.empty((1, shape.top_k), device="cuda")
        sg = torch.empty((1,), device="cuda")
        y = torch.empty((1, shape.hidden), dtype=torch.bfloat16, device="cuda")
        y32 = torch.empty((1, shape.hidden), device="cuda")
        B.moe_route(dl.cfg, x, 1, rep["w_router"], rep["router_bias"], rep["w_shared_gate"], idx, tw, sg, None,
                    ws, nb)
        B.moe_experts_forward(dl.cfg, rep["struct"], x, 1, idx, tw, sg, y, y32, ws, nb)
        torch.cuda.synchronize()
        assert B.moe_get_device_error() == 0
        ref = L.forward(x)
        if near_tie_tokens(ref["logits"], shape.top_k)[0]:
            continue
        np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
        assert_close(y32.cpu().numpy(), ref["y"], shape.act, f"{name} step {s}")


def test_fast_and_generic_kernels_agree():
    """The single-token kernels and the generic ones compute the same layer.

    The single-token kernels carry x and a in 16-bit fixed point per
    32-column chunk (step = chunk max / 32767, so each element is off by at
    most 2^-16 of its chunk's largest magnitude) and the generic kernels in
    fp32.  Those errors are independent across the 2048- and 512-term sums,
    so the outputs differ by a few 2^-16 of the output scale; the bound below
    is 2^-11 of it (an order of magnitude of headroom), far inside the
    oracle tolerance both paths are held to."""
    name = "80b-dec"
    dl = device_layer(name)
    xs = _xs(name, 3)
    try:
        for s in range(3):
            B.moe_set_kernel_path(0)
            a = layer_forward(dl, xs[s:s + 1])
            B.moe_set_kernel_path(1)
            b = layer_forward(dl, xs[s:s + 1])
            assert torch.equal(a[2], b[2])                      # same routing
            d = (a[1] - b[1]).abs().max().item()
            assert d <= 2.0 ** -11 * max(1.0, b[1].abs().max().item()), d
    finally:
        B.moe_set_kernel_path(0)


def test_pool_placement_never_changes_the_result():
    """The same layer behind two different slot tables gives bit-identical y."""
    name = "80b-dec"
    a, b = device_layer(name, 0), device_layer(name, -1)
    xs = _xs(name, 4)
    for s in range(4):
        ya = layer_forward(a, xs[s:s + 1])
        yb = layer_forward(b, xs[s:s + 1])
        assert torch.equal(ya[0], yb[0]) and torch.equal(ya[1], yb[1]) and torch.equal(ya[2], yb[2])


def test_missing_slot_is_reported_not_faulted():
    name = "tiny"
    shape, w, L = layer_of(name)
    dl = B.DeviceLayer(shape, w, synth.shuffled_slots(shape.n_experts, 3))
    x = _xs(name, 4)
    ref = L.forward(x)
    gone = int(ref["idx"][0, 0])
    dl.replicas[0]["slots"][gone] = -1
    T = x.shape[0]
    y = torch.empty((T, shape.hidden), device="cuda")
    nb = B.moe_layer_workspace_bytes(dl.cfg, T)
    B.moe_layer_forward(dl.cfg, dl.struct(), x, T, y, workspace=workspace(nb), ws_bytes=nb)
    assert B.moe_get_device_error() == B.MOE_ERR_NOT_RESIDENT
    assert torch.isfinite(y).all()
    assert B.moe_get_device_error() == 0          # read-and-clear


@pytest.mark.parametrize("T,k,E", [(1, 10, 512), (97, 8, 256), (4096, 10, 512), (3000, 2, 8)])
def test_bucket_parity(T, k, E):
    rng = np.random.default_rng(T)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    cfg = B.config_for(synth.DEC_80B)
    cfg.n_experts, cfg.top_k = E, k
    d_idx = torch.from_numpy(idx).cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pt = torch.empty(T * k, dtype=torch.int32, device="cuda")
    pr = torch.empty(T * k, dtype=torch.int32, device="cuda")
    nb = B.moe_bucket_workspace_bytes(cfg, T)
    B.moe_bucket(cfg, d_idx, T, counts, offsets, pt, pr, workspace(nb), nb)
    torch.cuda.synchronize()
    rc, ro, rt, rr = O.bucket(idx, E)
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(pt.cpu().numpy(), rt)
    np.testing.assert_array_equal(pr.cpu().numpy(), rr)
    assert B.moe_get_device_error() == 0

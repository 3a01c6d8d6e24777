"""Small decode batches (T = 2 ... 64) on the tensor cores: kernel path 2
sends them through the tcgen05 grouped GEMMs (token columns padded to 16)
instead of the generic kernels.  Every token is checked against the oracle
on the 80B-shaped layer, and against the generic kernels.

The Swiftlet README, "Four ways to use it": the OpenAI-compatible server batches the
tokens of concurrent sequences into one layer call.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_close, device_layer, layer_forward, layer_of, near_tie_tokens
from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth

pytestmark = pytest.mark.gpu

NAME = "80b-dec"


@pytest.fixture
def path():
    yield B.moe_set_kernel_path
    B.moe_set_kernel_path(0)


@pytest.mark.parametrize("T", [2, 8, 33, 64])
def test_small_batch_on_grouped_gemm_every_token(T, path):
    shape, w, L = layer_of(NAME)
    dl = device_layer(NAME)
    x = synth.make_x(shape, 900 + T, T, device="cuda")
    path(2)
    y, y32, idx, tw = layer_forward(dl, x)
    ref = L.forward(x)
    ok = ~near_tie_tokens(ref["logits"], shape.top_k)
    assert ok.sum() >= T - 1
    np.testing.assert_array_equal(idx.cpu().numpy()[ok], ref["idx"][ok])
    np.testing.assert_allclose(tw.cpu().numpy()[ok], ref["w"][ok], rtol=2e-5, atol=1e-6)
    assert_close(y32.cpu().numpy()[ok], ref["y"][ok], shape.act, f"T={T} y_f32")
    assert_close(y.float().cpu().numpy()[ok], ref["y"][ok], shape.act, f"T={T} y")


@pytest.mark.parametrize("T", [2, 16])
def test_small_batch_grouped_matches_generic(T, path):
    shape, w, L = layer_of(NAME)
    dl = device_layer(NAME)
    x = synth.make_x(shape, 950 + T, T, device="cuda")
    path(2)
    a = layer_forward(dl, x)
    path(1)
    b = layer_forward(dl, x)
    assert torch.equal(a[2], b[2])
    assert_close(a[1].cpu().numpy(), b[1].double().cpu().numpy(), shape.act, "grouped GEMM vs generic")


def test_workspace_size_follows_the_path(path):
    shape, w, L = layer_of(NAME)
    cfg = B.config_for(shape)
    path(0)
    n0 = B.moe_layer_workspace_bytes(cfg, 8)
    path(2)
    n2 = B.moe_layer_workspace_bytes(cfg, 8)
    assert n2 > n0

"""Failure path of a bounded device wait, without a fault.

A test hook (moe_debug_set_waits) shortens every device wait to 1 ms and
makes the single-token down kernel's copy barrier expect one arrival that
never comes, so that wait must run out.  The call has to return normally,
with MOE_ERR_TIMEOUT in the device error word (read and cleared by
moe_get_device_error); the kernel supplies the missing arrival itself, lets
its copies land and writes zeros.  With the hook reset, the next call must
match the oracle again.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_close, device_layer, layer_of, near_tie_tokens, workspace
from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth

pytestmark = pytest.mark.gpu

DEFAULT_WAIT_NS = 200_000_000


@pytest.fixture
def restore_waits():
    yield
    B.moe_debug_set_waits(DEFAULT_WAIT_NS, 0)


def _call(dl, x):
    shape = dl.shape
    y = torch.full((1, shape.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    y32 = torch.full((1, shape.hidden), float("nan"), device="cuda")
    idx = torch.empty((1, shape.top_k), dtype=torch.int32, device="cuda")
    nb = B.moe_layer_workspace_bytes(dl.cfg, 1)
    ws = workspace(nb)
    B.moe_set_kernel_path(0)
    B.moe_layer_forward(dl.cfg, dl.struct(), x, 1, y, y32, idx, None, ws, nb)
    return y, y32, idx


def test_wait_that_runs_out_is_reported_then_the_next_call_is_right(restore_waits):
    name = "80b-dec"
    shape, w, L = layer_of(name)
    dl = device_layer(name)
    xs = synth.decode_xs(shape, 2, device="cuda")
    assert B.moe_get_device_error() == 0
    B.moe_debug_set_waits(1_000_000, 1)
    y, y32, idx = _call(dl, xs[0:1])
    assert B.moe_get_device_error() == B.MOE_ERR_TIMEOUT
    assert torch.isfinite(y32).all()           # zeros, not garbage
    assert B.moe_get_device_error() == 0       # read and cleared
    B.moe_debug_set_waits(DEFAULT_WAIT_NS, 0)
    y, y32, idx = _call(dl, xs[1:2])
    assert B.moe_get_device_error() == 0
    ref = L.forward(xs[1:2])
    if not near_tie_tokens(ref["logits"], shape.top_k)[0]:
        np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
    assert_close(y32.cpu().numpy(), ref["y"], shape.act, "call after the timeout")

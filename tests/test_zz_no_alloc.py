"""The allocation-free layer entry point (collected last on purpose).

moe_layer_forward_noalloc is for callers that cannot allocate device memory
where they run the layer; its scratch is built into the library.  It must
give the same result as moe_layer_forward with a caller workspace, call after
call, whether it runs alone in a fresh process or after every other test.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL
from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "35b-dec"])
def test_noalloc_matches_layer_forward_on_consecutive_calls(name):
    shape = synth.SHAPES[name]
    w = synth.make_layer(shape, device="cuda")
    dl = B.DeviceLayer(shape, w, synth.shuffled_slots(shape.n_experts, 11))
    T = shape.tokens
    act = synth.torch_dtype(shape.act)
    nb = B.moe_layer_workspace_bytes(dl.cfg, T)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    mx, rl = TOL[shape.act]
    for call, seed in enumerate((21, 22)):
        x = synth.make_x(shape, seed, T, device="cuda")
        y_ref = torch.empty((T, shape.hidden), dtype=act, device="cuda")
        y32_ref = torch.empty((T, shape.hidden), device="cuda")
        idx_ref = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
        B.moe_layer_forward(dl.cfg, dl.struct(), x, T, y_ref, y32_ref, idx_ref, None, ws, nb)
        y = torch.full((T, shape.hidden), float("nan"), dtype=act, device="cuda")
        y32 = torch.full((T, shape.hidden), float("nan"), device="cuda")
        idx = torch.full((T, shape.top_k), -1, dtype=torch.int32, device="cuda")
        B.moe_layer_forward_noalloc(dl.cfg, dl.struct(), x, T, y, y32, idx)
        torch.cuda.synchronize()
        assert B.moe_get_device_error() == 0
        assert torch.equal(idx, idx_ref), f"call {call}"
        got, ref = y32.double().cpu().numpy(), y32_ref.double().cpu().numpy()
        err = np.abs(got - ref).max()
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert err <= mx and rel <= rl, f"call {call}: max-abs {err}, rel-L2 {rel}"
        assert torch.isfinite(y.float()).all()


@pytest.mark.gpu
def test_noalloc_rejects_tokens_beyond_its_scratch():
    shape = synth.DEC_80B
    cfg = B.config_for(shape)
    big = 4096
    assert B.moe_layer_workspace_bytes(cfg, big) > 4 << 20
    with pytest.raises(B.MoEError) as ei:
        B.moe_layer_forward_noalloc(cfg, B.moe_layer(), 0x1000, big, 0x2000)
    assert ei.value.status == B.MOE_ERR_OOM and "scratch" in ei.value.message

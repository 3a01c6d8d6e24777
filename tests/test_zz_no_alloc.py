"""The allocation-free layer entry point (collected last on purpose).

moe_layer_forward_noalloc is for callers that cannot allocate device memory
where they run the layer; its scratch is built into the library.  It runs
the same kernels as moe_layer_forward with a caller workspace, so its results
must be bit-identical to that call's, call after call, whether it runs alone
in a fresh process or after every other test: the single-token path (T = 1),
the tiny layer, and the many-token generic path with the tensor-core router
(T = 16, 32 and 63, the largest T whose scratch fits).
"""
import pytest
import torch

from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth

SCRATCH = 4 << 20


@pytest.mark.gpu
@pytest.mark.parametrize("name,T", [("tiny", 4), ("35b-dec", 1), ("80b-dec", 1), ("80b-dec", 16),
                                    ("80b-dec", 32), ("80b-dec", 63)])
def test_noalloc_matches_layer_forward_on_consecutive_calls(name, T):
    shape = synth.SHAPES[name]
    w = synth.make_layer(shape, device="cuda")
    dl = B.DeviceLayer(shape, w, synth.shuffled_slots(shape.n_experts, 11))
    act = synth.torch_dtype(shape.act)
    nb = B.moe_layer_workspace_bytes(dl.cfg, T)
    assert nb <= SCRATCH
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((21, 22)):
        x = synth.make_x(shape, seed, T, device="cuda")
        y_ref = torch.empty((T, shape.hidden), dtype=act, device="cuda")
        y32_ref = torch.empty((T, shape.hidden), device="cuda")
        idx_ref = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
        w_ref = torch.empty((T, shape.top_k), device="cuda")
        B.moe_layer_forward(dl.cfg, dl.struct(), x, T, y_ref, y32_ref, idx_ref, w_ref, ws, nb)
        y = torch.full((T, shape.hidden), float("nan"), dtype=act, device="cuda")
        y32 = torch.full((T, shape.hidden), float("nan"), device="cuda")
        idx = torch.full((T, shape.top_k), -1, dtype=torch.int32, device="cuda")
        tw = torch.full((T, shape.top_k), float("nan"), device="cuda")
        B.moe_layer_forward_noalloc(dl.cfg, dl.struct(), x, T, y, y32, idx, tw)
        torch.cuda.synchronize()
        assert B.moe_get_device_error() == 0
        assert torch.equal(idx, idx_ref), f"call {call}"
        assert torch.equal(tw, w_ref), f"call {call}"
        assert torch.equal(y32, y32_ref), f"call {call}"
        assert torch.equal(y, y_ref), f"call {call}"


@pytest.mark.gpu
def test_noalloc_rejects_tokens_beyond_its_scratch():
    shape = synth.DEC_80B
    cfg = B.config_for(shape)
    for big in (64, 4096):
        assert B.moe_layer_workspace_bytes(cfg, big) > SCRATCH
        with pytest.raises(B.MoEError) as ei:
            B.moe_layer_forward_noalloc(cfg, B.moe_layer(), 0x1000, big, 0x2000)
        assert ei.value.status == B.MOE_ERR_OOM and "scratch" in ei.value.message

"""Shared helpers of the GPU parity tests (imported by test modules only)."""
import functools

import numpy as np
import torch

from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth
from oracle import oracle as O

# Tolerances of the layer output against the fp64 oracle.
#  bf16 activations, fp32 accumulation: max-abs <= 2e-2 and rel-L2 <= 5e-3.
#  fp32 activations (tiny workload): 1e-4 on both.
TOL = {"bf16": (2e-2, 5e-3), "f32": (1e-4, 1e-4)}


def rel_l2(a, b) -> float:
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def assert_close(got, ref, act: str, what: str = ""):
    mx, rl = TOL[act]
    got = np.asarray(got, np.float64)
    err = float(np.abs(got - ref).max())
    r = rel_l2(got, ref)
    assert err <= mx and r <= rl, f"{what}: max-abs {err:.3g} (<= {mx}), rel-L2 {r:.3g} (<= {rl})"
    return err, r


@functools.lru_cache(maxsize=4)
def layer_of(name: str):
    """(shape, weights on cuda, oracle Layer) for a named workload."""
    shape = synth.SHAPES[name]
    w = synth.make_layer(shape, device="cuda")
    return shape, w, O.Layer(w, shape.group, shape.top_k)


@functools.lru_cache(maxsize=4)
def device_layer(name: str, table_seed: int = 0):
    shape, w, _ = layer_of(name)
    slots = synth.shuffled_slots(shape.n_experts, table_seed) if table_seed >= 0 \
        else torch.arange(shape.n_experts, dtype=torch.int32)
    return B.DeviceLayer(shape, w, slots)


def workspace(nbytes: int) -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")


def layer_forward(dl: B.DeviceLayer, x: torch.Tensor, rep: int = 0):
    """Run moe_layer_forward on x [T,H] (cuda).  -> (y, y32, idx, w)."""
    shape = dl.shape
    T = x.shape[0]
    y = torch.empty((T, shape.hidden), dtype=synth.torch_dtype(shape.act), device="cuda")
    y32 = torch.empty((T, shape.hidden), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, shape.top_k), dtype=torch.int32, device="cuda")
    tw = torch.empty((T, shape.top_k), dtype=torch.float32, device="cuda")
    nb = B.moe_layer_workspace_bytes(dl.cfg, T)
    ws = workspace(nb)
    B.moe_layer_forward(dl.cfg, dl.struct(rep), x, T, y, y32, idx, tw, ws, nb)
    torch.cuda.synchronize()
    assert B.moe_get_device_error() == 0
    return y, y32, idx, tw


def near_tie_tokens(logits: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th oracle logits are within 1e-4*max(1,|l_k|)."""
    srt = np.sort(logits, axis=1)[:, ::-1]
    if srt.shape[1] <= k:
        return np.zeros(len(logits), bool)
    gap = srt[:, k - 1] - srt[:, k]
    return gap <= 1e-4 * np.maximum(1.0, np.abs(srt[:, k - 1]))

"""Seeded synthetic inputs for the routed int4 MoE layer.

This module only *produces inputs*: random draws, the min-max affine 4-bit
quantiser that turns dense draws into stored weights (the checkpoint
preparation step that MLX-style affine group quantisation performs before a
model ever runs; the layer itself only ever dequantises), the Zipf-shaped
router bias of the skewed workloads, and shuffled slot tables.  It evaluates
none of the layer's forward arithmetic (no router product, no top-k, no
dequantisation, no SwiGLU, no combine), so both the CPU oracle and the CUDA
path can consume its output without sharing any of the method's code.

Stored-weight format (MLX affine group quantisation, named on the Swiftlet
project page "Relation to TurboFieldfare" section as the scheme its kernels
implement):
  * a matrix W of shape [out, in] is cut into groups of G consecutive input
    columns; each group keeps a scale s and a bias b, and each weight keeps a
    4-bit code q in 0..15 with W ~= s*q + b;
  * codes are packed 8 per 32-bit word, the lowest column in the lowest
    nibble: q[o, c] lives in word [o, c // 8] at bits 4*(c % 8) .. 4*(c % 8)+3;
  * scale and bias are row-major [out, in // G] in the scale dtype.

Shapes follow the workloads the project pages describe (Qwen3-Next-80B-A3B:
10 of 512 experts; Qwen3.6-35B-A3B: 8 of 256 experts, the Swiftlet README "How it works"),
with hidden 2048, expert intermediate 512 and group 64.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

# --------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class MoEShape:
    name: str
    hidden: int           # H
    n_experts: int        # E
    top_k: int            # k
    inter: int            # I, routed expert intermediate
    shared_inter: int     # I_s, shared expert intermediate (0 = none)
    group: int            # G, quantisation group along the input dim
    act: str              # 'f32' | 'bf16'   activations x and y
    router: str           # 'f32' | 'bf16'   router and shared-gate weights
    qscale: str           # 'f32' | 'f16'    per-group scale and bias
    w_std: float          # std of the dense expert draws before quantisation
    router_std: float     # std of router / shared-gate draws
    tokens: int = 1       # T per step
    zipf_s: float = 0.0   # 0 = unbiased router
    layers: int = 1
    pool_slots: int = 0   # slots per layer in a bounded pool (0 = all resident)
    weight_seed: int = 0
    router_on_grid: bool = False  # router and shared gate drawn, then put on the affine 4-bit grid
    bits: int = 4                 # code width of the expert weights (MLX affine int4 or int8)


TINY = MoEShape("tiny", 64, 8, 2, 32, 32, 32, "f32", "f32", "f32", 0.05, 0.05,
                tokens=4, weight_seed=0, router_on_grid=True)
DEC_35B = MoEShape("35b-dec", 2048, 256, 8, 512, 512, 64, "bf16", "bf16", "f16",
                   0.02, 0.02, weight_seed=1)
DEC_80B = MoEShape("80b-dec", 2048, 512, 10, 512, 512, 64, "bf16", "bf16", "f16",
                   0.02, 0.02, weight_seed=2)
STACK_80B = MoEShape("80b-stack", 2048, 512, 10, 512, 512, 64, "bf16", "bf16", "f16",
                     0.02, 0.02, zipf_s=1.1, layers=48, pool_slots=128, weight_seed=3)
PREFILL_80B = MoEShape("80b-prefill", 2048, 512, 10, 512, 512, 64, "bf16", "bf16",
                       "f16", 0.02, 0.02, tokens=4096, zipf_s=1.1, weight_seed=2)

# The same layers with affine int8 codes (Swiftlet README "Relation to TurboFieldfare"
# names int4 and int8 group quantisation).
DEC_35B_INT8 = dataclasses.replace(DEC_35B, name="35b-dec-int8", bits=8)
DEC_80B_INT8 = dataclasses.replace(DEC_80B, name="80b-dec-int8", bits=8)

SHAPES = {s.name: s for s in (TINY, DEC_35B, DEC_80B, STACK_80B, PREFILL_80B, DEC_35B_INT8, DEC_80B_INT8)}

# Seeds of the per-step activations (decode: 1000 + step; stack: 5000 + step;
# prefill: 7; tiny: 0).
DECODE_X_SEED0 = 1000
STACK_X_SEED0 = 5000
PREFILL_X_SEED = 7
TINY_X_SEED = 0

# Logit scale of the Zipf router bias: bias_e = -ZIPF_BETA * s * ln(rank_e),
# rank_e a seeded permutation of 1..E.  A Gumbel-tail argument only gives the
# order of magnitude, so the constant was fitted on the oracle's routing of
# 2000 N(0,1) tokens through an 80B-shaped router (E=512, top-10): at 0.44 the
# log-log slope of selection frequency against rank is -1.1 (fit over experts
# picked by 0.25%..90% of tokens).  tests/test_synth_recipe.py re-checks it.
ZIPF_BETA = 0.44

_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def torch_dtype(tag: str) -> torch.dtype:
    return _DT[tag]


# --------------------------------------------------------------------------
# Random draws
# --------------------------------------------------------------------------


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, std, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def quantise_affine4(w: torch.Tensor, group: int, scale_dtype: torch.dtype, bits: int = 4):
    """Min-max affine quantiser with b-bit codes, b = bits (4 or 8; checkpoint
    preparation, not the forward).

    w: [..., out, in] float32.  Per group of `group` input columns, with
    m = 2^b - 1: scale = (max - min) / m, bias = min, code = clamp(
    round_half_even((w - bias) / scale), 0, m) (code 0 where the group is
    constant).  Returns (packed int32 [..., out, in*b/32] holding uint32 bit
    patterns, 32/b codes a word with the lowest column in the lowest bits,
    scale [..., out, in/G], bias [..., out, in/G]) in `scale_dtype`.
    """
    *lead, n_out, n_in = w.shape
    per = 32 // bits
    levels = (1 << bits) - 1
    assert n_in % group == 0 and n_in % per == 0
    g = w.reshape(*lead, n_out, n_in // group, group)
    lo = g.amin(dim=-1)
    hi = g.amax(dim=-1)
    scale = (hi - lo) / float(levels)
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    code = torch.round((g - lo.unsqueeze(-1)) / safe.unsqueeze(-1))
    code = torch.where(scale.unsqueeze(-1) > 0, code, torch.zeros_like(code))
    code = code.clamp_(0, levels).to(torch.int64).reshape(*lead, n_out, n_in // per, per)
    shifts = torch.arange(0, 32, bits, device=w.device, dtype=torch.int64)
    words = (code << shifts).sum(dim=-1)                       # 0 .. 2^32-1
    words = torch.where(words >= 2**31, words - 2**32, words)  # same bits as int32
    return words.to(torch.int32), scale.to(scale_dtype), lo.to(scale_dtype)


def _quantised_matrix_stack(n, n_out, n_in, shape: MoEShape, gen, device, chunk=64):
    """Draw n dense [n_out, n_in] matrices ~ N(0, w_std^2) and quantise them."""
    sd = torch_dtype(shape.qscale)
    qs, ss, bs = [], [], []
    for s0 in range(0, n, chunk):
        m = min(chunk, n - s0)
        w = _randn((m, n_out, n_in), shape.w_std, gen, device)
        q, s, b = quantise_affine4(w, shape.group, sd, shape.bits)
        qs.append(q), ss.append(s), bs.append(b)
        del w
    return torch.cat(qs), torch.cat(ss), torch.cat(bs)


def make_experts(shape: MoEShape, n: int, inter: int, seed: int, device="cpu") -> Dict[str, torch.Tensor]:
    """n experts in MLX form: q_gate/q_up [n, inter, H/8], q_down [n, H, inter/8],
    s_*/b_* the matching [.., in/G] scale and bias."""
    gen = _gen(seed, device)
    H = shape.hidden
    out = {}
    for name, (n_out, n_in) in (("gate", (inter, H)), ("up", (inter, H)), ("down", (H, inter))):
        q, s, b = _quantised_matrix_stack(n, n_out, n_in, shape, gen, device)
        out["q_" + name], out["s_" + name], out["b_" + name] = q, s, b
    return out


def zipf_router_bias(shape: MoEShape, seed: int, device="cpu") -> Optional[torch.Tensor]:
    """bias_e = -ZIPF_BETA * s * ln(rank_e) with rank a seeded permutation of 1..E."""
    if shape.zipf_s <= 0:
        return None
    gen = _gen(seed * 7919 + 17, "cpu")
    rank = torch.randperm(shape.n_experts, generator=gen).to(torch.float64) + 1.0
    bias = -ZIPF_BETA * shape.zipf_s * torch.log(rank)
    return bias.to(torch.float32).to(device)


def on_affine4_grid(w: torch.Tensor, group: int) -> torch.Tensor:
    """The dense fp32 values a checkpoint holds for w after min-max affine 4-bit
    quantisation with groups of `group` along the last dim (s * q + b for
    each weight).  A checkpoint-preparation step for weights the layer then
    reads as dense fp32 (the router and shared gate of the workload whose
    weights are all quantised); the layer's own int4 path never calls it."""
    *lead, n = w.shape
    g = w.reshape(*lead, n // group, group)
    lo = g.amin(dim=-1, keepdim=True)
    scale = (g.amax(dim=-1, keepdim=True) - lo) / 15.0
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    code = torch.where(scale > 0, torch.round((g - lo) / safe), torch.zeros_like(g)).clamp_(0, 15)
    return (code * scale + lo).reshape(w.shape)


def make_router(shape: MoEShape, seed: Optional[int] = None, device="cpu") -> Dict[str, torch.Tensor]:
    """The resident routing weights of a layer, exactly as make_layer draws
    them: w_router [E,H], w_shared_gate [H], router_bias [E] fp32 or None.
    With shape.router_on_grid the draws are first put on the affine 4-bit
    grid (group shape.group) and kept as dense values."""
    seed = shape.weight_seed if seed is None else seed
    gen = _gen(seed, device)
    rd = torch_dtype(shape.router)
    wr = _randn((shape.n_experts, shape.hidden), shape.router_std, gen, device)
    wsg = _randn((shape.hidden,), shape.router_std, gen, device)
    if shape.router_on_grid:
        wr = on_affine4_grid(wr, shape.group)
        wsg = on_affine4_grid(wsg, shape.group)
    return {
        "w_router": wr.to(rd),
        "w_shared_gate": wsg.to(rd),
        "router_bias": zipf_router_bias(shape, seed, device),
    }


def make_layer(shape: MoEShape, seed: Optional[int] = None, device="cpu") -> Dict[str, torch.Tensor]:
    """One layer's stored weights, all in the dtypes the shape names.

    Keys: w_router [E,H], w_shared_gate [H], router_bias [E] fp32 or None,
    routed experts (make_experts keys, leading dim E) and the shared expert
    under 'shared_' + key (leading dim 1).
    """
    seed = shape.weight_seed if seed is None else seed
    layer = make_router(shape, seed, device)
    layer["bits"] = shape.bits
    layer.update(make_experts(shape, shape.n_experts, shape.inter, seed * 31 + 1, device))
    if shape.shared_inter > 0:
        sh = make_experts(shape, 1, shape.shared_inter, seed * 31 + 2, device)
        layer.update({"shared_" + k: v for k, v in sh.items()})
    return layer


def make_x(shape: MoEShape, seed: int, tokens: Optional[int] = None, device="cpu") -> torch.Tensor:
    """Activations x ~ N(0, 1), [T, H] in the activation dtype (bf16: RNE from fp32)."""
    T = shape.tokens if tokens is None else tokens
    gen = _gen(seed, device)
    return torch.randn((T, shape.hidden), generator=gen, device=device,
                       dtype=torch.float32).to(torch_dtype(shape.act))


def decode_xs(shape: MoEShape, steps: int, seed0: int = DECODE_X_SEED0, device="cpu") -> torch.Tensor:
    """[steps, H]: step i is make_x(seed0 + i, T=1)."""
    return torch.cat([make_x(shape, seed0 + i, 1, device) for i in range(steps)])


def shuffled_slots(n_experts: int, seed: int, n_slots: Optional[int] = None) -> torch.Tensor:
    """An expert -> slot table with every expert resident at a seeded shuffled slot."""
    n_slots = n_experts if n_slots is None else n_slots
    gen = _gen(seed * 104729 + 5, "cpu")
    return torch.randperm(n_slots, generator=gen)[:n_experts].to(torch.int32)


def bytes_per_qmatrix(n_out: int, n_in: int, group: int, scale_bytes: int, bits: int = 4) -> int:
    """Stored bytes of one quantised matrix: packed codes + scale + bias."""
    return n_out * n_in * bits // 8 + 2 * n_out * (n_in // group) * scale_bytes


def expert_bytes(shape: MoEShape, inter: Optional[int] = None) -> int:
    I = shape.inter if inter is None else inter
    sb = 2 if shape.qscale == "f16" else 4
    return (2 * bytes_per_qmatrix(I, shape.hidden, shape.group, sb, shape.bits)
            + bytes_per_qmatrix(shape.hidden, I, shape.group, sb, shape.bits))


def active_expert_bytes(shape: MoEShape) -> int:
    """Bytes one decode token must stream per layer: k routed + the shared expert."""
    return shape.top_k * expert_bytes(shape) + (expert_bytes(shape, shape.shared_inter)
                                               if shape.shared_inter else 0)


assert expert_bytes(DEC_80B) == 1_769_472
assert active_expert_bytes(DEC_80B) == 19_464_192
assert expert_bytes(DEC_80B_INT8) == 3 * (512 * 2048 + 2 * 512 * 32 * 2)
assert math.isclose(ZIPF_BETA, 0.44)

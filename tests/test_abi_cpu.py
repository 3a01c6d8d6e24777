"""The C-ABI library on the CPU: it loads, exports every declared symbol,
validates arguments without touching a GPU, and its host-side pieces (blob
layout, repack, the slot policy under each eviction rule) agree with
independent versions."""
import ctypes
import random

import numpy as np
import pytest
import torch

from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth
from oracle.slot_policy import SlotPolicy


def test_library_exports_every_header_function():
    lib = B.lib()
    names = B.header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert B.moe_version().startswith("moe_int4")


def test_blob_layout_80b_and_tiny():
    l80 = B.moe_blob_layout_get(B.config_for(synth.DEC_80B), 512)
    assert (l80.q_gate, l80.q_up, l80.q_down) == (0, 524288, 1048576)
    assert l80.bytes == 1_769_472 == synth.expert_bytes(synth.DEC_80B)
    lt = B.moe_blob_layout_get(B.config_for(synth.TINY), 32)
    assert lt.bytes == 4608 == synth.expert_bytes(synth.TINY)
    for n, _ in B.moe_blob_layout._fields_:
        assert getattr(l80, n) % 256 == 0


@pytest.mark.parametrize("shape", [synth.TINY, synth.DEC_35B])
def test_pack_expert_matches_blob_packer(shape):
    cfg = B.config_for(shape)
    ex = synth.make_experts(shape, 3, shape.inter, seed=4)
    stride = B.moe_blob_layout_get(cfg, shape.inter).bytes
    ref = B.pack_blobs(cfg, shape.inter, ex, torch.tensor([2, 0, 1], dtype=torch.int32), 3, stride)
    for e, slot in ((0, 2), (1, 0), (2, 1)):
        dst = torch.full((stride,), 0xAB, dtype=torch.uint8)
        B.moe_pack_expert(cfg, shape.inter, B.expert_struct(ex, e), dst)
        assert torch.equal(dst, ref[slot])


@pytest.mark.parametrize("field,value,status", [
    ("hidden", 48, B.MOE_ERR_INVALID_ARG), ("n_experts", 2000, B.MOE_ERR_INVALID_ARG),
    ("top_k", 0, B.MOE_ERR_INVALID_ARG), ("top_k", 17, B.MOE_ERR_INVALID_ARG),
    ("group_size", 16, B.MOE_ERR_UNSUPPORTED), ("inter", 40, B.MOE_ERR_INVALID_ARG),
    ("act_dtype", B.MOE_F16, B.MOE_ERR_UNSUPPORTED), ("qscale_dtype", B.MOE_BF16, B.MOE_ERR_UNSUPPORTED)])
def test_bad_config_rejected_on_host(field, value, status):
    cfg = B.config_for(synth.DEC_80B)
    setattr(cfg, field, value)
    assert B.moe_layer_workspace_bytes(cfg, 1) == 0
    with pytest.raises(B.MoEError) as ei:
        B.moe_blob_layout_get(cfg, 512)
    assert ei.value.status == status


def test_null_arguments_rejected_without_gpu_work():
    cfg = B.config_for(synth.DEC_80B)
    with pytest.raises(B.MoEError) as ei:
        B.moe_route(cfg, None, 1, None, None, None, None, None, None, stream=0)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG and "NULL" in ei.value.message
    with pytest.raises(B.MoEError) as ei:
        B.moe_layer_forward(cfg, B.moe_layer(), 0x1000, 1, 0x2000, workspace=0x3000, ws_bytes=16, stream=0)
    assert ei.value.status == B.MOE_ERR_OOM
    # T == 0 is a no-op that succeeds
    B.moe_layer_forward(cfg, B.moe_layer(), None, 0, None, stream=0)


FAKE_DEV = 0x7F0000000000  # a 256-byte aligned address; lookups never dereference it


def _pool(n_layers, n_slots, shape=synth.DEC_80B):
    cfg = B.config_for(shape)
    stride = B.moe_blob_layout_get(cfg, shape.inter).bytes
    return B.slot_pool_create(cfg, n_layers, n_slots, FAKE_DEV, n_layers * n_slots * stride, FAKE_DEV,
                              stride, side_stream=0)


@pytest.mark.parametrize("rule, code", [("lfu_recency", B.MOE_POOL_LFU_RECENCY), ("lru", B.MOE_POOL_LRU),
                                        ("lfu", B.MOE_POOL_LFU)])
def test_slot_policy_matches_oracle_on_zipf_traces(rule, code):
    L, E, S, k = 3, 512, 32, 10
    p = _pool(L, S)
    if code != B.MOE_POOL_LFU_RECENCY:
        B.slot_pool_set_policy(p, code)
    ref = SlotPolicy(L, E, S, rule)
    rng = random.Random(0)
    w = [1.0 / (r + 1) ** 1.1 for r in range(E)]
    try:
        for step in range(300):
            for layer in range(L):
                need = []
                while len(need) < k:
                    e = rng.choices(range(E), weights=w)[0]
                    if e not in need:
                        need.append(e)
                slots, miss = B.slot_pool_lookup(p, layer, need)
                rslots, rfills = ref.lookup(layer, need)
                assert slots == rslots
                assert miss == [e for e, _ in rfills]
                assert B.slot_pool_table_host(p, layer, E) == ref.table[layer]
        st = B.slot_pool_stats(p)
        assert (st["hits"], st["misses"], st["evictions"]) == (ref.hits, ref.misses, ref.evictions)
        assert st["lookups"] == 300 * L and st["bytes_filled"] == 0
    finally:
        B.slot_pool_destroy(p)


def test_slot_pool_rejects_unknown_policy():
    p = _pool(1, 4)
    try:
        with pytest.raises(B.MoEError) as ei:
            B.slot_pool_set_policy(p, 3)
        assert ei.value.status == B.MOE_ERR_INVALID_ARG
    finally:
        B.slot_pool_destroy(p)


def test_slot_pool_exhaustion_and_fill_mismatch():
    p = _pool(1, 4)
    try:
        with pytest.raises(B.MoEError) as ei:
            B.slot_pool_lookup(p, 0, [0, 1, 2, 3, 4])
        assert ei.value.status == B.MOE_ERR_POOL_EXHAUSTED
        slots, miss = B.slot_pool_lookup(p, 0, [5, 6, 5])
        assert slots == [0, 1, 0] and miss == [5, 6]
        with pytest.raises(B.MoEError) as ei:
            B.slot_pool_fill(p, 0, [6, 5])
        assert ei.value.status == B.MOE_ERR_INVALID_ARG
        with pytest.raises(B.MoEError):
            B.slot_pool_lookup(p, 1, [0])
        with pytest.raises(B.MoEError):
            B.slot_pool_lookup(p, 0, [512])
    finally:
        B.slot_pool_destroy(p)


def test_strided_tensors_are_refused_before_any_call():
    import torch
    cfg = B.config_for(synth.DEC_80B)
    x = torch.zeros((4, 2 * synth.DEC_80B.hidden), dtype=torch.bfloat16)[:, ::2]
    with pytest.raises(ValueError):
        B.moe_layer_forward(cfg, B.moe_layer(), x, 4, None, stream=0)


def test_debug_wait_hook_validates_before_touching_a_device():
    with pytest.raises(B.MoEError) as ei:
        B.moe_debug_set_waits(0, 0)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoEError) as ei:
        B.moe_debug_set_waits(1_000_000, 5)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG


def test_noalloc_scratch_bound_stated_in_the_header():
    """The header states T <= 63 for the 35B- and 80B-shaped layers: the
    built-in 4 MiB scratch holds the single-token and generic paths' buffers,
    and from T = 64 on the grouped-GEMM buffers alone exceed it."""
    for shape in (synth.DEC_35B, synth.DEC_80B):
        cfg = B.config_for(shape)
        assert B.moe_layer_workspace_bytes(cfg, 63) <= 4 << 20 < B.moe_layer_workspace_bytes(cfg, 64)


def test_kernel_path_values_and_workspace_follow_the_path():
    """Paths 0, 1, 2 are accepted (per thread), others refused; the grouped-GEMM
    buffers join the workspace from T = 2 under path 2 only, and the
    single-token buffers up to T = 12 under path 0 (the token loop)."""
    cfg = B.config_for(synth.DEC_80B)
    try:
        for bad in (-1, 3):
            with pytest.raises(B.MoEError) as ei:
                B.moe_set_kernel_path(bad)
            assert ei.value.status == B.MOE_ERR_INVALID_ARG
        sizes, sizes16 = {}, {}
        for p in (0, 1, 2):
            B.moe_set_kernel_path(p)
            sizes[p] = B.moe_layer_workspace_bytes(cfg, 8)
            sizes16[p] = B.moe_layer_workspace_bytes(cfg, 16)
        assert sizes[1] < sizes[0] < sizes[2]                    # T = 8: token loop on path 0
        assert sizes16[0] == sizes16[1] < sizes16[2]             # T = 16: generic kernels on both
        B.moe_set_kernel_path(0)
        one = B.moe_layer_workspace_bytes(cfg, 1)
        B.moe_set_kernel_path(2)
        assert B.moe_layer_workspace_bytes(cfg, 1) == one      # T = 1 stays on the single-token kernels
    finally:
        B.moe_set_kernel_path(0)


def test_file_tier_pool_validates_on_the_host(tmp_path):
    """slot_pool_create_file checks path, alignment and file size before any
    device work; a valid one is created and destroyed without a GPU."""
    cfg = B.config_for(synth.DEC_80B)
    lay = B.moe_blob_layout_get(cfg, synth.DEC_80B.inter)
    fstride = (lay.bytes + 4095) // 4096 * 4096
    E = synth.DEC_80B.n_experts
    path = tmp_path / "one_layer.qpack"
    with open(path, "wb") as f:
        f.truncate(E * fstride)
    fake_pool = 1 << 20                                   # never dereferenced on the host
    with pytest.raises(B.MoEError) as ei:
        B.slot_pool_create_file(cfg, 1, 8, fake_pool, 8 * fstride, str(tmp_path / "missing"), 0, fstride)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
    with pytest.raises(B.MoEError):
        B.slot_pool_create_file(cfg, 1, 8, fake_pool, 8 * fstride, str(path), 0, fstride - 256)   # not 4 KiB
    with pytest.raises(B.MoEError):
        B.slot_pool_create_file(cfg, 2, 8, fake_pool, 16 * fstride, str(path), 0, fstride)      # file too small
    h = B.slot_pool_create_file(cfg, 1, 8, fake_pool, 8 * fstride, str(path), 0, fstride, readers=2)
    try:
        st = B.slot_pool_file_stats(h)
        assert st["bytes_read"] == 0 and st["read_ns"] == 0
    finally:
        B.slot_pool_destroy(h)

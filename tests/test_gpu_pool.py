"""The bounded expert pool on the GPU, through moe_pooled_layer_forward.

Pins "streaming never changes model semantics" (Swiftlet README repost,
"Correctness"): every layer output served from the pool is bit-identical to
the same layer served all-resident; the pool's slots hold byte-for-byte the
backing store's blobs; the device table, the host table and the independent
oracle policy agree exactly after every step; sampled outputs match the CPU
oracle on the GPU's own layer inputs.
"""
import dataclasses

import numpy as np
import pytest
import torch

from gpu_util import assert_close, near_tie_tokens
from int4_routed_expert_06_b300 import binding as B
from int4_routed_expert_06_b300 import synth
from bench import layer_input
from int4_routed_expert_06_b300.stack import PooledStack
from oracle import oracle as O
from oracle.slot_policy import SlotPolicy

pytestmark = pytest.mark.gpu

# An 80B-shaped layer with fewer experts so the stack test stays small; the
# router is Zipf-biased as in the 48-layer workload, and 25% of the experts fit.
SHAPE = dataclasses.replace(synth.STACK_80B, name="pool-test", n_experts=64, top_k=8, layers=3, pool_slots=16)


@pytest.fixture(scope="module")
def weights():
    return [synth.make_layer(SHAPE, seed=40 + l, device="cuda") for l in range(SHAPE.layers)]


@pytest.fixture(scope="module", params=["host", "device", "file"])
def stack(request, weights, tmp_path_factory):
    path = str(tmp_path_factory.mktemp("tier") / "layers.qpack") if request.param == "file" else None
    st = PooledStack(SHAPE, SHAPE.layers, SHAPE.pool_slots, lambda l: weights[l],
                     device_policy=request.param == "device", file_path=path)
    resident = [B.DeviceLayer(SHAPE, weights[l], torch.arange(SHAPE.n_experts, dtype=torch.int32))
                for l in range(SHAPE.layers)]
    yield st, weights, resident
    st.close()


def test_pool_stack_bit_identical_to_resident_and_policy_exact(stack):
    """Host policy, device policy, and host policy over the file tier: the
    same outputs, tables and counters."""
    st, weights, resident = stack
    L, E, k = SHAPE.layers, SHAPE.n_experts, SHAPE.top_k
    policy = SlotPolicy(L, E, SHAPE.pool_slots)
    oracles = [O.Layer(weights[l], SHAPE.group, k) for l in range(L)]
    nb = B.moe_layer_workspace_bytes(st.cfg, 1)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    checked = 0
    for step in range(24):
        h = synth.make_x(SHAPE, synth.STACK_X_SEED0 + step, 1, device="cuda")
        for l in range(L):
            x = layer_input(h)
            y = torch.empty((1, SHAPE.hidden), dtype=torch.bfloat16, device="cuda")
            y32 = torch.empty((1, SHAPE.hidden), device="cuda")
            idx = torch.empty((1, k), dtype=torch.int32, device="cuda")
            st.layer_forward(l, x, y, y32, idx)
            yr = torch.empty_like(y)
            yr32 = torch.empty_like(y32)
            idr = torch.empty_like(idx)
            B.moe_layer_forward(st.cfg, resident[l].struct(), x, 1, yr, yr32, idr, None, ws, nb)
            torch.cuda.synchronize()
            assert B.moe_get_device_error() == 0
            assert torch.equal(idx, idr) and torch.equal(y, yr) and torch.equal(y32, yr32), (step, l)
            # policy: the same lookup in the independent oracle policy
            _, fills = policy.lookup(l, idx[0].tolist())
            host = B.slot_pool_table_host(st.handle, l, E)
            assert host == policy.table[l], (step, l)
            assert st.table_device(l).tolist() == host
            for e, s in fills:                      # freshly filled slots hold the backing blob
                assert torch.equal(st.slot_bytes(l, s).cpu(), st.blob(l, e))
            if step % 8 == 3:                        # oracle on the GPU's own layer input
                ref = oracles[l].forward(x)
                if not near_tie_tokens(ref["logits"], k)[0]:
                    np.testing.assert_array_equal(idx.cpu().numpy(), ref["idx"])
                    assert_close(y32.cpu().numpy(), ref["y"], "bf16", f"step {step} layer {l}")
                    checked += 1
            h = (h.float() + y.float()).to(torch.bfloat16)    # residual stream into the next layer
    assert checked >= 6
    s = st.stats()
    assert (s["hits"], s["misses"], s["evictions"]) == (policy.hits, policy.misses, policy.evictions)
    assert s["bytes_filled"] == policy.misses * st.blob_bytes
    assert s["lookups"] == 24 * L
    assert (s["exposed_copy_ns"] > 0) == (not st.device_policy)
    if st.file_path:
        f = B.slot_pool_file_stats(st.handle)
        assert f["bytes_read"] >= policy.misses * st.blob_bytes and f["read_ns"] > 0
    assert policy.hits > 0 and policy.evictions > 0


def test_pool_exhaustion_is_an_error_not_a_fault(stack):
    st, weights, _ = stack
    small = dataclasses.replace(SHAPE, pool_slots=4)
    p = PooledStack(small, 1, 4, lambda l: weights[0])
    try:
        x = synth.make_x(SHAPE, 1, 1, device="cuda")
        y = torch.empty((1, SHAPE.hidden), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(B.MoEError) as ei:
            p.layer_forward(0, x, y)
        assert ei.value.status == B.MOE_ERR_POOL_EXHAUSTED
        torch.cuda.synchronize()
        assert B.moe_get_device_error() == 0
    finally:
        p.close()


def test_device_policy_stack_in_one_cuda_graph(weights):
    """Device mode has no host round trip: several tokens through every
    layer, captured once and replayed, stay bit-identical to the resident
    layers, and the pool counters advance by one lookup per layer-token."""
    L, E, k = SHAPE.layers, SHAPE.n_experts, SHAPE.top_k
    st = PooledStack(SHAPE, L, SHAPE.pool_slots, lambda l: weights[l], device_policy=True)
    resident = [B.DeviceLayer(SHAPE, weights[l], torch.arange(E, dtype=torch.int32)) for l in range(L)]
    try:
        n_tok = 6
        x0 = synth.decode_xs(SHAPE, n_tok, seed0=synth.STACK_X_SEED0 + 100, device="cuda")
        Y = torch.empty((n_tok, L, SHAPE.hidden), dtype=torch.bfloat16, device="cuda")
        stream = torch.cuda.Stream()
        st.workspace(1)

        def run():
            for j in range(n_tok):
                h = x0[j:j + 1]
                for l in range(L):
                    st.layer_forward(l, layer_input(h), Y[j, l:l + 1], stream=stream)
                    h = (h.float() + Y[j, l:l + 1].float()).to(torch.bfloat16)

        with torch.cuda.stream(stream):
            run()                                     # eager once: kernel attributes before capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run()
        s0 = st.stats()
        for _ in range(3):
            Y.zero_()
            with torch.cuda.stream(stream):
                g.replay()
            torch.cuda.synchronize()
            assert B.moe_get_device_error() == 0
            nb = B.moe_layer_workspace_bytes(st.cfg, 1)
            ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
            yr = torch.empty((1, SHAPE.hidden), dtype=torch.bfloat16, device="cuda")
            for j in range(n_tok):
                h = x0[j:j + 1]
                for l in range(L):
                    B.moe_layer_forward(st.cfg, resident[l].struct(), layer_input(h), 1, yr, None, None, None, ws, nb)
                    torch.cuda.synchronize()
                    assert torch.equal(yr, Y[j, l:l + 1]), (j, l)
                    h = (h.float() + yr.float()).to(torch.bfloat16)
        s1 = st.stats()
        assert s1["lookups"] - s0["lookups"] == 3 * n_tok * L
        assert s1["hits"] + s1["misses"] > s0["hits"] + s0["misses"]
    finally:
        st.close()


def test_device_step_bad_ids_recorded_not_faulted(weights):
    st = PooledStack(SHAPE, 1, 4, lambda l: weights[0], device_policy=True)
    try:
        bad = torch.tensor([3, SHAPE.n_experts + 5], dtype=torch.int32, device="cuda")
        B.slot_pool_step_device(st.handle, 0, bad, 2)
        torch.cuda.synchronize()
        assert B.moe_get_device_error() == B.MOE_ERR_DEVICE_FAULT
        many = torch.arange(8, dtype=torch.int32, device="cuda")   # 8 distinct, 4 slots
        B.slot_pool_step_device(st.handle, 0, many, 8)
        torch.cuda.synchronize()
        assert B.moe_get_device_error() == B.MOE_ERR_POOL_EXHAUSTED
        assert B.slot_pool_table_host(st.handle, 0, SHAPE.n_experts) == [-1] * SHAPE.n_experts
        ok = torch.tensor([5, 9, 5], dtype=torch.int32, device="cuda")
        B.slot_pool_step_device(st.handle, 0, ok, 3)
        torch.cuda.synchronize()
        assert B.moe_get_device_error() == 0
        t = B.slot_pool_table_host(st.handle, 0, SHAPE.n_experts)
        assert (t[5], t[9]) == (0, 1) and sum(v >= 0 for v in t) == 2
        with pytest.raises(B.MoEError):
            B.slot_pool_lookup(st.handle, 0, [1, 2])      # host lookups refused in device mode
    finally:
        st.close()


def test_device_policy_needs_a_device_readable_backing_store():
    cfg = B.config_for(SHAPE)
    lay = B.moe_blob_layout_get(cfg, SHAPE.inter)
    stride = (lay.bytes + 255) // 256 * 256
    pool = torch.empty(stride * 4, dtype=torch.uint8, device="cuda")
    pageable = torch.empty(stride * SHAPE.n_experts, dtype=torch.uint8)     # not pinned
    h = B.slot_pool_create(cfg, 1, 4, pool, pool.numel(), pageable, stride, None)
    try:
        with pytest.raises(B.MoEError) as ei:
            B.slot_pool_enable_device(h)
        assert ei.value.status == B.MOE_ERR_UNSUPPORTED
    finally:
        B.slot_pool_destroy(h)

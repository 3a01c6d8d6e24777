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
def stack():
    weights = [synth.make_layer(SHAPE, seed=40 + l, device="cuda") for l in range(SHAPE.layers)]
    st = PooledStack(SHAPE, SHAPE.layers, SHAPE.pool_slots, lambda l: weights[l])
    resident = [B.DeviceLayer(SHAPE, weights[l], torch.arange(SHAPE.n_experts, dtype=torch.int32))
                for l in range(SHAPE.layers)]
    yield st, weights, resident
    st.close()


def test_pool_stack_bit_identical_to_resident_and_policy_exact(stack):
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
                assert torch.equal(st.slot_bytes(l, s).cpu(), st.backing[l, e, :st.blob_bytes])
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
    assert s["exposed_copy_ns"] > 0 and s["lookups"] == 24 * L
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

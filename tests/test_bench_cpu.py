"""Host-side pieces of the measurement harness and the stack plumbing (no GPU)."""
import hashlib
import os

import pytest

import torch

import bench
from int4_routed_expert_06_b300 import synth
from bench import layer_input


def test_metric_names_follow_the_workload():
    assert bench.metric_of(synth.DEC_80B) == bench.METRIC
    assert "256e top-8" in bench.metric_of(synth.DEC_35B)
    assert "prefill" in bench.metric_of(synth.PREFILL_80B)
    assert "stack" in bench.metric_of(synth.STACK_80B)
    assert "prefill" in bench.workload_desc(synth.PREFILL_80B)
    assert "48-layer" in bench.workload_desc(synth.STACK_80B)


def test_prefill_flops_match_the_scope_table():
    # 4096 tokens of the 80B layer: routed 257.7 + shared 25.8 + router 8.6 GFLOP
    f = bench.prefill_flops(synth.PREFILL_80B, 4096)
    assert abs(f / 1e9 - 292.07) < 0.01
    # linear in T, and the router alone when no expert exists
    assert bench.prefill_flops(synth.PREFILL_80B, 8) * 512 == f


def test_recorded_traffic_needs_the_same_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "int4_routed_expert_06_b300" / "csrc"
    src.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (src / "kernels_token.cu").write_text("kernel v1\n")
    digest = hashlib.sha256(b"kernel v1\n").hexdigest()
    (tmp_path / "profiles" / "decode_layer_traffic.txt").write_text(
        "# comment\n" f"80b-dec {digest} 1 2 3\n" "35b-dec 00 1 2 4\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("80b-dec") == 3
    assert bench.recorded_traffic("35b-dec") is None        # recorded for another source
    assert bench.recorded_traffic("80b-prefill") is None    # not recorded
    (src / "kernels_token.cu").write_text("kernel v2\n")
    assert bench.recorded_traffic("80b-dec") is None        # source changed since the capture


@pytest.mark.parametrize("record,workload", [("decode_layer_traffic.txt", "80b-dec"),
                                             ("prefill_layer_traffic.txt", "80b-prefill")])
def test_committed_traffic_record_is_well_formed(record, workload):
    p = os.path.join(bench.ROOT, "profiles", record)
    rows = [l.split() for l in open(p) if l.strip() and not l.startswith("#")]
    assert rows and all(len(r) >= 5 for r in rows)
    assert any(r[0] == workload for r in rows)
    for r in rows:                      # workload, digest, per-kernel bytes ..., total
        digest, parts, total = r[1], [int(v) for v in r[2:-1]], int(r[-1])
        assert len(digest) == 64 and sum(parts) == total


def test_traffic_is_null_once_the_sources_change(monkeypatch):
    """The record names the kernel sources' digest: a different digest (a
    changed source) makes the bench report traffic as null."""
    monkeypatch.setattr(bench, "sources_digest", lambda names: "0" * 64)
    assert bench.recorded_traffic("80b-dec") is None
    assert bench.recorded_traffic("80b-prefill") is None


def test_stack_layer_input_is_unit_rms_and_scale_free():
    g = torch.Generator().manual_seed(3)
    h = (torch.randn(5, 2048, generator=g) * torch.tensor([0.1, 1.0, 7.0, 300.0, 1e4])[:, None]).to(torch.bfloat16)
    u = layer_input(h)
    assert u.dtype == torch.bfloat16 and u.shape == h.shape
    rms = u.float().pow(2).mean(-1).sqrt()
    assert torch.allclose(rms, torch.ones(5), atol=1e-2)
    # the same residual stream scaled by a power of two gives the same input
    # (up to one bf16 rounding step: eps is not scaled along)
    u4 = layer_input((h.float() * 4).to(torch.bfloat16))
    assert torch.allclose(u4.float(), u.float(), rtol=2 ** -7, atol=0)


def test_policy_study_runs_the_library_policy_and_uniform_routing_hits_the_pool_fraction(capsys):
    import argparse
    import json
    bench.run_policy_study(argparse.Namespace(steps=64))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    rows = line["table"]
    assert len(rows) == 4 * 3 * 3 and 0.0 < line["value"] < 1.0
    for r in rows:
        assert 0.0 <= r["hit_rate"] <= 1.0
        if r["zipf_s"] == 0.0:   # no skew: a pool holding a fraction f of the experts hits about f
            assert abs(r["hit_rate"] - r["pool_fraction"]) < 0.06, r


def test_routing_trace_uses_the_stack_router():
    shape = synth.STACK_80B
    t = bench.routing_trace(shape, 0, 8)
    assert t.shape == (8, shape.top_k) and t.dtype == torch.int32
    assert all(len(set(row.tolist())) == shape.top_k for row in t)
    assert int(t.min()) >= 0 and int(t.max()) < shape.n_experts

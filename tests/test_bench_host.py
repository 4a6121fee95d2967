"""Host-side logic of bench.py (no GPU): roofline byte counts and the lookup
of profiled DRAM traffic, which is valid only while the profiled kernel's own
source files are unchanged."""
import json
import os

import numpy as np

import bench
import workloads as W


def test_kernel_source_lists_exist():
    csrc = os.path.join(bench.ROOT, "fp8_routed_expert_gb300", "csrc")
    for kernel, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (kernel, f)
        assert len(bench.kernel_source_sha(kernel)) == 16


def test_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = tmp_path / "fp8_routed_expert_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES["decode_ffn"] + ("gemv.cu",):
        (csrc / f).write_text("// " + f)
    sha = bench.kernel_source_sha("decode_ffn")
    (prof / "traffic.json").write_text(json.dumps(
        {"decode_ffn/olmoe_decode_T8": {"dram_bytes_per_launch": 123.0, "source_sha": sha}}))
    assert bench.profiled_traffic("decode_ffn", "olmoe_decode_T8") == 123.0
    assert bench.profiled_traffic("decode_ffn", "olmoe_decode_T1") is None
    # a file outside the kernel's sources does not invalidate the record ...
    (csrc / "gemv.cu").write_text("// changed")
    assert bench.profiled_traffic("decode_ffn", "olmoe_decode_T8") == 123.0
    # ... one of its own sources does
    (csrc / "decode_mma.cu").write_text("// changed")
    assert bench.profiled_traffic("decode_ffn", "olmoe_decode_T8") is None


def test_committed_traffic_records_name_their_sources():
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for key, e in d.items():
        kernel, workload = key.split("/")
        assert kernel in bench.KERNEL_SOURCES, key
        assert tuple(e["sources"]) == bench.KERNEL_SOURCES[kernel], key
        W.parse_workload(workload)
        assert os.path.exists(os.path.join(bench.ROOT, "profiles", e["profile"])), key


def test_selected_bytes_count_active_experts_only():
    fam = W.family("olmoe_decode")
    counts = np.zeros(fam.n_experts, dtype=np.int32)
    counts[[1, 5, 9]] = [3, 1, 4]
    sb = bench.selected_bytes(fam, counts)
    assert sb["n_active"] == 3
    H, I = fam.hidden, fam.inter
    per13 = 2 * I * H + 4 * (2 * I // 128) * (H // 128)
    per2 = H * I + 4 * (H // 128) * (I // 128)
    assert sb["w13"] == 3 * per13 and sb["w2"] == 3 * per2
    assert sb["w13"] + sb["w2"] == 3 * fam.expert_bytes


class _FakeLayer:
    """Stands in for MoELayer's timing API: two kernel steps were timed."""

    def __init__(self, fail=False):
        self.mask, self.fail, self.steps = None, fail, 0

    def set_timing(self, kernels=()):
        if self.fail and kernels:
            raise RuntimeError("timing unavailable")
        self.mask = kernels

    def kernel_time(self, name):
        return {"gate_up": (2.0, 4), "combine": (0.04, 4)}.get(name, (0.0, 0))


def test_kernel_breakdown(monkeypatch):
    import torch
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a: None)
    layer = _FakeLayer()
    calls = []
    out = bench.kernel_breakdown(layer, lambda: calls.append("step"), lambda: calls.append("flush"),
                                 None, 4)
    assert out == {"gate_up": 500.0, "combine": 10.0}
    assert calls == ["flush", "step"] * 4
    assert layer.mask == ()  # timing switched off again
    bad = _FakeLayer(fail=True)
    out = bench.kernel_breakdown(bad, lambda: None, lambda: None, None, 2)
    assert "unavailable" in out and bad.mask == ()

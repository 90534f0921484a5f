"""Host-side pieces of the benchmark (no GPU): the algorithmic flop count of the
chunked prefill and the rule that a DRAM traffic record is reported only for
the kernel source it was measured on."""
import hashlib
import json
import os

import bench
from continuous_linear_attention_gb300 import synth


def test_prefill_flops_per_token_at_full_dims():
    """Hv (2 C (3 d_k + 2 d_v) + 6 d_k d_v) with C = 64, d = 128, Hv = 32 is
    5,767,168 flop per token of a sequence longer than one token."""
    wl = synth.make_workload("f", synth.FULL_DIMS, [130, 1, 64], [0, 1, 0], 8, 3)
    assert bench.prefill_flops(wl) == 5_767_168 * (130 + 64)


def test_prefill_flops_counts_no_decode_tokens():
    wl = synth.make_workload("d", synth.FULL_DIMS, [1, 1, 1], [1, 1, 1], 8, 4)
    assert bench.prefill_flops(wl) == 0.0


def _tree(tmp_path, source: bytes, recorded: bytes):
    csrc = tmp_path / "continuous_linear_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_bytes(source)
    (tmp_path / "profiles").mkdir()
    rec = {"k.cu": {"dram_bytes_per_launch": 123,
                    "source_sha256_16": hashlib.sha256(recorded).hexdigest()[:16]}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))


def test_traffic_record_matches_its_source(tmp_path, monkeypatch):
    _tree(tmp_path, b"kernel v1", b"kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("k.cu") == 123


def test_traffic_record_dropped_once_the_kernel_changed(tmp_path, monkeypatch):
    _tree(tmp_path, b"kernel v2", b"kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("k.cu") is None
    assert bench.traffic_record("missing.cu") is None


def test_committed_traffic_record_names_a_kernel_source():
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for name, entry in rec.items():
        assert os.path.exists(os.path.join(bench.ROOT, "continuous_linear_attention_gb300", "csrc", name))
        assert entry["dram_bytes_per_launch"] > 0 and len(entry["source_sha256_16"]) == 16

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


def test_decode_bytes_at_full_dims():
    """State 2 x 32 x 128 x 128 x 4, conv state 2 x 3 x 8192 x 2, x 8192 x 2,
    a and b 2 x 32 x 2, out 32 x 128 x 2 per request; weights 8192 x 4 x 2 +
    2 x 32 x 4 once: 4,317,312 per request + 65,792."""
    wl = synth.make_workload("d", synth.FULL_DIMS, [1] * 4, [1] * 4, 8, 4)
    assert bench.decode_bytes(wl) == 4 * 4_317_312 + 65_792


def test_decode_bytes_with_channel_gates():
    """The gate input grows to 32 x 128 bf16 per request and dt_bias to
    32 x 128 fp32 once."""
    wl = synth.make_workload("d", synth.FULL_DIMS, [1] * 4, [1] * 4, 8, 4, channel_gate=True)
    assert bench.decode_bytes(wl) == 4 * (4_317_312 + 32 * 127 * 2) + 65_792 + 32 * 127 * 4


def test_mamba2_decode_bytes():
    """H = 128, P = 64, N = 128, G = 8, K = 4, bf16 (C = 10240): state
    2 x 4 MiB, conv state 2 x 3 x 10240 x 2, xbc 10240 x 2, dt 128 x 2,
    y 128 x 64 x 2 per request; weights 10240 x 4 x 2 + 3 x 128 x 4."""
    dims = synth.SsdDims(H=128, P=64, N=128, G=8, K=4, act="bf16")
    wl = synth.make_ssd_workload("m", dims, [1] * 2, [1] * 2, 4, 0)
    per = 2 * 4_194_304 + 2 * 3 * 10240 * 2 + 10240 * 2 + 256 + 16384
    assert bench.ssd_decode_bytes(wl) == 2 * per + 10240 * 8 + 1536


def test_cpu_baseline_reports_cores_and_one_thread_rate():
    """The oracle leg runs on the host alone (no GPU): a bounded sample, the
    threads it used, and the one-thread rate."""
    wl = synth.make_workload("d", synth.TINY_DIMS, [1] * 8, [1] * 8, 16, 2)
    cb = bench.cpu_baseline(wl, budget_s=0.2, one_thread_s=0.1)
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["cores"] >= 1
    assert cb["value"] > 0 and cb["value_1_thread"] > 0


def test_mamba2_prefill_cost():
    """Two sequences of 130 and 1 tokens (only the 130-token one counts):
    bytes 130 x (10240 + 128 + 8192) x 2; flops per token and head
    2*128*64 + 2*128*64 + 2*64*128 + 2*128*128/16 = 51,200."""
    dims = synth.SsdDims(H=128, P=64, N=128, G=8, K=4, act="bf16")
    wl = synth.make_ssd_workload("m", dims, [130, 1], [0, 1], 4, 0)
    nbytes, flops = bench.ssd_prefill_cost(wl)
    assert nbytes == 130 * (10240 + 128 + 8192) * 2
    assert flops == 130 * 128 * 51_200

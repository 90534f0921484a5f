"""Helpers of the GPU parity tests: run a workload through the C ABI and
compare every output with the fp64 oracle."""
import json
import os

import numpy as np
import torch

import oracle
from continuous_linear_attention_gb300 import harness

# Tolerances (relative L2 over a whole tensor): fp32 activations everywhere
# 1e-5; bf16 activations with fp32 states 5e-3.
TOL = {"f32": 1e-5, "bf16": 5e-3}


def log_errs(errs):
    """Append the measured errors of the running test to the file named by
    GDN_PARITY_LOG (one JSON object per line), when that variable is set."""
    path = os.environ.get("GDN_PARITY_LOG")
    if path:
        name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
        with open(path, "a") as f:
            f.write(json.dumps({"test": name, **{k: float(v) for k, v in errs.items()}}) + "\n")


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def written_blocks(wl, skip):
    cu = wl.cu_seqlens.tolist()
    return [int(wl.block_idx[s]) for s in range(wl.N)
            if not skip[s] and int(wl.block_idx[s]) >= 0 and cu[s + 1] > cu[s]]


def mask_written(mem, run, blocks):
    m = mem.clone()
    for blk in blocks:
        o = run.block_offset(blk)
        m[o + run.conv_off: o + run.conv_off + run.conv_bytes] = 0
        m[o + run.rec_off: o + run.rec_off + run.rec_bytes] = 0
    return m


def check_against_oracle(wl, run=None, seqs=None, tol=None, expect_flags=0, ref=None,
                         prefill="auto"):
    """Run ``wl`` on the GPU (unless ``run`` has already been run) and compare
    with the oracle: out rows, new conv states (bit-exact: they are copies of
    inputs), recurrent states (rel-L2), untouched pool bytes and out rows of
    skipped sequences (byte-equal).  ``seqs`` restricts the out/state
    comparison to some sequences (the oracle still runs on the whole
    workload unless ``ref`` is given).  Returns a dict of the errors."""
    d = wl.dims
    tol = TOL[d.act] if tol is None else tol
    if run is None:
        run = harness.DeviceRun(wl, prefill=prefill)
        before = run.mem.clone()
        run.run()
        torch.cuda.synchronize()
    else:
        before = None
    flags = run.pool.error_flags()
    assert flags == expect_flags, f"error flags {flags:#x} != {expect_flags:#x}"
    if ref is None:
        ref = oracle.forward(wl)
    skip = ref["skip"]
    cu = wl.cu_seqlens.tolist()
    seqs = range(wl.N) if seqs is None else seqs
    out = run.out.float().cpu().numpy().astype(np.float64)
    errs = {"out": 0.0, "rec": 0.0}
    ref_blocks = [int(v) for v in wl.ref_blocks]
    rows = []
    for s in seqs:
        if skip[s] or int(wl.block_idx[s]) < 0 or cu[s + 1] == cu[s]:
            continue
        rows.extend(range(cu[s], cu[s + 1]))
    if rows:
        errs["out"] = rel_l2(out[rows], ref["out"][rows])
    blocks = [int(wl.block_idx[s]) for s in seqs
              if not skip[s] and int(wl.block_idx[s]) >= 0 and cu[s + 1] > cu[s]]
    if blocks:
        raw = run.block_bytes(blocks).numpy().reshape(-1)
        conv, rec = oracle.read_pool_states(raw, 0, range(len(blocks)), d, len(blocks), 1,
                                            block_align=run.block_align)
        idx = [ref_blocks.index(b) for b in blocks]
        np.testing.assert_array_equal(conv, ref["conv_state"][idx])
        errs["rec"] = rel_l2(rec, ref["rec_state"][idx])
    # rows of skipped / padding sequences untouched
    for s in range(wl.N):
        if skip[s] or int(wl.block_idx[s]) < 0:
            assert (out[cu[s]:cu[s + 1]] == harness.OUT_SENTINEL).all(), f"seq {s} out written"
    if before is not None:
        after = run.mem
        wb = written_blocks(wl, skip)
        assert torch.equal(mask_written(before, run, wb), mask_written(after, run, wb)), \
            "bytes outside the written sub-states changed"
    log_errs(errs)
    assert errs["out"] <= tol and errs["rec"] <= tol, errs
    return errs


def check_ssd_against_oracle(wl, tol=None, expect_flags=0):
    """Run a Mamba2 workload through gdn_ssd_varlen_forward and compare with
    the oracle: y rows (rel-L2), new conv states (bit-exact), SSM states
    (rel-L2), y rows of skipped sequences and every pool byte outside the
    written sub-states (byte-equal)."""
    d = wl.dims
    tol = TOL[d.act] if tol is None else tol
    run = harness.SsdDeviceRun(wl)
    before = run.mem.clone()
    run.run()
    torch.cuda.synchronize()
    flags = run.pool.error_flags()
    assert flags == expect_flags, f"error flags {flags:#x} != {expect_flags:#x}"
    ref = oracle.ssd_forward(wl)
    skip = ref["skip"]
    cu = wl.cu_seqlens.tolist()
    y = run.y.float().cpu().numpy().astype(np.float64)
    active = [s for s in range(wl.N)
              if not skip[s] and int(wl.block_idx[s]) >= 0 and cu[s + 1] > cu[s]]
    rows = [r for s in active for r in range(cu[s], cu[s + 1])]
    errs = {"y": rel_l2(y[rows], ref["y"][rows]) if rows else 0.0, "ssm": 0.0}
    blocks = [int(wl.block_idx[s]) for s in active]
    ref_blocks = [int(v) for v in wl.ref_blocks]
    if blocks:
        raw = run.block_bytes(blocks).numpy().reshape(-1)
        conv, ssm = oracle.read_ssd_pool_states(raw, 0, range(len(blocks)), d, len(blocks), 1)
        idx = [ref_blocks.index(b) for b in blocks]
        np.testing.assert_array_equal(conv, ref["conv_state"][idx])
        errs["ssm"] = rel_l2(ssm, ref["ssm_state"][idx])
    for s in range(wl.N):
        if s not in active:
            assert (y[cu[s]:cu[s + 1]] == harness.OUT_SENTINEL).all(), f"seq {s} y written"
    masked_before, masked_after = before.clone(), run.mem.clone()
    for blk in blocks:
        o = run.block_offset(blk)
        for m in (masked_before, masked_after):
            m[o: o + run.conv_bytes] = 0
            m[o + run.ssm_off: o + run.ssm_off + run.ssm_bytes] = 0
    assert torch.equal(masked_before, masked_after), "bytes outside the written sub-states changed"
    run.close()
    log_errs(errs)
    assert errs["y"] <= tol and errs["ssm"] <= tol, errs
    return errs

"""GPU parity over several calls on one pool: every request's tokens arrive
spread over consecutive calls in segments of mixed kinds — nothing, a single
token (the decode kernel), a short or a multi-chunk prefill (the chunked
path), with or without a past — so that one call mixes decodes and prefills
and a request's state passes from one kernel path to another between calls.
The concatenated outputs and the final states must equal the oracle's single
pass over the whole sequences (scalar gate, and one case with the
per-channel decay).  This exercises the per-call reset of the
persistent kernels' counters, the late decode behind the recurrence, and the
continuation of conv and recurrent states across paths."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from continuous_linear_attention_gb300 import harness, synth

from gpu_check import TOL, log_errs, rel_l2

pytestmark = pytest.mark.gpu


def _calls(whole, bounds):
    """Split every sequence s of ``whole`` at the offsets bounds[s] (0 = b_0 <=
    b_1 <= ... <= b_K = length) into K consecutive calls on the same blocks; a
    request whose earlier segments were all empty keeps its own has_past."""
    cu = whole.cu_seqlens.tolist()
    n_calls = len(bounds[0]) - 1
    calls = []
    for k in range(n_calls):
        rows, lens, hp = [], [], []
        for s in range(whole.N):
            lo, hi = cu[s] + bounds[s][k], cu[s] + bounds[s][k + 1]
            rows.extend(range(lo, hi))
            lens.append(hi - lo)
            hp.append(int(whole.has_past[s]) if bounds[s][k] == 0 else 1)
        idx = torch.tensor(rows, dtype=torch.int64)
        ncu = np.zeros(whole.N + 1, dtype=np.int32)
        ncu[1:] = np.cumsum(lens)
        calls.append(dataclasses.replace(
            whole, name=f"{whole.name}_call{k}", x=whole.x[idx].contiguous(),
            a=whole.a[idx].contiguous(), b=whole.b[idx].contiguous(),
            cu_seqlens=torch.from_numpy(ncu), has_past=torch.tensor(hp, dtype=torch.uint8)))
    return calls


@pytest.mark.parametrize("seed,channel_gate", [(81, False), (82, False), (83, True)])
def test_requests_spread_over_calls_of_mixed_kinds_match_one_pass(seed, channel_gate):
    rng = np.random.default_rng(seed)
    n_req, n_calls = 20, 5
    # per request and call: 0 tokens, 1 token, a short prefill or one over several chunks
    kinds = rng.choice(4, size=(n_req, n_calls), p=[0.15, 0.45, 0.25, 0.15])
    seg = np.where(kinds == 0, 0, np.where(kinds == 1, 1, np.where(
        kinds == 2, rng.integers(2, 64, size=kinds.shape), rng.integers(64, 300, size=kinds.shape))))
    seg[seg.sum(axis=1) == 0, 0] = 1  # every request has a token somewhere
    lens = seg.sum(axis=1).tolist()
    has_past = rng.integers(0, 2, size=n_req).tolist()
    dims = synth.Dims(Hk=4, Hv=8, dk=128, dv=128, K=4, act=synth.BF16)
    whole = synth.make_workload("multicall", dims, lens, has_past, 64, seed,
                                channel_gate=channel_gate)
    bounds = [[0] + np.cumsum(seg[s]).tolist() for s in range(n_req)]
    calls = _calls(whole, bounds)
    ref = oracle.forward(whole)

    run = harness.DeviceRun(calls[0])
    outs = []
    for k, wl in enumerate(calls):
        if k:
            run.set_inputs(wl)
        run.run()
        torch.cuda.synchronize()
        assert run.pool.error_flags() == 0, k
        outs.append(run.out.double().cpu().numpy())
    # each request's rows, call after call, in the whole batch's order
    got = np.concatenate([
        np.concatenate([outs[k][int(calls[k].cu_seqlens[s]):int(calls[k].cu_seqlens[s + 1])]
                        for k in range(n_calls)])
        for s in range(n_req)])
    err_out = rel_l2(got, ref["out"])
    ref_blocks = [int(v) for v in whole.ref_blocks]
    err_rec = 0.0
    for s in range(n_req):
        blk = int(whole.block_idx[s])
        r = ref_blocks.index(blk)
        err_rec = max(err_rec, rel_l2(run.rec_view(blk).cpu().numpy(), ref["rec_state"][r]))
        np.testing.assert_array_equal(run.conv_view(blk).float().cpu().numpy().astype(np.float64),
                                      ref["conv_state"][r])
    log_errs({"out": err_out, "rec": err_rec})
    assert err_out <= TOL["bf16"] and err_rec <= TOL["bf16"], (err_out, err_rec)


def _ssd_calls(whole, bounds):
    """The Mamba2 workload's sequences split at ``bounds`` into consecutive
    calls, as ``_calls`` does for the gated delta rule."""
    cu = whole.cu_seqlens.tolist()
    n_calls = len(bounds[0]) - 1
    calls = []
    for k in range(n_calls):
        rows, lens, hp = [], [], []
        for s in range(whole.N):
            lo, hi = cu[s] + bounds[s][k], cu[s] + bounds[s][k + 1]
            rows.extend(range(lo, hi))
            lens.append(hi - lo)
            hp.append(int(whole.has_past[s]) if bounds[s][k] == 0 else 1)
        idx = torch.tensor(rows, dtype=torch.int64)
        ncu = np.zeros(whole.N + 1, dtype=np.int32)
        ncu[1:] = np.cumsum(lens)
        calls.append(dataclasses.replace(
            whole, name=f"{whole.name}_call{k}", xbc=whole.xbc[idx].contiguous(),
            dt=whole.dt[idx].contiguous(), cu_seqlens=torch.from_numpy(ncu),
            has_past=torch.tensor(hp, dtype=torch.uint8)))
    return calls


def test_mamba2_requests_spread_over_calls_match_one_pass():
    """The same over the Mamba2 scan: requests' tokens over five calls in
    segments of mixed kinds (decode kernel, chunked scan), y and the final
    conv and SSM states against the oracle's single pass."""
    rng = np.random.default_rng(91)
    n_req, n_calls = 12, 5
    kinds = rng.choice(4, size=(n_req, n_calls), p=[0.15, 0.45, 0.25, 0.15])
    seg = np.where(kinds == 0, 0, np.where(kinds == 1, 1, np.where(
        kinds == 2, rng.integers(2, 64, size=kinds.shape), rng.integers(64, 300, size=kinds.shape))))
    seg[seg.sum(axis=1) == 0, 0] = 1
    lens = seg.sum(axis=1).tolist()
    has_past = rng.integers(0, 2, size=n_req).tolist()
    dims = synth.SsdDims(H=16, P=64, N=128, G=2, K=4, act="bf16")
    whole = synth.make_ssd_workload("ssd_multicall", dims, lens, has_past, 32, 91)
    bounds = [[0] + np.cumsum(seg[s]).tolist() for s in range(n_req)]
    calls = _ssd_calls(whole, bounds)
    ref = oracle.ssd_forward(whole)

    run = harness.SsdDeviceRun(calls[0])
    ys = []
    for k, wl in enumerate(calls):
        if k:
            run.set_inputs(wl)
        run.run()
        torch.cuda.synchronize()
        assert run.pool.error_flags() == 0, k
        ys.append(run.y.float().cpu().numpy().astype(np.float64))
    got = np.concatenate([
        np.concatenate([ys[k][int(calls[k].cu_seqlens[s]):int(calls[k].cu_seqlens[s + 1])]
                        for k in range(n_calls)])
        for s in range(n_req)])
    err_y = rel_l2(got, ref["y"])
    blocks = [int(whole.block_idx[s]) for s in range(n_req)]
    raw = run.block_bytes(blocks).numpy().reshape(-1)
    conv, ssm = oracle.read_ssd_pool_states(raw, 0, range(len(blocks)), dims, len(blocks), 1)
    ref_blocks = [int(v) for v in whole.ref_blocks]
    idx = [ref_blocks.index(b) for b in blocks]
    np.testing.assert_array_equal(conv, ref["conv_state"][idx])
    err_ssm = rel_l2(ssm, ref["ssm_state"][idx])
    log_errs({"y": err_y, "ssm": err_ssm})
    assert err_y <= TOL["bf16"] and err_ssm <= TOL["bf16"], (err_y, err_ssm)
    run.close()


def test_one_captured_graph_replayed_over_changing_batches():
    """A serving loop's pattern: one CUDA graph captured for a fixed token
    count and request count (after the prefill scratch is reserved), then
    replayed over batches of different compositions written into its input
    buffers — decodes, prefills, a padding request (block -1) taking the
    leftover rows.  Every replay equals an eager call on the same inputs from
    the same pool state, bit for bit (outputs of the real requests and the
    whole pool)."""
    T, n_req = 512, 8
    rng = np.random.default_rng(7)
    dims = synth.FULL_DIMS
    # requests on blocks 1..7 (with past states), the padding request last
    base = synth.make_workload("graph_serve", dims, [1] * 7 + [T - 7], [1] * 7 + [0], 16, 71,
                               block_idx=list(range(1, n_req)) + [-1])
    steps = []
    for k in range(4):
        kinds = rng.choice(3, size=n_req - 1, p=[0.2, 0.5, 0.3])
        lens = [0 if c == 0 else (1 if c == 1 else int(rng.integers(2, 150))) for c in kinds]
        if sum(lens) > T:
            lens = [1] * (n_req - 1)
        lens.append(T - sum(lens))  # the padding request takes the leftover rows
        cu = np.zeros(n_req + 1, dtype=np.int32)
        cu[1:] = np.cumsum(lens)
        g = torch.Generator().manual_seed(100 + k)
        steps.append(dataclasses.replace(
            base, name=f"graph_serve_{k}",
            x=torch.randn(T, dims.C, generator=g).to(base.x.dtype),
            a=torch.randn(T, dims.Hv, generator=g).to(base.a.dtype),
            b=torch.randn(T, dims.Hv, generator=g).to(base.b.dtype),
            cu_seqlens=torch.from_numpy(cu),
            block_idx=torch.tensor(list(range(1, n_req)) + [-1], dtype=torch.int32),
            has_past=torch.tensor([1] * (n_req - 1) + [0], dtype=torch.uint8)))
    eager = harness.DeviceRun(steps[0])
    graphed = harness.DeviceRun(steps[0])
    snapshot = graphed.mem.clone()
    graphed.pool.reserve(T)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graphed.run(stream=s)  # warm-up outside the capture
    torch.cuda.synchronize()
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg, stream=s):
        graphed.run(stream=s)
    graphed.mem.copy_(snapshot)
    torch.cuda.synchronize()
    for k, st in enumerate(steps):
        if k:
            eager.set_inputs(st)
        eager.run()
        for dst, src in ((graphed.x, st.x), (graphed.a, st.a), (graphed.b, st.b),
                         (graphed.cu, st.cu_seqlens), (graphed.idx, st.block_idx),
                         (graphed.has_past, st.has_past)):
            dst.copy_(src)
        cg.replay()
        torch.cuda.synchronize()
        assert eager.pool.error_flags() == 0 and graphed.pool.error_flags() == 0
        real = int(st.cu_seqlens[n_req - 1])  # rows of the real requests
        assert torch.equal(eager.out[:real], graphed.out[:real]), k
        assert torch.equal(eager.mem, graphed.mem), k

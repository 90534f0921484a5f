"""GPU parity of the C-ABI forward against the fp64 oracle, and the invariants
of continuous batching checked on the GPU path (all calls go through the C
ABI via the ctypes binding)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from continuous_linear_attention_gb300 import binding, harness, synth

from gpu_check import TOL, check_against_oracle, rel_l2

pytestmark = pytest.mark.gpu


def _slice(wl, seqs):
    cu = wl.cu_seqlens.tolist()
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]).astype(np.int64)
    ncu = np.zeros(len(seqs) + 1, dtype=np.int32)
    ncu[1:] = np.cumsum([cu[s + 1] - cu[s] for s in seqs])
    idx = torch.from_numpy(rows)
    return dataclasses.replace(wl, x=wl.x[idx], a=wl.a[idx], b=wl.b[idx],
                               cu_seqlens=torch.from_numpy(ncu),
                               block_idx=wl.block_idx[list(seqs)],
                               has_past=wl.has_past[list(seqs)])


# ----------------------------------------------------------------------------
# The standard cases.

def test_tiny_packed_fp32():
    errs = check_against_oracle(synth.tiny_packed(0))
    assert errs["out"] <= 1e-5


def test_tiny_packed_fp32_slow_decay():
    check_against_oracle(synth.tiny_packed(0, slow_decay=True))


@pytest.mark.parametrize("seed", [0, 5])
def test_tiny_dims_bf16_mixed(seed):
    dims = dataclasses.replace(synth.TINY_DIMS, act="bf16")
    wl = synth.make_workload("tiny_bf16", dims, [70, 1, 1, 129, 3], [1, 1, 0, 0, 1], 16, seed)
    check_against_oracle(wl)


@pytest.mark.parametrize("d", [64])
def test_head_dim_64(d):
    dims = synth.Dims(Hk=2, Hv=4, dk=d, dv=d, K=4, act="bf16")
    wl = synth.make_workload("d64", dims, [65, 1, 130], [0, 1, 1], 8, 3)
    check_against_oracle(wl)


def test_equal_heads_ratio_one():
    dims = synth.Dims(Hk=3, Hv=3, dk=32, dv=32, K=3, act="f32")
    wl = synth.make_workload("r1", dims, [9, 1, 66], [1, 1, 0], 8, 4)
    check_against_oracle(wl)


def test_decode_batch_full():
    """256 decode requests, bf16 activations, fp32 states, 512-block pool."""
    check_against_oracle(synth.decode_batch())


@pytest.mark.parametrize("prefill", ["auto", "fused"])
def test_prefill_full_dims_ragged(prefill):
    """Full head dims, lengths spanning several 64-token chunks and ragged tails;
    both the split (conv kernel + TMA-fed chunked kernel) and the fused form."""
    wl = synth.make_workload("prefill_small", synth.FULL_DIMS, [130, 64, 257, 2, 1, 65],
                             [0, 1, 0, 1, 1, 1], 16, 7)
    check_against_oracle(wl, prefill=prefill)


def test_prefill_full_size_sampled():
    """The ~16k-token packed prefill at full size; the oracle checks the two
    shortest sequences (a packed batch equals each sequence alone)."""
    wl = synth.packed_prefill()
    lens = wl.seqlens()
    pick = sorted(range(wl.N), key=lambda s: lens[s])[:2]
    ref = oracle.forward(_slice(wl, pick))
    run = harness.DeviceRun(wl)
    before = run.mem.clone()
    run.run()
    torch.cuda.synchronize()
    # map the sliced oracle back onto the full batch's rows
    cu = wl.cu_seqlens.tolist()
    full_out = np.full((wl.T, wl.dims.Hv, wl.dims.dv), np.nan)
    off = 0
    for s in pick:
        L = cu[s + 1] - cu[s]
        full_out[cu[s]:cu[s + 1]] = ref["out"][off:off + L]
        off += L
    ref_full = dict(ref, out=full_out, skip=[False] * wl.N)
    check_against_oracle(wl, run=run, seqs=pick, ref=ref_full)
    # nothing outside the written sub-states moved
    from gpu_check import mask_written, written_blocks
    wb = written_blocks(wl, [False] * wl.N)
    assert torch.equal(mask_written(before, run, wb), mask_written(run.mem, run, wb))


@pytest.mark.parametrize("prefill", ["auto", "fused"])
def test_mixed_batch_full(prefill):
    """64 decodes + 6 prefill continuations with past, 8192 tokens, 1024 blocks."""
    check_against_oracle(synth.mixed_batch(), prefill=prefill)


@pytest.mark.parametrize("prefill", ["split", "fused"])
def test_many_decodes_behind_the_prefill(prefill):
    """400 decodes among three prefill continuations: the decode kernel runs
    behind the prefill's recurrence (its CTAs start while the recurrence's last
    chains run) and takes its units from a counter, many more than its CTAs."""
    rng = np.random.default_rng(61)
    lens = [1] * 400 + [200, 130, 65]
    rng.shuffle(lens)
    wl = synth.make_workload("many_dec", synth.FULL_DIMS, lens, [1] * len(lens), len(lens) + 9, 61)
    check_against_oracle(wl, prefill=prefill)


def test_long_context_split_equals_single_pass():
    """4 x 32768 tokens then a 4096-token continuation from the saved states
    equals one 36864-token pass; the oracle checks a prefix of sequence 0."""
    first, cont, whole = synth.long_context()
    # split run
    run = harness.DeviceRun(first)
    run.run()
    run.set_inputs(cont)
    run.run()
    torch.cuda.synchronize()
    assert run.pool.error_flags() == 0
    out_cont = run.out.float().cpu()
    # first part's out again (set_inputs replaced it): rerun on a fresh pool
    run1 = harness.DeviceRun(first)
    run1.run()
    torch.cuda.synchronize()
    out_first = run1.out.float().cpu()
    # single pass
    single = harness.DeviceRun(whole)
    single.run()
    torch.cuda.synchronize()
    n, L1, L2 = 4, 32768, 4096
    d = whole.dims
    out_single = single.out.float().cpu().view(n, L1 + L2, d.Hv, d.dv)
    split = torch.cat([out_first.view(n, L1, d.Hv, d.dv), out_cont.view(n, L2, d.Hv, d.dv)], 1)
    assert rel_l2(split.numpy(), out_single.numpy()) <= TOL["bf16"]
    for s in range(n):
        blk = int(whole.block_idx[s])
        assert rel_l2(run.rec_view(blk).cpu().numpy(), single.rec_view(blk).cpu().numpy()) <= 1e-3
        assert torch.equal(run.conv_view(blk).cpu(), single.conv_view(blk).cpu())
    # oracle on the first 2048 tokens of sequence 0
    pre = dataclasses.replace(_slice(first, [0]), x=first.x[:2048], a=first.a[:2048],
                              b=first.b[:2048], cu_seqlens=torch.tensor([0, 2048], dtype=torch.int32))
    ref = oracle.forward(pre)
    assert rel_l2(out_first[:2048].numpy(), ref["out"]) <= TOL["bf16"]


# ----------------------------------------------------------------------------
# Edge cases of the batch description.

def test_padding_and_empty_sequences():
    dims = synth.TINY_DIMS
    wl = synth.make_workload("pad", dims, [4, 0, 1, 0, 7, 2], [1, 0, 1, 1, 0, 0], 12, 8,
                             block_idx=[3, 5, -1, -1, 6, 9])
    check_against_oracle(wl)


def test_zero_tokens():
    dims = synth.TINY_DIMS
    wl = synth.make_workload("empty", dims, [0, 0], [0, 0], 4, 9, block_idx=[1, 2])
    check_against_oracle(wl)


@pytest.mark.parametrize("blocks,flag", [
    ([2, 2, 5], binding.FLAG_DUPLICATE),
    ([0, 3, 5], binding.FLAG_TRASH_WRITE),
    ([2, 3, 99], binding.FLAG_BLOCK_RANGE),
])
def test_bad_block_indices_are_flagged_and_skipped(blocks, flag):
    dims = synth.TINY_DIMS
    wl = synth.make_workload("bad", dims, [3, 1, 4], [1, 1, 0], 8, 10, block_idx=blocks)
    check_against_oracle(wl, expect_flags=flag)


def test_decode_hint_skips_and_flags_longer_sequences():
    """max_seqlen_hint = 1 launches only the decode path; a longer sequence is
    skipped (block and out rows untouched) and flagged, the others match."""
    wl = synth.make_workload("hint", synth.FULL_DIMS, [1, 5, 1, 1], [1, 1, 0, 1], 8, 15)
    run = harness.DeviceRun(wl)
    before = run.mem.clone()
    run.run(max_seqlen_hint=1)
    torch.cuda.synchronize()
    assert run.pool.error_flags() == binding.FLAG_HINT
    blk = int(wl.block_idx[1])
    assert torch.equal(run.rec_view(blk), before[run.block_offset(blk) + run.rec_off:][
        :run.rec_bytes].view(torch.float32).view(run.rec_view(blk).shape))
    assert (run.out[1:6].float() == harness.OUT_SENTINEL).all()
    keep = [0, 2, 3]
    ref = oracle.forward(_slice(wl, keep))
    cu = wl.cu_seqlens.tolist()
    got = torch.cat([run.out[cu[s]:cu[s + 1]] for s in keep]).double().cpu().numpy()
    assert rel_l2(got, ref["out"]) <= TOL["bf16"]


def test_bad_cu_seqlens_skip_everything():
    dims = synth.TINY_DIMS
    wl = synth.make_workload("badcu", dims, [3, 1, 4], [1, 1, 0], 8, 11)
    wl = dataclasses.replace(wl, cu_seqlens=torch.tensor([0, 3, 2, 8], dtype=torch.int32))
    run = harness.DeviceRun(wl)
    before = run.mem.clone()
    run.run()
    torch.cuda.synchronize()
    assert run.pool.error_flags() == binding.FLAG_SEQLENS
    assert torch.equal(before, run.mem)
    assert (run.out.float() == harness.OUT_SENTINEL).all()


def test_host_argument_errors_launch_nothing():
    wl = synth.tiny_packed(0)
    run = harness.DeviceRun(wl)
    with pytest.raises(binding.GdnError):
        binding.varlen_forward(run.pool, 1, run.x, run.a, run.b, run.cu, run.idx, run.has_past,
                               run.conv_w, run.A_log, run.dt_bias, run.out, wl.T, wl.N)
    with pytest.raises(binding.GdnError):
        binding.varlen_forward(run.pool, 0, run.x.data_ptr() + 4, run.a, run.b, run.cu, run.idx,
                               run.has_past, run.conv_w, run.A_log, run.dt_bias, run.out, wl.T,
                               wl.N)
    torch.cuda.synchronize()
    assert (run.out.float() == harness.OUT_SENTINEL).all()


# ----------------------------------------------------------------------------
# Invariants on the GPU path.

def test_packed_equals_each_alone_gpu():
    dims = dataclasses.replace(synth.FULL_DIMS)
    wl = synth.make_workload("pack", dims, [70, 1, 129, 1, 3], [0, 1, 1, 1, 0], 8, 12)
    run = harness.DeviceRun(wl)
    run.run()
    torch.cuda.synchronize()
    cu = wl.cu_seqlens.tolist()
    for s in range(wl.N):
        one = harness.DeviceRun(_slice(wl, [s]))
        one.run()
        torch.cuda.synchronize()
        assert torch.equal(one.out, run.out[cu[s]:cu[s + 1]])
        blk = int(wl.block_idx[s])
        assert torch.equal(one.rec_view(blk), run.rec_view(blk))
        assert torch.equal(one.conv_view(blk), run.conv_view(blk))


@pytest.mark.parametrize("prefill", ["auto", "fused"])
def test_beta_zero_only_decays_gpu(prefill):
    wl = synth.make_workload("beta0", synth.FULL_DIMS, [5, 1, 66], [1, 1, 1], 8, 13)
    wl = dataclasses.replace(wl, b=torch.full_like(wl.b, -1000.0))
    check_against_oracle(wl, prefill=prefill)


def test_split_and_fused_prefill_agree():
    """The two prefill forms give the same outputs and states within rounding."""
    wl = synth.make_workload("forms", synth.FULL_DIMS, [300, 1, 77, 2], [1, 1, 0, 0], 8, 18)
    a = harness.DeviceRun(wl)
    b = harness.DeviceRun(wl, prefill="fused")
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert rel_l2(a.out.float().cpu().numpy(), b.out.float().cpu().numpy()) <= 2e-3
    for blk in [int(v) for v in wl.block_idx]:
        assert rel_l2(a.rec_view(blk).cpu().numpy(), b.rec_view(blk).cpu().numpy()) <= 2e-3
        assert torch.equal(a.conv_view(blk), b.conv_view(blk))


def test_graph_capture_replays_the_same_result():
    wl = synth.make_workload("graph", synth.FULL_DIMS, [1, 1, 200, 1, 67], [1, 1, 1, 1, 0], 16, 14)
    eager = harness.DeviceRun(wl)
    eager.run()
    torch.cuda.synchronize()
    graphed = harness.DeviceRun(wl)
    snapshot = graphed.mem.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graphed.run(stream=s)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graphed.mem.copy_(snapshot)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.run()
    graphed.mem.copy_(snapshot)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(graphed.out, eager.out)
    assert torch.equal(graphed.mem, eager.mem)


def test_inputs_rewritten_after_stream_order_are_safe():
    """Batch buffers reused across calls on one stream (the warmup race: a
    forward must see the inputs as they were when it was enqueued)."""
    wls = [synth.make_workload(f"r{i}", synth.TINY_DIMS, [3, 1, 6], [0, 1, 0], 8, 20 + i,
                               block_idx=[1, 2, 3]) for i in range(3)]
    run = harness.DeviceRun(wls[0])
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for wl in wls:
            run.x.copy_(wl.x.to(run.device, non_blocking=False))
            run.run(stream=s)
            outs.append(run.out.clone())
    torch.cuda.synchronize()
    ref = harness.DeviceRun(wls[0])
    for i, wl in enumerate(wls):
        ref.x.copy_(wl.x.cuda())
        ref.run()
        torch.cuda.synchronize()
        assert torch.equal(outs[i], ref.out)


# ----------------------------------------------------------------------------
# Pool lifecycle: several layers, aligned blocks, fork.

def test_second_layer_of_a_multi_layer_pool_with_aligned_blocks():
    """Layer 1 of a two-layer pool with 64 KiB block alignment: results equal the
    oracle and layer 0 stays byte-identical."""
    wl = synth.make_workload("layer1", synth.FULL_DIMS, [1, 70, 1], [1, 0, 1], 8, 16)
    run = harness.DeviceRun(wl, num_layers=2, layer=1, block_align=1 << 16)
    assert run.stride % (1 << 16) == 0
    page0 = run.mem[:run.page].clone()
    before = run.mem.clone()
    run.run()
    torch.cuda.synchronize()
    assert torch.equal(run.mem[:run.page], page0)
    check_against_oracle(wl, run=run)
    from gpu_check import mask_written, written_blocks
    wb = written_blocks(wl, [False] * wl.N)
    assert torch.equal(mask_written(before, run, wb), mask_written(run.mem, run, wb))


def test_fork_copies_a_block_and_both_continue_identically():
    """A block copied on fork (gdn_state_pool_copy_block) continues exactly like
    the original."""
    wl = synth.make_workload("fork", synth.FULL_DIMS, [9], [1], 8, 17, block_idx=[3])
    run = harness.DeviceRun(wl)
    run.pool.copy_block(0, 3, 5)
    torch.cuda.synchronize()
    assert torch.equal(run.mem[run.block_offset(5):run.block_offset(5) + run.stride],
                       run.mem[run.block_offset(3):run.block_offset(3) + run.stride])
    two = dataclasses.replace(
        wl, x=torch.cat([wl.x, wl.x]), a=torch.cat([wl.a, wl.a]), b=torch.cat([wl.b, wl.b]),
        cu_seqlens=torch.tensor([0, 9, 18], dtype=torch.int32),
        block_idx=torch.tensor([3, 5], dtype=torch.int32),
        has_past=torch.tensor([1, 1], dtype=torch.uint8))
    run.set_inputs(two)
    run.run()
    torch.cuda.synchronize()
    assert torch.equal(run.out[:9], run.out[9:])
    assert torch.equal(run.rec_view(3), run.rec_view(5))
    assert torch.equal(run.conv_view(3), run.conv_view(5))
    with pytest.raises(binding.GdnError):
        run.pool.copy_block(0, 3, 0)  # the trash block is never written


def test_captured_prefill_after_reserve_takes_the_split_path():
    """A prefill captured in a CUDA graph after gdn_state_pool_reserve runs the
    split kernels (the query says so) and replays to the eager result; on a
    pool with no scratch, capture never allocates and reports the fused
    kernel; an eager call grows the scratch stream-ordered and takes the split
    path."""
    wl = synth.make_workload("cap", synth.FULL_DIMS, [300, 1, 129, 70], [1, 1, 0, 1], 16, 22)
    eager = harness.DeviceRun(wl)
    eager.run()
    torch.cuda.synchronize()
    assert eager.pool.last_prefill_path() == binding.PREFILL_SPLIT
    for reserve, path in [(wl.T, binding.PREFILL_SPLIT), (None, binding.PREFILL_FUSED)]:
        run = harness.DeviceRun(wl)
        snapshot = run.mem.clone()
        if reserve is not None:
            run.pool.reserve(reserve)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            run.run(stream=s)
        assert run.pool.last_prefill_path() == path
        run.mem.copy_(snapshot)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert run.pool.error_flags() == 0
        if path == binding.PREFILL_SPLIT:
            assert torch.equal(run.out, eager.out)
            assert torch.equal(run.mem, eager.mem)
        else:
            assert rel_l2(run.out.float().cpu().numpy(), eager.out.float().cpu().numpy()) <= 2e-3
    decode = synth.make_workload("dec_only", synth.FULL_DIMS, [1, 1], [1, 1], 8, 23)
    d = harness.DeviceRun(decode)
    d.run(max_seqlen_hint=1)
    assert d.pool.last_prefill_path() == binding.PREFILL_NONE

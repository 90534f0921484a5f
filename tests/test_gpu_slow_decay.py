"""Full-size GPU parity in the regime where the carried state matters.

With the default gates (A_log = log U(1, 16), a ~ N(0, 1)) the log decay
averages about -7 per token, so a state forgets within a few tokens: the past
state and the state handed from one 64-token chunk to the next contribute
almost nothing to the outputs.  With slow decay (A_log = log U(0.01, 0.1),
dt_bias = -8) the decay is about e^{-1e-5} per token, so those hand-overs
dominate, and an indexing or precision slip confined to them (the past state
read, the chunk-to-chunk state in the tensor-core prefill, the continuation
of a split sequence) shows in the outputs and the final states.

"Continuous batching for linear attention layers": the recurrence continues
from each request's recurrent state through cu_seqlens, and a request's block
is overwritten in place by every forward, so a sequence split across calls
continues exactly from what the previous call left.  Every case here is
compared element by element with the fp64 oracle at the bf16 bar (rel-L2
<= 5e-3 over outputs and written states; new conv states bit-exact).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from continuous_linear_attention_gb300 import harness, synth

from gpu_check import TOL, check_against_oracle, log_errs, rel_l2

pytestmark = pytest.mark.gpu


def _states(run, wl, ref):
    """rel-L2 of the recurrent states of every sequence's block against the
    oracle's, and bit-exact conv states."""
    ref_blocks = [int(v) for v in wl.ref_blocks]
    err = 0.0
    for s in range(wl.N):
        blk = int(wl.block_idx[s])
        r = ref_blocks.index(blk)
        err = max(err, rel_l2(run.rec_view(blk).cpu().numpy(), ref["rec_state"][r]))
        conv = run.conv_view(blk).float().cpu().numpy().astype(np.float64)
        np.testing.assert_array_equal(conv, ref["conv_state"][r])
    return err


def test_decode_batch_slow_decay():
    """The 256-request decode batch: the output is dominated by S_{t-1} q."""
    errs = check_against_oracle(synth.decode_batch(slow_decay=True))
    assert errs["out"] <= TOL["bf16"]


def test_mixed_batch_slow_decay():
    """64 decodes + 6 continuations with past, every state carried."""
    check_against_oracle(synth.mixed_batch(slow_decay=True))


@pytest.mark.parametrize("slow", [False, True])
def test_prefill_16k_every_sequence(slow):
    """The ~16k-token packed prefill at full size, every sequence against the
    oracle (outputs, final states, conv states, untouched pool bytes)."""
    check_against_oracle(synth.packed_prefill(slow_decay=slow))


@pytest.mark.parametrize("slow", [False, True])
def test_long_prefill_with_past_split_at_chunk_edges(slow):
    """Two sequences with a past state, 4160 and 4225 tokens, each split once
    (after 2047 = 32 * 64 - 1 and 2113 = 33 * 64 + 1 tokens) and continued in
    a second call: the outputs of both calls and the states after each call
    equal the oracle's one pass."""
    whole = synth.make_workload("split_edges", synth.FULL_DIMS, [4160, 4225], [1, 1], 8, 21,
                                slow_decay=slow)
    first, cont = synth.row_split(whole, [2047, 2113])
    ref_whole = oracle.forward(whole)
    ref_first = oracle.forward(first)
    run = harness.DeviceRun(first)
    before = run.mem.clone()
    run.run()
    torch.cuda.synchronize()
    assert run.pool.error_flags() == 0
    out1 = run.out.double().cpu().numpy()
    assert rel_l2(out1, ref_first["out"]) <= TOL["bf16"]
    assert _states(run, first, ref_first) <= TOL["bf16"]
    run.set_inputs(cont)
    run.run()
    torch.cuda.synchronize()
    assert run.pool.error_flags() == 0
    out2 = run.out.double().cpu().numpy()
    cu, c1, c2 = (w.cu_seqlens.tolist() for w in (whole, first, cont))
    got = np.concatenate([np.concatenate([out1[c1[s]:c1[s + 1]], out2[c2[s]:c2[s + 1]]])
                          for s in range(whole.N)])
    err_out, err_rec = rel_l2(got, ref_whole["out"]), _states(run, whole, ref_whole)
    log_errs({"out": err_out, "rec": err_rec})
    assert err_out <= TOL["bf16"] and err_rec <= TOL["bf16"], (err_out, err_rec)
    from gpu_check import mask_written
    blocks = [int(v) for v in whole.block_idx]
    assert torch.equal(mask_written(before, run, blocks), mask_written(run.mem, run, blocks))


@pytest.mark.parametrize("slow", [False, True])
def test_long_context_full_sequence_against_oracle(slow):
    """The long-context case: 4 x 32768 tokens with no past, then 4096 more
    each from the saved states.  Sequence 0's 36864 outputs and its final
    recurrent and conv states are compared with the oracle's single pass."""
    first, cont, whole = synth.long_context(slow_decay=slow)
    run = harness.DeviceRun(first)
    run.run()
    torch.cuda.synchronize()
    out1 = run.out[:32768].double().cpu().numpy()
    run.set_inputs(cont)
    run.run()
    torch.cuda.synchronize()
    assert run.pool.error_flags() == 0
    out2 = run.out[:4096].double().cpu().numpy()
    seq0 = dataclasses.replace(
        whole, x=whole.x[:36864], a=whole.a[:36864], b=whole.b[:36864],
        cu_seqlens=torch.tensor([0, 36864], dtype=torch.int32),
        block_idx=whole.block_idx[:1], has_past=whole.has_past[:1])
    ref = oracle.forward(seq0)
    got = np.concatenate([out1, out2])
    err_out = rel_l2(got, ref["out"])
    blk = int(whole.block_idx[0])
    r = [int(v) for v in seq0.ref_blocks].index(blk)
    err_rec = rel_l2(run.rec_view(blk).cpu().numpy(), ref["rec_state"][r])
    np.testing.assert_array_equal(run.conv_view(blk).float().cpu().numpy().astype(np.float64),
                                  ref["conv_state"][r])
    log_errs({"out": err_out, "rec": err_rec})
    assert err_out <= TOL["bf16"] and err_rec <= TOL["bf16"], (err_out, err_rec)

"""Parity of the per-channel-decay (KDA) rule's split prefill (conv pass,
chunk products with running decay products, tensor-core recurrence) against
the fp64 oracle: chunk edges, many short sequences, long chains with slowly
decaying states (where the state hand-over between chunks carries the
result), values outside the fp16 range of the chunk operands (recomputed
token-serially), and agreement with the token-serial kernel."""
import dataclasses

import numpy as np
import pytest
import torch

from continuous_linear_attention_gb300 import binding, harness, synth
from gpu_check import TOL, check_against_oracle, rel_l2

pytestmark = pytest.mark.gpu


def _kda(name, lens, past, blocks, seed, slow=False, **kw):
    return synth.make_workload(name, synth.FULL_DIMS, lens, past, blocks, seed, slow_decay=slow,
                               channel_gate=True, **kw)


def _run_split(wl):
    run = harness.DeviceRun(wl)
    run.run()
    torch.cuda.synchronize()
    assert run.pool.last_prefill_path() == binding.PREFILL_SPLIT
    return run


@pytest.mark.parametrize("slow", [False, True])
@pytest.mark.parametrize("past", [0, 1])
def test_chunk_boundaries(past, slow):
    """Lengths on and next to multiples of the 64-token chunk, with a decode
    token among them."""
    lens = [64, 128, 63, 65, 127, 129, 192, 2, 1]
    wl = _kda("kda_chunk_edges", lens, [past] * len(lens), 17, 40 + past, slow)
    check_against_oracle(wl, run=_run_split(wl))


def test_many_short_sequences():
    """120 sequences of 2..9 tokens among a few around the chunk size, with
    and without past."""
    rng = np.random.default_rng(41)
    lens = [int(v) for v in rng.integers(2, 10, size=120)] + [63, 64, 65, 1, 1]
    rng.shuffle(lens)
    past = [int(v) for v in rng.integers(0, 2, size=len(lens))]
    wl = _kda("kda_many_short", lens, past, len(lens) + 9, 42)
    check_against_oracle(wl, run=_run_split(wl))


@pytest.mark.parametrize("slow", [False, True])
def test_long_chains(slow):
    """Chains of 12 and 19 chunks from a past state: with slow decay the
    state carried across every chunk boundary dominates outputs and final
    states."""
    wl = _kda("kda_long", [1200, 760, 1], [1, 0, 1], 8, 43, slow)
    check_against_oracle(wl, run=_run_split(wl))


def test_many_decodes_behind_the_prefill():
    """300 decodes among two prefill continuations: the per-channel-decay
    decode kernel runs behind the split prefill's recurrence and takes its
    units from a counter."""
    rng = np.random.default_rng(47)
    lens = [1] * 300 + [150, 70]
    rng.shuffle(lens)
    wl = _kda("kda_many_dec", lens, [1] * len(lens), len(lens) + 9, 47)
    check_against_oracle(wl, run=_run_split(wl))


def test_split_and_token_serial_agree():
    """The split prefill and the token-serial kernel (a pool without
    prefill scratch) on the same batch."""
    wl = _kda("kda_both", [300, 1, 129, 64], [1, 1, 0, 1], 8, 44, True)
    a = _run_split(wl)
    b = harness.DeviceRun(wl, prefill="fused")  # no scratch: token-serial
    b.run()
    torch.cuda.synchronize()
    assert b.pool.last_prefill_path() == binding.PREFILL_SERIAL
    err = rel_l2(a.out.float().cpu().numpy(), b.out.float().cpu().numpy())
    assert err <= TOL["bf16"], err
    assert a.pool.error_flags() == 0 and b.pool.error_flags() == 0
    a.close()
    b.close()


def test_past_state_outside_fp16_is_recomputed():
    """A past recurrent state of magnitude 1e5 cannot enter the fp16 state
    operand: that sequence's v-heads are recomputed token-serially in the same
    call, and every output and state matches the oracle with no flag."""
    wl = _kda("kda_big_state", [130, 70], [1, 0], 8, 45)
    rec = wl.rec_state.clone()
    rec[[int(b) for b in wl.ref_blocks].index(int(wl.block_idx[0]))] = 1.0e5
    wl = dataclasses.replace(wl, rec_state=rec)
    check_against_oracle(wl, run=_run_split(wl))


def test_inputs_outside_fp16_are_recomputed():
    """The v channels of one k-head scaled to about 1e5 in one sequence: both
    v-heads of that k-head are recomputed token-serially (the conv pass marks
    them), everything else keeps the tensor-core result."""
    wl = _kda("kda_big_v", [200, 1, 90], [1, 1, 0], 8, 46)
    d = wl.dims
    x = wl.x.float().clone()
    c0 = 2 * d.Hk * d.dk + 6 * d.dv  # v of heads 6 and 7 (k-head 3)
    x[0:200, c0:c0 + 2 * d.dv] *= 1.0e5
    wl = dataclasses.replace(wl, x=x.to(torch.bfloat16))
    check_against_oracle(wl, run=_run_split(wl))



def test_captured_prefill_replays_the_eager_result():
    """A per-channel-decay prefill captured in a CUDA graph on a pool whose
    scratch an eager call has grown runs the split kernels (no allocation, no
    host sync inside the capture) and replays to the eager result bit for bit;
    on a pool without prefill scratch the capture takes the token-serial
    kernel."""
    wl = _kda("kda_cap", [300, 1, 129, 70], [1, 1, 0, 1], 16, 49, True)
    eager = _run_split(wl)
    run = harness.DeviceRun(wl)
    snapshot = run.mem.clone()
    run.run()  # eager: grows the scratch to this call's size
    torch.cuda.synchronize()
    run.mem.copy_(snapshot)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run.run(stream=s)
    assert run.pool.last_prefill_path() == binding.PREFILL_SPLIT
    run.mem.copy_(snapshot)
    run.out.fill_(harness.OUT_SENTINEL)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert run.pool.error_flags() == 0
    assert torch.equal(run.out, eager.out)
    assert torch.equal(run.mem, eager.mem)
    # a pool without prefill scratch: the capture runs the token-serial kernel
    small = harness.DeviceRun(wl, prefill="fused")
    snap2 = small.mem.clone()
    s2 = torch.cuda.Stream()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s2):
        small.run(stream=s2)
    assert small.pool.last_prefill_path() == binding.PREFILL_SERIAL
    small.mem.copy_(snap2)
    torch.cuda.synchronize()
    g2.replay()
    torch.cuda.synchronize()
    assert small.pool.error_flags() == 0
    err = rel_l2(small.out.float().cpu().numpy(), eager.out.float().cpu().numpy())
    assert err <= TOL["bf16"], err
    run.close()
    small.close()
    eager.close()


def test_scalar_and_per_channel_forwards_share_a_pool():
    """Scalar-gate and per-channel-decay prefills alternate on one pool (and
    so on one prefill scratch, laid out differently by each); each matches its
    own oracle."""
    kda = _kda("kda_share", [200, 90, 1], [0, 1, 1], 8, 50)
    run = _run_split(kda)
    check_against_oracle(kda, run=run)
    scal = synth.make_workload("scalar_share", synth.FULL_DIMS, [150, 64, 1], [0, 0, 1], 8, 51)
    # the same pool: the scalar forward on its own inputs and states
    blocks = [int(b) for b in scal.ref_blocks]
    run.upload_states(blocks, scal.conv_state, scal.rec_state)
    run.wl = scal
    run.set_inputs(scal)
    run.conv_w, run.A_log, run.dt_bias = (scal.conv_w.to(run.device), scal.A_log.to(run.device),
                                          scal.dt_bias.to(run.device))
    run.run()
    torch.cuda.synchronize()
    assert run.pool.last_prefill_path() == binding.PREFILL_SPLIT
    check_against_oracle(scal, run=run)
    run.close()

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


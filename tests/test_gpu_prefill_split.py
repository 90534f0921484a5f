"""Parity of the split prefill path (chunk-parallel kernel, recurrence
kernel) on the shapes that stress its bookkeeping: many short sequences,
sequences ending on and next to chunk boundaries, values outside the fp16
range of the chunk products (recomputed token-serially), and a pool whose
prefill scratch an earlier call left non-finite."""
import dataclasses

import numpy as np
import pytest
import torch

from continuous_linear_attention_gb300 import binding, harness, synth
from gpu_check import check_against_oracle

pytestmark = pytest.mark.gpu


def test_many_short_sequences():
    """150 sequences of 2..9 tokens among a few around the chunk size, with
    and without past: hundreds of partial chunks and short chains."""
    rng = np.random.default_rng(11)
    lens = [int(v) for v in rng.integers(2, 10, size=150)] + [63, 64, 65, 127, 128, 129, 1, 1]
    rng.shuffle(lens)
    past = [int(v) for v in rng.integers(0, 2, size=len(lens))]
    wl = synth.make_workload("many_short", synth.FULL_DIMS, lens, past, len(lens) + 9, 21)
    check_against_oracle(wl)


@pytest.mark.parametrize("past", [0, 1])
def test_chunk_boundaries(past):
    """Lengths on and next to multiples of the 64-token chunk."""
    lens = [64, 128, 63, 65, 127, 129, 192, 2]
    wl = synth.make_workload("chunk_edges", synth.FULL_DIMS, lens, [past] * len(lens), 17, 22)
    check_against_oracle(wl)


def test_after_an_overflowing_call_the_next_call_is_exact():
    """A first call whose every value is scaled by 1e5 overflows the fp16
    operands of all chunk products: every v-head is recomputed token-serially
    and matches the oracle, with no flag.  It leaves non-finite values in the
    pool's prefill scratch; a second call on the same pool (a decode token
    and a padding sequence among partial chunks) must not read any of them."""
    big = synth.make_workload("overflow", synth.FULL_DIMS, [300, 200], [0, 0], 8, 23)
    big = dataclasses.replace(big, x=(big.x.float() * 1e5).to(big.x.dtype))
    run = harness.DeviceRun(big)
    run.run()
    torch.cuda.synchronize()
    check_against_oracle(big, run=run)
    small = synth.make_workload("after_overflow", synth.FULL_DIMS, [100, 1, 70, 20, 3],
                                [0, 0, 0, 0, 0], 8, 24, block_idx=[1, 2, 3, -1, 4])
    small = dataclasses.replace(small, conv_w=big.conv_w, A_log=big.A_log, dt_bias=big.dt_bias)
    run.set_inputs(small)
    run.run()
    torch.cuda.synchronize()
    check_against_oracle(small, run=run)
    run.close()


@pytest.mark.parametrize("prefill", ["auto", "fused"])
@pytest.mark.parametrize("sign", [-1.0, 1.0])
def test_past_state_outside_fp16_is_recomputed(sign, prefill):
    """A past recurrent state of magnitude 1e5 cannot enter the chunked
    prefill's fp16 operands, whatever its sign: that sequence's v-heads are
    recomputed by the token-serial kernel in the same call, so every output
    and state matches the oracle and no flag is raised (the other sequence
    keeps the tensor-core result)."""
    wl = synth.make_workload("big_state", synth.FULL_DIMS, [130, 70], [1, 0], 8, 25)
    rec = wl.rec_state.clone()
    rec[[int(b) for b in wl.ref_blocks].index(int(wl.block_idx[0]))] = sign * 1.0e5
    wl = dataclasses.replace(wl, rec_state=rec)
    check_against_oracle(wl, prefill=prefill)


@pytest.mark.parametrize("prefill", ["auto", "fused"])
def test_inputs_outside_fp16_are_recomputed(prefill):
    """The v channels of one k-head scaled to about 1e5 in one sequence: its
    values (and u) leave the fp16 range in the chunk products, both v-heads of
    that k-head are recomputed token-serially, and everything matches the
    oracle with no flag raised."""
    wl = synth.make_workload("big_v", synth.FULL_DIMS, [200, 1, 90], [1, 1, 0], 8, 26)
    d = wl.dims
    x = wl.x.float().clone()
    c0 = 2 * d.Hk * d.dk + 6 * d.dv  # v of heads 6 and 7 (k-head 3)
    x[0:200, c0:c0 + 2 * d.dv] *= 1.0e5
    wl = dataclasses.replace(wl, x=x.to(torch.bfloat16))
    check_against_oracle(wl, prefill=prefill)

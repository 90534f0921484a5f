"""Parity of the split prefill path (conv kernel, chunk-parallel kernel,
recurrence kernel) on the shapes that stress its bookkeeping: many short
sequences, sequences ending on and next to chunk boundaries, and rows of the
pool's prefill scratch left non-finite by an earlier call."""
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


def test_stale_nonfinite_scratch_rows_do_not_leak():
    """A first call whose v rows overflow fp16 (and is flagged for it) leaves
    non-finite values in the prefill scratch.  In a second call on the same
    pool, the rows of a decode token and of a padding sequence are never
    written by the prefill kernels, so they still hold those values, and the
    TMA boxes of the partial chunks next to them read them: they must not
    reach a product."""
    big = synth.make_workload("overflow", synth.FULL_DIMS, [300, 200], [0, 0], 8, 23)
    big = dataclasses.replace(big, x=(big.x.float() * 1e5).to(big.x.dtype))
    run = harness.DeviceRun(big)
    run.run()
    torch.cuda.synchronize()
    assert run.pool.error_flags() & binding.FLAG_RANGE
    # rows 100 (a decode token) and 171..190 (padding) keep the first call's values
    small = synth.make_workload("after_overflow", synth.FULL_DIMS, [100, 1, 70, 20, 3],
                                [0, 0, 0, 0, 0], 8, 24, block_idx=[1, 2, 3, -1, 4])
    small = dataclasses.replace(small, conv_w=big.conv_w, A_log=big.A_log, dt_bias=big.dt_bias)
    run.set_inputs(small)
    run.run()
    torch.cuda.synchronize()
    check_against_oracle(small, run=run)
    run.close()


@pytest.mark.parametrize("sign", [-1.0, 1.0])
def test_range_flag_on_a_past_state_outside_fp16(sign):
    """A past recurrent state of magnitude 1e5 cannot enter the recurrence's
    fp16 D-product operand, whatever its sign: the range flag goes up."""
    wl = synth.make_workload("big_state", synth.FULL_DIMS, [130, 70], [1, 0], 8, 25)
    rec = wl.rec_state.clone()
    rec[[int(b) for b in wl.ref_blocks].index(int(wl.block_idx[0]))] = sign * 1.0e5
    wl = dataclasses.replace(wl, rec_state=rec)
    run = harness.DeviceRun(wl)
    run.run()
    torch.cuda.synchronize()
    assert run.pool.error_flags() & binding.FLAG_RANGE
    run.close()

"""GPU parity of the per-channel-decay (KDA) forward against the fp64 oracle,
through the C ABI (gdn_kda_varlen_forward): the decode kernel on the
256-request batch, the token-serial kernel on packed prefills and other head
sizes, and the reduction to the scalar-gate forward when every key channel
has the same gate."""
import dataclasses

import numpy as np
import pytest
import torch

from continuous_linear_attention_gb300 import harness, synth

import oracle
from gpu_check import TOL, check_against_oracle, rel_l2

pytestmark = pytest.mark.gpu


def _kda(name, dims, lens, past, blocks, seed, slow=False):
    return synth.make_workload(name, dims, lens, past, blocks, seed, slow_decay=slow,
                               channel_gate=True)


def test_tiny_packed_fp32():
    check_against_oracle(_kda("kda_tiny", synth.TINY_DIMS, [5, 1, 9], [0, 1, 0], 8, 0))


def test_tiny_packed_fp32_slow_decay():
    check_against_oracle(_kda("kda_tiny_slow", synth.TINY_DIMS, [5, 1, 9], [0, 1, 0], 8, 0,
                              slow=True))


@pytest.mark.parametrize("d", [32, 64])
def test_bf16_mixed_lengths(d):
    dims = synth.Dims(Hk=2, Hv=4, dk=d, dv=d, K=4, act="bf16")
    check_against_oracle(_kda("kda_mixed", dims, [70, 1, 1, 129, 3], [1, 1, 0, 0, 1], 16, 5))


def test_decode_batch_full():
    """256 requests x 1 token at full dims: the HBM-streaming decode kernel."""
    wl = _kda("kda_decode", synth.FULL_DIMS, [1] * 256, [1] * 256, 512, 1)
    check_against_oracle(wl)


def test_mixed_batch_full_dims():
    """Decodes and short continuations together: decode kernel + token-serial
    kernel in one call."""
    lens = [1] * 32 + [65, 130, 17, 200]
    wl = _kda("kda_mixed_full", synth.FULL_DIMS, lens, [1] * len(lens), 64, 3)
    check_against_oracle(wl)


def test_equal_channel_gates_match_the_scalar_forward():
    base = synth.make_workload("g", synth.FULL_DIMS, [1] * 16 + [40], [1] * 17, 32, 6)
    d = base.dims
    kda = dataclasses.replace(
        base, a=base.a[:, :, None].expand(-1, -1, d.dk).contiguous(),
        dt_bias=base.dt_bias[:, None].expand(-1, d.dk).contiguous())
    r1, r2 = harness.DeviceRun(base), harness.DeviceRun(kda)
    r1.run()
    r2.run()
    torch.cuda.synchronize()
    assert r1.pool.error_flags() == 0 and r2.pool.error_flags() == 0
    # the KDA kernels with equal channel gates against the scalar rule's oracle
    check_against_oracle(base, run=r2, ref=oracle.forward(base))
    # and against the scalar forward on the GPU: both sides round their outputs
    # to bf16 on their own (about 1.6e-3 rms apart) and the scalar side's
    # prefill runs on fp16 tensor-core operands, so the bf16 bar applies
    err = rel_l2(r2.out.float().cpu().numpy(), r1.out.float().cpu().numpy())
    assert err <= TOL["bf16"], err


def test_decode_hint_and_graph_replay():
    """A pure decode batch with max_seqlen_hint = 1 (decode kernel only),
    captured once in a CUDA graph and replayed from the same pool contents:
    the replay gives the eager result bit for bit."""
    wl = _kda("kda_graph", synth.FULL_DIMS, [1] * 16, [1] * 16, 32, 7)
    eager = harness.DeviceRun(wl)
    pool0 = eager.mem.clone()
    eager.run(max_seqlen_hint=1)
    torch.cuda.synchronize()
    check_against_oracle(wl, run=eager)
    g = torch.cuda.CUDAGraph()
    eager.mem.copy_(pool0)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        eager.run(torch.cuda.current_stream(), max_seqlen_hint=1)
    eager.mem.copy_(pool0)
    out_eager = eager.out.clone()
    eager.out.fill_(harness.OUT_SENTINEL)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.out, out_eager)


@pytest.mark.parametrize("blocks,flag", [([3, 9, 5], 0x2), ([3, 0, 5], 0x4), ([3, 5, 5], 0x8)])
def test_bad_block_indices_are_flagged_and_skipped(blocks, flag):
    wl = synth.make_workload("kda_bad", synth.TINY_DIMS, [4, 1, 3], [1, 1, 0], 8, 2,
                             block_idx=blocks, channel_gate=True)
    check_against_oracle(wl, expect_flags=flag)

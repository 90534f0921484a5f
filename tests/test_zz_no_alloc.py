"""The allocation-free forward entry point (gdn_varlen_forward_noalloc).

Callers that cannot allocate device memory -- engines that plan all device
memory ahead and forbid runtime allocation, or code running under another
allocator's budget -- pass the pool memory themselves and get the scheduler's
work area from a static device array.  This file is collected last on
purpose: if it fails, a run that stops at the first failure has already run
every other test.  It must pass alone in a fresh process too.
"""
import dataclasses

import numpy as np
import pytest
import torch

from continuous_linear_attention_gb300 import binding, harness, synth

pytestmark = pytest.mark.gpu

TOL = 5e-3  # bf16 activations, fp32 states


def _rel(a, b):
    a = a.double()
    b = b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


def _continuation(wl, seed):
    """A second batch for the same requests (every one has a past now)."""
    nxt = synth.make_workload("noalloc_next", wl.dims, wl.seqlens(), [1] * wl.N, wl.num_blocks,
                              seed, block_idx=[int(v) for v in wl.block_idx])
    return dataclasses.replace(nxt, has_past=torch.ones_like(wl.has_past))


def _noalloc_call(mem, wl, run, x, a, b, cu, idx, hp, out, flags):
    d = wl.dims
    binding.varlen_forward_noalloc(
        mem, wl.num_blocks, 1, d.Hk, d.Hv, d.dk, d.dv, d.K, d.act, 0, 0, x, a, b, cu, idx, hp,
        run.conv_w, run.A_log, run.dt_bias, out, wl.T, wl.N, 0, flags)


def test_noalloc_matches_the_pool_entry_point_on_two_calls():
    wl = synth.make_workload("noalloc", synth.FULL_DIMS, [1, 70, 1, 129, 1, 3], [1, 1, 0, 0, 1, 1],
                             16, 31)
    wl2 = _continuation(wl, 32)
    ref = harness.DeviceRun(wl)
    mem = ref.mem.clone()  # the same pool bytes, for the allocation-free calls
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call, batch in enumerate((wl, wl2)):
        if call:
            ref.set_inputs(batch)
        ref.run()
        dev = {k: getattr(batch, k).cuda() for k in ("x", "a", "b", "cu_seqlens", "block_idx",
                                                     "has_past")}
        out = torch.full_like(ref.out, harness.OUT_SENTINEL)
        _noalloc_call(mem, batch, ref, dev["x"], dev["a"], dev["b"], dev["cu_seqlens"],
                      dev["block_idx"], dev["has_past"], out, flags)
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        assert ref.pool.error_flags() == 0
        assert _rel(out.float(), ref.out.float()) <= TOL, f"call {call}: out differs"
        for s in range(batch.N):
            o = ref.block_offset(int(batch.block_idx[s]))
            r0, r1 = o + ref.rec_off, o + ref.rec_off + ref.rec_bytes
            c0, c1 = o + ref.conv_off, o + ref.conv_off + ref.conv_bytes
            assert _rel(mem[r0:r1].view(torch.float32), ref.mem[r0:r1].view(torch.float32)) <= TOL
            assert torch.equal(mem[c0:c1], ref.mem[c0:c1])
    # bytes outside the written blocks never moved
    written = {int(v) for v in wl.block_idx}
    for blk in range(wl.num_blocks):
        if blk not in written:
            o = ref.block_offset(blk)
            assert torch.equal(mem[o:o + ref.stride], ref.mem[o:o + ref.stride])


def test_noalloc_reports_flags_and_rejects_oversized_pools():
    wl = synth.make_workload("noalloc_bad", synth.TINY_DIMS, [3, 2], [0, 0], 8, 33,
                             block_idx=[2, 2])
    run = harness.DeviceRun(wl)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(run.out, harness.OUT_SENTINEL)
    _noalloc_call(run.mem, wl, run, run.x, run.a, run.b, run.cu, run.idx, run.has_past, out, flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == binding.FLAG_DUPLICATE
    assert (out.float() == harness.OUT_SENTINEL).all()
    d = wl.dims
    with pytest.raises(binding.GdnError) as e:
        binding.varlen_forward_noalloc(
            run.mem, 5000, 1, d.Hk, d.Hv, d.dk, d.dv, d.K, d.act, 0, 0, run.x, run.a, run.b,
            run.cu, run.idx, run.has_past, run.conv_w, run.A_log, run.dt_bias, out, wl.T, wl.N,
            0, flags)
    assert e.value.status == -3


def test_noalloc_with_scratch_after_the_pool_runs_the_split_prefill():
    """Pool memory with gdn_prefill_scratch_bytes more bytes after the pool's
    layout: the allocation-free call runs the split prefill kernels in them,
    exactly as the pool entry point does (bit-identical outputs and states)."""
    wl = synth.make_workload("noalloc_split", synth.FULL_DIMS, [1, 300, 1, 129, 64, 3],
                             [1, 1, 0, 0, 1, 1], 16, 35)
    d = wl.dims
    ref = harness.DeviceRun(wl)
    snapshot = ref.mem.clone()
    ref.run()
    torch.cuda.synchronize()
    assert ref.pool.last_prefill_path() == binding.PREFILL_SPLIT
    extra = binding.prefill_scratch_bytes(wl.num_blocks, d.Hk, d.Hv, d.dk, d.dv, wl.T)
    assert extra > 0
    total = snapshot.numel()
    mem = torch.zeros((total + 255) // 256 * 256 + extra, dtype=torch.uint8, device="cuda")
    mem[:total].copy_(snapshot)
    dev = {k: getattr(wl, k).cuda() for k in ("x", "a", "b", "cu_seqlens", "block_idx",
                                              "has_past")}
    out = torch.full_like(ref.out, harness.OUT_SENTINEL)
    flags = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _noalloc_call(mem, wl, ref, dev["x"], dev["a"], dev["b"], dev["cu_seqlens"],
                  dev["block_idx"], dev["has_past"], out, flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    assert torch.equal(out, ref.out)
    assert torch.equal(mem[:total], ref.mem)

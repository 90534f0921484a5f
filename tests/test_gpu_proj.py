"""GPU parity of the layer's dense neighbours (gdn_in_proj, gdn_out_proj)
against the fp64 oracle, through the C ABI, at the full head dims with
d_model = 2048: each projection alone on ragged row counts, and the whole
layer (input projection -> varlen forward -> gated norm and output
projection) on a packed batch with decodes and prefills."""
import numpy as np
import pytest
import torch

import oracle
from continuous_linear_attention_gb300 import binding, harness, synth

from gpu_check import TOL, log_errs, rel_l2

pytestmark = pytest.mark.gpu


def _bf16(a):
    """The oracle's fp64 value rounded to bf16 (round to nearest even), as the
    interface stores it."""
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("T", [1, 77, 300])
def test_in_proj_matches_the_oracle(T):
    d = synth.FULL_DIMS
    lw = synth.layer_weights(d)
    h = synth.hidden_states(T)
    ref = oracle.in_proj(h, lw.w_qkv, lw.w_z, lw.w_b, lw.w_a)
    dev = "cuda"
    outs = [torch.full((T, n), 7.0, dtype=torch.bfloat16, device=dev)
            for n in (d.C, d.Hv * d.dv, d.Hv, d.Hv)]
    flags = torch.zeros(1, dtype=torch.int32, device=dev)
    binding.in_proj(h.to(dev), lw.w_qkv.to(dev), lw.w_z.to(dev), lw.w_b.to(dev), lw.w_a.to(dev),
                    *outs, d.C, d.Hv, d.dv, flags=flags)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    errs = {name: rel_l2(o.double().cpu().numpy(), r)
            for name, o, r in zip(("x_qkv", "z", "b", "a"), outs, ref)}
    log_errs(errs)
    assert max(errs.values()) <= TOL["bf16"], errs


@pytest.mark.parametrize("T", [3, 200])
def test_out_proj_matches_the_oracle(T):
    d = synth.FULL_DIMS
    lw = synth.layer_weights(d)
    g = torch.Generator().manual_seed(T)
    o = torch.randn(T, d.Hv, d.dv, generator=g).to(torch.bfloat16)
    z = torch.randn(T, d.Hv, d.dv, generator=g).to(torch.bfloat16)
    ref_norm = oracle.gated_rmsnorm(o, z, lw.norm_w, lw.eps)
    ref_y = oracle.out_proj(ref_norm, lw.w_out)
    dev = "cuda"
    o_norm = torch.empty(T, d.Hv, d.dv, dtype=torch.bfloat16, device=dev)
    y = torch.empty(T, lw.d_model, dtype=torch.bfloat16, device=dev)
    binding.out_proj(o.to(dev), z.to(dev), lw.norm_w.to(dev), lw.eps, lw.w_out.to(dev), o_norm, y)
    torch.cuda.synchronize()
    errs = {"o_norm": rel_l2(o_norm.double().cpu().numpy(), ref_norm),
            "y": rel_l2(y.double().cpu().numpy(), ref_y)}
    log_errs(errs)
    assert max(errs.values()) <= TOL["bf16"], errs


def test_whole_layer_matches_the_oracle():
    """hidden -> gdn_in_proj -> gdn_varlen_forward -> gdn_out_proj on a batch
    of decodes and prefills with past states, against the oracle chain
    (in_proj in fp64 rounded to the bf16 the interface stores, the token-loop
    forward, the gated norm and the output projection in fp64)."""
    d = synth.FULL_DIMS
    lw = synth.layer_weights(d)
    wl = synth.make_workload("layer", d, [1, 1, 150, 1, 70], [1, 1, 1, 0, 0], 8, 33)
    h = synth.hidden_states(wl.T, seed=34)
    x_r, z_r, b_r, a_r = oracle.in_proj(h, lw.w_qkv, lw.w_z, lw.w_b, lw.w_a)
    import dataclasses
    wl_ref = dataclasses.replace(wl, x=_bf16(x_r), a=_bf16(a_r), b=_bf16(b_r))
    ref = oracle.forward(wl_ref)
    o_ref = _bf16(ref["out"])  # the forward stores its output in bf16
    z_ref = _bf16(z_r).view(wl.T, d.Hv, d.dv)
    y_ref = oracle.out_proj(oracle.gated_rmsnorm(o_ref, z_ref, lw.norm_w, lw.eps), lw.w_out)

    run = harness.DeviceRun(wl)
    dev = run.device
    z = torch.empty(wl.T, d.Hv * d.dv, dtype=torch.bfloat16, device=dev)
    binding.in_proj(h.to(dev), lw.w_qkv.to(dev), lw.w_z.to(dev), lw.w_b.to(dev), lw.w_a.to(dev),
                    run.x, z, run.b, run.a, d.C, d.Hv, d.dv)
    run.run()
    o_norm = torch.empty(wl.T, d.Hv, d.dv, dtype=torch.bfloat16, device=dev)
    y = torch.empty(wl.T, lw.d_model, dtype=torch.bfloat16, device=dev)
    binding.out_proj(run.out, z.view(wl.T, d.Hv, d.dv), lw.norm_w.to(dev), lw.eps,
                     lw.w_out.to(dev), o_norm, y)
    torch.cuda.synchronize()
    assert run.pool.error_flags() == 0
    errs = {"out": rel_l2(run.out.double().cpu().numpy(), ref["out"]),
            "y": rel_l2(y.double().cpu().numpy(), y_ref)}
    log_errs(errs)
    assert max(errs.values()) <= TOL["bf16"], errs

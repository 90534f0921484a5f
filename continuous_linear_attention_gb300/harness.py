"""Device staging of a synthetic workload for the C-ABI forward.

Puts a generated workload (see ``synth``) on the GPU: a state pool whose
memory is a torch uint8 tensor (so tests can look at every byte), every pool
byte outside block 0 filled with a seeded pattern, the workload's referenced
blocks written at the library's reported offsets, inputs and weights as
device tensors and ``out`` pre-filled with a sentinel.  ``run()`` is one call
of ``gdn_varlen_forward`` (``gdn_kda_varlen_forward`` for per-channel gates).
No arithmetic of the layer happens here.
"""
from __future__ import annotations

import torch

from . import binding
from .synth import SsdWorkload, Workload

OUT_SENTINEL = 12.5


class DeviceRun:
    def __init__(self, wl: Workload, device: str = "cuda", block_align: int = 0,
                 num_layers: int = 1, layer: int = 0, fill: bool = True,
                 prefill: str = "auto"):
        d = wl.dims
        self.wl = wl
        self.layer = layer
        self.device = device
        self.block_align = block_align
        stride, conv_off, rec_off, total = binding.layout_for(
            wl.num_blocks, num_layers, d.Hk, d.Hv, d.dk, d.dv, d.K, d.act, block_align)
        self.mem = torch.empty(total, dtype=torch.uint8, device=device)
        self.pool = binding.Pool(wl.num_blocks, num_layers, d.Hk, d.Hv, d.dk, d.dv, d.K, d.act,
                                 block_align, memory=self.mem)
        if prefill == "fused":
            self.pool.reserve(0)  # one fused prefill kernel, no scratch
        self.stride = stride
        self.conv_off = conv_off
        self.rec_off = rec_off
        self.act_bytes = 4 if d.act == "f32" else 2
        self.conv_bytes = (d.K - 1) * d.C * self.act_bytes
        self.rec_bytes = d.Hv * d.dk * d.dv * 4
        self.page = layer * wl.num_blocks * stride
        if fill:
            g = torch.Generator(device=device)
            g.manual_seed(wl.fill_seed)
            pat = torch.randint(0, 256, (total,), dtype=torch.uint8, device=device, generator=g)
            self.mem.copy_(pat)
            del pat
            for l in range(num_layers):
                base = l * wl.num_blocks * stride
                self.mem[base: base + stride].zero_()  # the trash block reads zeros
        self.upload_states(wl.ref_blocks.tolist(), wl.conv_state, wl.rec_state)
        act = d.torch_act
        self.x = wl.x.to(device)
        self.a = wl.a.to(device)
        self.b = wl.b.to(device)
        self.conv_w = wl.conv_w.to(device)
        self.A_log = wl.A_log.to(device)
        self.dt_bias = wl.dt_bias.to(device)
        self.cu = wl.cu_seqlens.to(device)
        self.idx = wl.block_idx.to(device)
        self.has_past = wl.has_past.to(device)
        self.out = torch.full((wl.T, d.Hv, d.dv), OUT_SENTINEL, dtype=act, device=device)
        torch.cuda.synchronize()

    # -- pool byte views ---------------------------------------------------
    def block_offset(self, blk: int) -> int:
        return self.page + blk * self.stride

    def conv_view(self, blk: int) -> torch.Tensor:
        o = self.block_offset(blk) + self.conv_off
        d = self.wl.dims
        return self.mem[o: o + self.conv_bytes].view(d.torch_act).view(d.K - 1, d.C)

    def rec_view(self, blk: int) -> torch.Tensor:
        o = self.block_offset(blk) + self.rec_off
        d = self.wl.dims
        return self.mem[o: o + self.rec_bytes].view(torch.float32).view(d.Hv, d.dk, d.dv)

    def upload_states(self, blocks, conv_state, rec_state):
        for i, blk in enumerate(blocks):
            self.conv_view(int(blk)).copy_(conv_state[i])
            self.rec_view(int(blk)).copy_(rec_state[i])

    def block_bytes(self, blocks) -> torch.Tensor:
        """CPU uint8 [len(blocks)][stride] copies of whole blocks."""
        return torch.stack([self.mem[self.block_offset(int(b)): self.block_offset(int(b)) +
                                     self.stride] for b in blocks]).cpu()

    # -- the call ----------------------------------------------------------
    def run(self, stream=None, max_seqlen_hint: int = 0):
        """One forward call: gdn_varlen_forward, or gdn_kda_varlen_forward for a
        workload with one gate per key channel."""
        fwd = binding.kda_varlen_forward if self.wl.channel_gate else binding.varlen_forward
        fwd(self.pool, self.layer, self.x, self.a, self.b, self.cu, self.idx, self.has_past,
            self.conv_w, self.A_log, self.dt_bias, self.out, self.wl.T, self.wl.N,
            max_seqlen_hint, stream)

    def set_inputs(self, wl: Workload):
        """Point the run at another batch over the same pool (a continuation)."""
        dev = self.device
        self.wl = wl
        self.x, self.a, self.b = wl.x.to(dev), wl.a.to(dev), wl.b.to(dev)
        self.cu, self.idx, self.has_past = (wl.cu_seqlens.to(dev), wl.block_idx.to(dev),
                                            wl.has_past.to(dev))
        self.out = torch.full((wl.T, wl.dims.Hv, wl.dims.dv), OUT_SENTINEL,
                              dtype=wl.dims.torch_act, device=dev)

    def close(self):
        self.pool.close()


class SsdDeviceRun:
    """The same staging for a Mamba2 mixer workload (``synth.SsdWorkload``):
    a Mamba2 pool in a torch byte tensor filled with a seeded pattern outside
    the trash block, the referenced blocks' conv and SSM states written at the
    library's offsets, inputs on the device, ``y`` pre-filled with the
    sentinel.  ``run()`` is one call of ``gdn_ssd_varlen_forward``."""

    def __init__(self, wl: SsdWorkload, device: str = "cuda", fill_seed: int = 7):
        d = wl.dims
        self.wl = wl
        self.layer = 0
        self.block_align = 0
        stride, conv_off, ssm_off, total = binding.ssd_layout_for(
            wl.num_blocks, 1, d.H, d.P, d.N, d.G, d.K, d.act)
        self.mem = torch.empty(total, dtype=torch.uint8, device=device)
        self.pool = binding.SsdPool(wl.num_blocks, 1, d.H, d.P, d.N, d.G, d.K, d.act,
                                    memory=self.mem)
        self.stride, self.conv_off, self.ssm_off = stride, conv_off, ssm_off
        act = torch.float32 if d.act == "f32" else torch.bfloat16
        self.conv_bytes = (d.K - 1) * d.C * (4 if d.act == "f32" else 2)
        self.ssm_bytes = d.H * d.P * d.N * 4
        g = torch.Generator(device=device)
        g.manual_seed(fill_seed)
        self.mem.copy_(torch.randint(0, 256, (total,), dtype=torch.uint8, device=device,
                                     generator=g))
        self.mem[:stride].zero_()  # the trash block reads zeros
        for i, blk in enumerate(wl.ref_blocks.tolist()):
            o = int(blk) * stride
            self.mem[o: o + self.conv_bytes].view(act).copy_(wl.conv_state[i].reshape(-1))
            self.mem[o + ssm_off: o + ssm_off + self.ssm_bytes].view(torch.float32).copy_(
                wl.ssm_state[i].reshape(-1))
        self.xbc, self.dt = wl.xbc.to(device), wl.dt.to(device)
        self.conv_w = wl.conv_w.to(device)
        self.A_log, self.dt_bias, self.D = (wl.A_log.to(device), wl.dt_bias.to(device),
                                            wl.D.to(device))
        self.cu, self.idx, self.has_past = (wl.cu_seqlens.to(device), wl.block_idx.to(device),
                                            wl.has_past.to(device))
        self.y = torch.full((wl.T, d.H, d.P), OUT_SENTINEL, dtype=act, device=device)
        torch.cuda.synchronize()

    def block_offset(self, blk: int) -> int:
        return blk * self.stride

    def block_bytes(self, blocks) -> torch.Tensor:
        return torch.stack([self.mem[self.block_offset(int(b)): self.block_offset(int(b)) +
                                     self.stride] for b in blocks]).cpu()

    def set_inputs(self, wl: SsdWorkload):
        """Point the run at another batch over the same pool (a continuation)."""
        dev = self.xbc.device
        self.wl = wl
        self.xbc, self.dt = wl.xbc.to(dev), wl.dt.to(dev)
        self.cu, self.idx, self.has_past = (wl.cu_seqlens.to(dev), wl.block_idx.to(dev),
                                            wl.has_past.to(dev))
        act = torch.bfloat16 if wl.dims.act == "bf16" else torch.float32
        self.y = torch.full((wl.T, wl.dims.H, wl.dims.P), OUT_SENTINEL, dtype=act, device=dev)

    def run(self, stream=None, max_seqlen_hint: int = 0):
        binding.ssd_varlen_forward(self.pool, self.layer, self.xbc, self.dt, self.cu, self.idx,
                                   self.has_past, self.conv_w, self.A_log, self.dt_bias, self.D,
                                   self.y, self.wl.T, self.wl.N, max_seqlen_hint, stream)

    def close(self):
        self.pool.close()

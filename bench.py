"""Benchmark of the varlen gated-delta-net layer forward through the C ABI.

One step = one gdn_varlen_forward over one packed batch (scheduler + conv +
recurrence + state write-back, every kernel of the path).  The default
workload is the 256-request decode batch (one token per request, all with a
past, 16 k-heads / 32 v-heads, d_k = d_v = 128, K = 4, bf16 activations, fp32
states, 512-block pool); its state traffic (1 GiB per step) is far larger
than L2, so no flush is needed between steps.

Prints one JSON line: tokens/s of the whole job, the roofline of the dominant
(compute) kernel timed live with CUDA events on the launching stream, the
end-to-end number with host<->device copies from pinned memory inside the
timed region, SM clocks sampled during the timed region, and the fp64 CPU
oracle timed on the host cores on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica of the batch on its
own GPU (requests are independent: no collective on the data path); value is
the tokens of all ranks over the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN varlen layer tokens/s (prefill, decode); decode state HBM GB/s vs peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm = float(d.get("hbm_gbs") or d.get("hbm_GBs") or d["hbm"])
        bf16 = float(d.get("bf16_tflops"))
        bf16s = float(d.get("bf16_tflops_sustained", bf16))
        return {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": bf16s,
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def decode_bytes(wl, requests=None) -> int:
    """Algorithmic HBM bytes of one decode forward (of `requests` decode
    requests, all of the batch's by default): per request the recurrent state
    read + write, the conv state read + write, x, a, b and out; the conv
    weight, A_log and dt_bias once.  With one gate per key channel (KDA) a has
    d_k entries per v-head and dt_bias is [Hv][d_k]."""
    d = wl.dims
    act = 4 if d.act == "f32" else 2
    gate = d.dk if wl.channel_gate else 1
    per_req = (2 * d.Hv * d.dk * d.dv * 4 + 2 * (d.K - 1) * d.C * act + d.C * act
               + d.Hv * gate * act + d.Hv * act + d.Hv * d.dv * act)
    weights = d.C * d.K * act + d.Hv * 4 + d.Hv * gate * 4
    return (wl.N if requests is None else requests) * per_req + weights


def ssd_decode_bytes(wl) -> int:
    """Algorithmic HBM bytes of one Mamba2 decode forward: per request the SSM
    state read + write (H x P x N fp32), the conv state read + write, the xbc
    row, dt and y; the conv weight, A_log, dt_bias and D once."""
    d = wl.dims
    act = 4 if d.act == "f32" else 2
    per_req = (2 * d.H * d.P * d.N * 4 + 2 * (d.K - 1) * d.C * act + d.C * act + d.H * act
               + d.H * d.P * act)
    weights = d.C * d.K * act + 3 * d.H * 4
    return wl.N * per_req + weights


class ClockSampler:
    """nvidia-smi clocks/throttle reasons every 50 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.05)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def traffic_record(kernel_file: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        entry = rec[kernel_file]
        src = os.path.join(ROOT, "continuous_linear_attention_gb300", "csrc", kernel_file)
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if entry.get("source_sha256_16") != digest:
            return None
        return entry["dram_bytes_per_launch"]
    except Exception:
        return None


def prefill_flops(wl, chunk: int = 64) -> float:
    """Algorithmic flops of the chunked form for the tokens of sequences longer
    than one token: per token and v-head 2C(3 d_k + 2 d_v) + 6 d_k d_v (the
    intra-chunk products K K^T, Q K^T, the T-weighted k and v, the P-weighted
    updates; the state products W S^T, Q S^T, U^T K), triangular solve
    excluded."""
    d = wl.dims
    per = 2 * chunk * (3 * d.dk + 2 * d.dv) + 6 * d.dk * d.dv
    toks = sum(L for L in wl.seqlens() if L > 1)
    return float(d.Hv * per * toks)


def prefill_cost(wl):
    """Algorithmic HBM bytes (x, gate inputs and out rows of the sequences
    longer than one token; the per-channel rule's gate input a has d_k values
    per v-head) and the chunked form's flops."""
    d = wl.dims
    act = 4 if d.act == "f32" else 2
    toks = sum(L for L in wl.seqlens() if L > 1)
    gate = d.Hv * (d.dk if wl.channel_gate else 1)
    nbytes = toks * (d.C + gate + d.Hv + d.Hv * d.dv) * act
    return nbytes, prefill_flops(wl)


def time_secondary(harness, wl, steps, device, pk, graph=False, warmup=3):
    """Tokens/s and the compute kernels' roofline for another workload (the
    ~16k-token prefill, the mixed batch), timed like the main line; with
    graph=True also the forward replayed as a CUDA graph."""
    import torch
    run = harness.DeviceRun(wl, device=device)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        run.run(stream)
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in kb + ka:
        e.record(stream)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        run.pool.set_timing_events(kb[i], ka[i])
        run.run(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    run.pool.set_timing_events(None, None)
    ms = start.elapsed_time(stop) / steps
    kall = [kb[i].elapsed_time(ka[i]) for i in range(steps)]
    kms = statistics.mean(kall)
    gms = time_graph(run, steps) if graph else None
    flags = run.pool.error_flags()
    run.close()
    fl = prefill_flops(wl)
    tf = fl / (kms / 1e3) / 1e12
    res = {"workload": wl.name, "tokens": wl.T, "ms_per_step": ms,
           "tokens_per_s": wl.T / (ms / 1e3), "compute_kernels_ms": kms,
           "compute_kernels_ms_median": statistics.median(kall),
           "prefill_tflops": tf, "tensor_frac": tf / pk["bf16_tflops"],
           "algorithmic_flops": fl, "error_flags": flags}
    n_dec = sum(1 for L in wl.seqlens() if L == 1)
    if n_dec:
        # the decode part at the HBM roof and the prefill part at the tensor
        # roof, one after the other: the time a call could take if each part
        # ran at its own roofline; its ratio to the measured time
        dbytes = decode_bytes(wl, n_dec)
        roof_ms = (dbytes / (pk["hbm_gbs"] * 1e9) + fl / (pk["bf16_tflops"] * 1e12)) * 1e3
        res.update({"decode_requests": n_dec, "decode_algorithmic_bytes": dbytes,
                    "decode_gbs_over_call": dbytes / (kms / 1e3) / 1e9,
                    "roofline_sum_ms": roof_ms, "roofline_sum_frac": roof_ms / kms})
    if gms is not None:
        res["graph_replay_ms_per_step"] = gms
        res["graph_replay_tokens_per_s"] = wl.T / (gms / 1e3)
    return res


def time_variant_decode(harness, wl, steps, device, pk, nbytes):
    """One-token-per-request batch of another layer family (the per-channel
    decay rule, the Mamba2 scan): tokens/s and the HBM roofline of its decode
    kernel, timed like the main line."""
    import torch
    ssd = hasattr(wl, "ssm_state")
    run = (harness.SsdDeviceRun if ssd else harness.DeviceRun)(wl, device=device)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        run.run(stream, max_seqlen_hint=1)
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in kb + ka:
        e.record(stream)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        run.pool.set_timing_events(kb[i], ka[i])
        run.run(stream, max_seqlen_hint=1)
    stop.record(stream)
    torch.cuda.synchronize()
    run.pool.set_timing_events(None, None)
    ms = start.elapsed_time(stop) / steps
    kms = statistics.mean(kb[i].elapsed_time(ka[i]) for i in range(steps))
    flags = run.pool.error_flags()
    run.close()
    gbs = nbytes / (kms / 1e3) / 1e9
    return {"workload": wl.name, "tokens": wl.T, "ms_per_step": ms,
            "tokens_per_s": wl.T / (ms / 1e3), "compute_kernels_ms": kms,
            "achieved_gbs": gbs, "hbm_frac": gbs / pk["hbm_gbs"],
            "algorithmic_bytes": nbytes, "error_flags": flags}


def ssd_prefill_cost(wl, chunk: int = 128):
    """Algorithmic HBM bytes and flops of a Mamba2 prefill forward (sequences
    longer than one token): per token the xbc row read, dt and the y row
    written; per token and head the chunk form's products (C B^T shared by a
    group's heads, the masked M X, C h^T and the state step X'^T B)."""
    d = wl.dims
    act = 4 if d.act == "f32" else 2
    toks = sum(L for L in _seqlens(wl) if L > 1)
    nbytes = toks * (d.C * act + d.H * act + d.H * d.P * act)
    per_tok_head = (2 * chunk * d.P + 2 * d.N * d.P + 2 * d.P * d.N
                    + 2 * chunk * d.N / (d.H // d.G))
    return nbytes, toks * d.H * per_tok_head


def _seqlens(wl):
    cu = wl.cu_seqlens.tolist()
    return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]


def time_e2e(run, steps, warmup, hint, world):
    """End to end through the public call: every step copies its inputs from
    pinned host memory to the device and reads its output back to pinned host
    memory, inside the timed region.  As a serving loop does, the inputs travel
    as one packed host buffer into one of two device input sets, and the
    copies run on two copy streams (inputs, outputs): step i's input copy and
    step i-2's output read overlap the forward of step i-1 (the forwards
    themselves stay in order on the compute stream, each reading the states
    the previous one wrote).  Returns (ms for all steps, h2d bytes per step, d2h bytes per
    step)."""
    import torch
    import torch.distributed as dist
    dev = run.x.device
    names = ("x", "a", "b", "cu", "idx", "has_past")
    srcs = [getattr(run, k) for k in names]
    offs, off = [], 0
    for t in srcs:
        offs.append(off)
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    host_in = torch.zeros(off, dtype=torch.uint8).pin_memory()
    for t, o in zip(srcs, offs):
        n = t.numel() * t.element_size()
        host_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    h2d = off

    def views(raw):
        return {k: raw[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for k, t, o in zip(names, srcs, offs)}

    dev_raw = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
    dev_in = [views(r) for r in dev_raw]
    dev_out = [torch.empty_like(run.out) for _ in range(2)]
    host_out = [torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory() for _ in range(2)]
    d2h = host_out[0].numel() * host_out[0].element_size()
    comp = torch.cuda.current_stream()
    cs_in = torch.cuda.Stream(device=dev)
    cs_out = torch.cuda.Stream(device=dev)
    done = [torch.cuda.Event() for _ in range(2)]   # the last forward on this buffer set
    ready = [torch.cuda.Event() for _ in range(2)]  # its inputs landed
    read = [torch.cuda.Event() for _ in range(2)]   # its output read back
    used = [False, False]

    def step(i):
        b = i & 1
        with torch.cuda.stream(cs_in):
            if used[b]:
                cs_in.wait_event(done[b])  # the forward two steps back is done with these inputs
            dev_raw[b].copy_(host_in, non_blocking=True)
            ready[b].record(cs_in)
        comp.wait_event(ready[b])
        if used[b]:
            comp.wait_event(read[b])  # that forward's output has been read back
        for k in names:
            setattr(run, k, dev_in[b][k])
        run.out = dev_out[b]
        run.run(comp, max_seqlen_hint=hint)
        done[b].record(comp)
        with torch.cuda.stream(cs_out):
            cs_out.wait_event(done[b])
            host_out[b].copy_(dev_out[b], non_blocking=True)
            read[b].record(cs_out)
        used[b] = True

    saved = {k: getattr(run, k) for k in names}
    saved_out = run.out
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    cs_in.wait_stream(comp)
    cs_out.wait_stream(comp)
    for i in range(steps):
        step(warmup + i)
    comp.wait_stream(cs_out)  # the last output read back
    e1.record(comp)
    torch.cuda.synchronize()
    for k, v in saved.items():
        setattr(run, k, v)
    run.out = saved_out
    return e0.elapsed_time(e1), h2d, d2h


def ssd_prefill_workload(synth):
    """The Mamba2 prefill batch: the ~16k-token prefill's 8 lengths, no past,
    H = 128, P = 64, N = 128, G = 8, K = 4, bf16."""
    dims = synth.SsdDims(H=128, P=64, N=128, G=8, K=4, act="bf16")
    lens = synth.prefill_lengths()
    return synth.make_ssd_workload("mamba2_prefill_8seq_16k_h128_p64_n128_g8", dims, lens,
                                   [0] * len(lens), 64, 2)


def kda_prefill_workload(synth):
    """The ~16k-token prefill's lengths and head dims under the per-channel
    decay rule, no past."""
    lens = synth.prefill_lengths()
    return synth.make_workload("kda_prefill_8seq_16k", synth.FULL_DIMS, lens, [0] * len(lens),
                               64, 2, channel_gate=True)


def time_variant_prefill(harness, wl, steps, device, pk):
    """A prefill batch of another layer family (the Mamba2 scan, the
    per-channel decay rule): tokens/s and both roofline fractions of its
    compute kernels."""
    import torch
    ssd = hasattr(wl, "ssm_state")
    run = (harness.SsdDeviceRun if ssd else harness.DeviceRun)(wl, device=device)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        run.run(stream)
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for e in kb + ka:
        e.record(stream)
    torch.cuda.synchronize()
    for i in range(steps):
        run.pool.set_timing_events(kb[i], ka[i])
        run.run(stream)
    torch.cuda.synchronize()
    run.pool.set_timing_events(None, None)
    kms = statistics.mean(kb[i].elapsed_time(ka[i]) for i in range(steps))
    flags = run.pool.error_flags()
    run.close()
    nbytes, flops = ssd_prefill_cost(wl) if ssd else prefill_cost(wl)
    gbs = nbytes / (kms / 1e3) / 1e9
    tf = flops / (kms / 1e3) / 1e12
    return {"workload": wl.name, "tokens": wl.T, "compute_kernels_ms": kms,
            "tokens_per_s": wl.T / (kms / 1e3), "achieved_gbs": gbs,
            "hbm_frac": gbs / pk["hbm_gbs"], "tflops": tf, "tensor_frac": tf / pk["bf16_tflops"],
            "algorithmic_bytes": nbytes, "algorithmic_flops": flops, "error_flags": flags}


def time_projections(binding, synth, T, steps, device, pk):
    """The layer's dense neighbours on T tokens (d_model 2048, full head dims):
    gdn_in_proj (hidden -> x_qkv | z | b | a) and gdn_out_proj (gated norm +
    output projection), each timed with CUDA events; dense-contraction flops
    over their time against the bf16 peak."""
    import torch
    d = synth.FULL_DIMS
    lw = synth.layer_weights(d)
    h = synth.hidden_states(T).to(device)
    ws = [t.to(device) for t in (lw.w_qkv, lw.w_z, lw.w_b, lw.w_a, lw.w_out)]
    nw = lw.norm_w.to(device)
    outs = [torch.empty(T, n, dtype=torch.bfloat16, device=device)
            for n in (d.C, d.Hv * d.dv, d.Hv, d.Hv)]
    o = torch.randn(T, d.Hv, d.dv, device=device).to(torch.bfloat16)
    o_norm = torch.empty_like(o)
    y = torch.empty(T, lw.d_model, dtype=torch.bfloat16, device=device)

    def run_in():
        binding.in_proj(h, *ws[:4], *outs, d.C, d.Hv, d.dv)

    def run_out():
        binding.out_proj(o, outs[1].view(T, d.Hv, d.dv), nw, lw.eps, ws[4], o_norm, y)

    res = {"workload": f"layer_projections_{T}tok_dmodel{lw.d_model}", "tokens": T}
    n_in = d.C + d.Hv * d.dv + 2 * d.Hv
    for name, fn, fl in (("in_proj", run_in, 2.0 * T * lw.d_model * n_in),
                         ("out_proj", run_out, 2.0 * T * d.Hv * d.dv * lw.d_model)):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        tf = fl / (ms / 1e3) / 1e12
        res[name] = {"ms": ms, "tflops": tf, "tensor_frac": tf / pk["bf16_tflops"],
                     "algorithmic_flops": fl}
    return res


def time_graph(run, steps, hint=0):
    """The same forward captured once in a CUDA graph and replayed: ms per
    replay (the prefill scratch, if any, was grown by earlier calls)."""
    import torch
    stream = torch.cuda.current_stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run.run(torch.cuda.current_stream(), max_seqlen_hint=hint)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / steps


def time_long_context(harness, binding, synth, device, pk, steps=3):
    """The long-context case: 4 sequences of 32768 tokens with no past, then
    4096 more tokens each continued from the states the first call left; one
    step is both calls."""
    import torch
    first, cont, _ = synth.long_context()
    run = harness.DeviceRun(first, device=device)
    dims = cont.dims
    x2, a2, b2 = cont.x.to(device), cont.a.to(device), cont.b.to(device)
    cu2, idx2, hp2 = (cont.cu_seqlens.to(device), cont.block_idx.to(device),
                      cont.has_past.to(device))
    out2 = torch.empty((cont.T, dims.Hv, dims.dv), dtype=dims.torch_act, device=device)
    stream = torch.cuda.current_stream()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps + 1)]
    for e4 in ev:  # create the events (torch makes them on first record)
        for e in e4:
            e.record(stream)

    def step(e):
        run.pool.set_timing_events(e[0], e[1])
        run.run(stream)
        run.pool.set_timing_events(e[2], e[3])
        binding.varlen_forward(run.pool, run.layer, x2, a2, b2, cu2, idx2, hp2, run.conv_w,
                               run.A_log, run.dt_bias, out2, cont.T, cont.N, 0, stream)

    step(ev[steps])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(ev[i])
    e1.record(stream)
    torch.cuda.synchronize()
    run.pool.set_timing_events(None, None)
    ms = e0.elapsed_time(e1) / steps
    k_first = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(steps))
    k_cont = statistics.mean(ev[i][2].elapsed_time(ev[i][3]) for i in range(steps))
    flags = run.pool.error_flags()
    run.close()
    fl = prefill_flops(first) + prefill_flops(cont)
    tf = fl / (ms / 1e3) / 1e12
    tokens = first.T + cont.T
    kms = k_first + k_cont
    tfk = fl / (kms / 1e3) / 1e12
    return {"workload": "long_4x32768_then_4x4096", "tokens": tokens, "ms_per_step": ms,
            "tokens_per_s": tokens / (ms / 1e3), "compute_kernels_ms": kms,
            "compute_kernels_ms_first_call": k_first, "compute_kernels_ms_continuation": k_cont,
            "prefill_tflops": tfk, "tensor_frac": tfk / pk["bf16_tflops"],
            "algorithmic_flops": fl, "error_flags": flags,
            "note": "one step is both calls; TFLOP/s over the compute kernels' time"}


def max_over_ranks(values, device="cpu"):
    """Element-wise max of a list of floats over all ranks (identity when not
    distributed): the job's time is its slowest rank's."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def cpu_baseline(wl, budget_s: float = 12.0, one_thread_s: float = 0.0):
    """The fp64 oracle as it stands, on the host cores, on a bounded sample of
    the workload (its first requests), scaled to tokens/s.  With one_thread_s
    > 0 the same sample is also timed on one thread for about that long."""
    import dataclasses

    import oracle
    cu = wl.cu_seqlens.tolist()
    n = min(wl.N, 64)
    T = cu[n]
    sub = dataclasses.replace(wl, x=wl.x[:T], a=wl.a[:T], b=wl.b[:T],
                              cu_seqlens=wl.cu_seqlens[:n + 1].clone(),
                              block_idx=wl.block_idx[:n], has_past=wl.has_past[:n])

    def timed(budget, nthreads):
        reps, t0, threads = 0, time.perf_counter(), 1
        while True:
            res = oracle.forward(sub, nthreads=nthreads)
            threads = res["threads"]
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget or reps >= 50:
                return reps, el, threads

    reps, el, threads = timed(budget_s, 0)
    out = {"value": reps * T / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
           "sample": f"first {n} of {wl.N} requests ({T} tokens), {reps} passes, "
                     f"{el:.1f} s wall, fp64 token-by-token"}
    if one_thread_s > 0:
        r1, e1, _ = timed(one_thread_s, 1)
        out["value_1_thread"] = r1 * T / e1
    return out


def run_reference(args, rank, world):
    """The oracle (fp64, host cores) as the reference arm."""
    if rank != 0:
        return
    from continuous_linear_attention_gb300 import synth
    wl = synth.decode_batch()
    cb = cpu_baseline(wl, budget_s=max(2.0, 20.0 / max(1, args.steps + args.warmup)))
    line = {
        "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode_256req_bf16act_fp32state", "requests": wl.N,
                   "Hk": wl.dims.Hk, "Hv": wl.dims.Hv, "d": wl.dims.dk, "K": wl.dims.K},
        "cpu_baseline": cb,
        "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# the headline loop records the kernel events on one step in this many
KERNEL_EVERY = 8


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--requests", type=int, default=256,
                    help="decode requests per GPU (256 is the standard batch; smaller "
                         "batches are for profiler captures)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the prefill / mixed-batch / long-context measurements")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the long-context measurement (4 x 32768 + 4 x 4096 tokens)")
    ap.add_argument("--variants", action="store_true",
                    help="also time the decode batches of the per-channel-decay rule and of "
                         "the Mamba2 scan")
    ap.add_argument("--profile",
                    choices=["prefill", "mixed", "long", "proj", "ssd_prefill", "kda_prefill"],
                    default=None,
                    help="profiler aid: run only the ~16k-token prefill, the mixed batch, "
                         "the long-context pair of calls, the layer's projections on 15843 "
                         "tokens, or the Mamba2 or "
                         "per-channel-decay prefill of the same lengths, --warmup + --steps "
                         "times, and print their timing line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl")

    import __graft_entry__
    __graft_entry__.build()
    from continuous_linear_attention_gb300 import harness, synth

    if args.profile == "proj":
        from continuous_linear_attention_gb300 import binding
        res = time_projections(binding, synth, 15843, args.steps, f"cuda:{local_rank}", peaks())
        print(json.dumps({"profile": args.profile, **res}), flush=True)
        return
    if args.profile == "long":
        from continuous_linear_attention_gb300 import binding
        res = time_long_context(harness, binding, synth, f"cuda:{local_rank}", peaks(),
                                steps=args.steps)
        print(json.dumps({"profile": args.profile, **res}), flush=True)
        return
    if args.profile in ("ssd_prefill", "kda_prefill"):
        wl = (ssd_prefill_workload if args.profile == "ssd_prefill" else kda_prefill_workload)(synth)
        res = time_variant_prefill(harness, wl, args.steps, f"cuda:{local_rank}", peaks())
        print(json.dumps({"profile": args.profile, **res}), flush=True)
        return
    if args.profile:
        wl = synth.packed_prefill() if args.profile == "prefill" else synth.mixed_batch()
        res = time_secondary(harness, wl, args.steps, f"cuda:{local_rank}", peaks(),
                             warmup=args.warmup)
        print(json.dumps({"profile": args.profile, **res}), flush=True)
        return

    wl = synth.decode_batch(seed=1 + rank, n_req=args.requests,
                            num_blocks=max(512, 2 * args.requests))
    run = harness.DeviceRun(wl, device=f"cuda:{local_rank}")
    stream = torch.cuda.current_stream()

    # warm-up
    # every request of this batch has one new token: the decode fast path
    hint = 1
    for _ in range(args.warmup):
        run.run(stream, max_seqlen_hint=hint)
    torch.cuda.synchronize()

    # events around the compute kernels (inside the C-ABI call) on every
    # KERNEL_EVERY-th timed step: an event between the scheduler and the decode
    # kernel keeps that step's kernels from overlapping (programmatic
    # dependent launch), so the other steps run without one
    n_kev = (args.steps + KERNEL_EVERY - 1) // KERNEL_EVERY
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(n_kev)]
    ka = [torch.cuda.Event(enable_timing=True) for _ in range(n_kev)]
    for e in kb + ka:
        e.record(stream)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        clk.wait_first()
        start.record(stream)
        for i in range(args.steps):
            if i % KERNEL_EVERY == 0:
                run.pool.set_timing_events(kb[i // KERNEL_EVERY], ka[i // KERNEL_EVERY])
            elif i % KERNEL_EVERY == 1:
                run.pool.set_timing_events(None, None)
            run.run(stream, max_seqlen_hint=hint)
        stop.record(stream)
        torch.cuda.synchronize()
    run.pool.set_timing_events(None, None)
    elapsed_ms = start.elapsed_time(stop)
    graph_ms = time_graph(run, min(args.steps, 200), hint)
    kern_ms = [kb[i].elapsed_time(ka[i]) for i in range(n_kev)]
    flags = run.pool.error_flags()
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} during the bench")

    e2e_ms, h2d, d2h = time_e2e(run, args.steps, args.warmup, hint, world)

    # max over ranks
    elapsed_ms, e2e_ms, kern_mean_ms = max_over_ranks(
        [elapsed_ms, e2e_ms, statistics.mean(kern_ms)], device=f"cuda:{local_rank}")

    if rank == 0:
        pk = peaks()
        tokens = wl.T * world * args.steps
        value = tokens / (elapsed_ms / 1e3)
        alg_bytes = decode_bytes(wl)
        achieved = alg_bytes / (kern_mean_ms / 1e3) / 1e9
        traffic = traffic_record("gdn_decode.cu")
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": "decode_256req_bf16act_fp32state", "requests_per_gpu": wl.N,
                       "tokens_per_gpu": wl.T, "Hk": wl.dims.Hk, "Hv": wl.dims.Hv,
                       "d_k": wl.dims.dk, "d_v": wl.dims.dv, "K": wl.dims.K,
                       "act": wl.dims.act, "state": "fp32", "pool_blocks": wl.num_blocks,
                       "l2": "no flush: 1 GiB of state traffic per step, > 129 MB L2",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                         "traffic": traffic, "peak_source": pk["source"],
                         "kernel": "decode_kernel (the only compute kernel of a decode batch)",
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "kernel_ms_mean": kern_mean_ms,
                         "kernel_ms_median": statistics.median(kern_ms)},
            "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "copies": "per step one packed input copy from pinned host memory and the "
                              "output read back to pinned host memory, on two copy streams with "
                              "two device buffer sets, overlapping the neighbouring forwards"},
            "gpu_launches": 2 * args.steps,
            "timing_note": f"one device-timed step in {KERNEL_EVERY} also records, inside the "
                           "call, the CUDA events around its compute kernels that give "
                           f"roofline.achieved ({n_kev} launches averaged; such a step loses "
                           "the scheduler/decode launch overlap, a few µs); the e2e loop and "
                           "the graph replay record none",
            "clocks": clk.summary(),
            "graph_replay": {"ms_per_step": graph_ms,
                             "tokens_per_s": wl.T * world / (graph_ms / 1e3),
                             "note": "the decode step captured once as a CUDA graph and replayed"},
        }
        if not args.no_secondary:
            from continuous_linear_attention_gb300 import binding
            dev = f"cuda:{local_rank}"
            line["secondary"] = [
                time_secondary(harness, synth.packed_prefill(), 20, dev, pk),
                time_secondary(harness, synth.mixed_batch(), 20, dev, pk, graph=True),
            ]
            if not args.no_long:
                line["secondary"].append(time_long_context(harness, binding, synth, dev, pk))
            line["secondary"].append(time_projections(binding, synth, 15843, 20, dev, pk))
        if args.variants:
            dev = f"cuda:{local_rank}"
            kda = synth.make_workload("kda_decode_256req", synth.FULL_DIMS, [1] * 256, [1] * 256,
                                      512, 1, channel_gate=True)
            ssd = synth.make_ssd_workload("mamba2_decode_256req_h128_p64_n128_g8",
                                          synth.SsdDims(H=128, P=64, N=128, G=8, K=4,
                                                        act="bf16"),
                                          [1] * 256, [1] * 256, 512, 1)
            ssd_pre = ssd_prefill_workload(synth)
            line["variants"] = [
                time_variant_decode(harness, kda, 200, dev, pk, decode_bytes(kda)),
                time_variant_decode(harness, ssd, 200, dev, pk, ssd_decode_bytes(ssd)),
                time_variant_prefill(harness, ssd_pre, 10, dev, pk),
                time_variant_prefill(harness, kda_prefill_workload(synth), 5, dev, pk),
            ]
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl, one_thread_s=4.0)
        print(json.dumps(line), flush=True)
    run.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

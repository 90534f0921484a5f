"""Seeded synthetic workloads for the varlen gated-delta-net layer forward.

This module only draws random numbers and packs them; it holds none of the
layer's arithmetic, so both the CUDA path's tests and the fp64 oracle take
their inputs from here.

The workloads follow the shapes and value distributions of the five test
cases of this project (a tiny fp32 packed batch, a 256-request decode batch,
a ~16k-token packed prefill, a mixed continuous batch and a long-context
prefill continued from its saved states), plus a slow-decay variant used to
make split/continue checks meaningful (with the default gate distribution the
state forgets within a few tokens).

Value recipe (sigma is a standard deviation):
  x, a, b ~ N(0, 1);  conv weight ~ N(0, 0.5);  A_log = log U(1, 16);
  dt_bias ~ N(0, 0.1);  past recurrent states ~ N(0, 0.02) (fp32);
  past conv states ~ N(0, 1) (activation dtype).
Activation-dtype values are drawn in fp32 and rounded to bf16 (round to
nearest even) once; every consumer sees the rounded values.

Per-channel gates (the KDA variant): with ``channel_gate`` the gate input
``a`` has one entry per key channel, [T][Hv][dk] ~ N(0, 1), and ``dt_bias``
is [Hv][dk] ~ N(0, 0.1) (slow decay: -8 everywhere); nothing else changes.

Pool contents: block 0 is the zeroed trash block; blocks of requests with a
past hold their state; blocks written by requests without a past are filled
with NaN (so a kernel that reads them instead of the trash block is caught).
Only these referenced blocks are materialised here; every other pool byte is
filled by the harness from ``fill_seed`` and must survive byte for byte.

State orientation: ``rec[b][h][k][v]`` is element S_h[v][k] of the d_v x d_k
state matrix of v-head h in block b (k-major, v contiguous), which is also
the byte order of the recurrent sub-state inside a pool block.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

F32 = "f32"
BF16 = "bf16"


@dataclasses.dataclass
class Dims:
    Hk: int
    Hv: int
    dk: int
    dv: int
    K: int
    act: str  # "f32" or "bf16"

    @property
    def C(self) -> int:
        """Conv channels: q | k | v."""
        return 2 * self.Hk * self.dk + self.Hv * self.dv

    @property
    def torch_act(self):
        return torch.float32 if self.act == F32 else torch.bfloat16


@dataclasses.dataclass
class Workload:
    name: str
    dims: Dims
    num_blocks: int
    # inputs (CPU tensors)
    x: torch.Tensor  # [T][C] act
    a: torch.Tensor  # [T][Hv] act ([T][Hv][dk] with per-channel gates)
    b: torch.Tensor  # [T][Hv] act
    conv_w: torch.Tensor  # [C][K] act
    A_log: torch.Tensor  # [Hv] f32
    dt_bias: torch.Tensor  # [Hv] f32 ([Hv][dk] with per-channel gates)
    cu_seqlens: torch.Tensor  # [N+1] int32
    block_idx: torch.Tensor  # [N] int32
    has_past: torch.Tensor  # [N] uint8
    # pool contents before the call, for the referenced blocks only:
    # ref_blocks[0] == 0 (trash), then every block the batch names, ascending.
    ref_blocks: torch.Tensor  # [R] int64
    conv_state: torch.Tensor  # [R][K-1][C] act
    rec_state: torch.Tensor  # [R][Hv][dk][dv] f32
    fill_seed: int = 0  # seed of the pattern held by every other pool byte

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def N(self) -> int:
        return int(self.block_idx.numel())

    @property
    def channel_gate(self) -> bool:
        """One gate per key channel (KDA) rather than one per head."""
        return self.a.dim() == 3

    def seqlens(self) -> List[int]:
        cu = self.cu_seqlens.tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]


def _rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def _normal(rng: np.random.Generator, shape, sigma: float = 1.0) -> np.ndarray:
    out = rng.standard_normal(shape, dtype=np.float32)
    if sigma != 1.0:
        out *= np.float32(sigma)
    return out


def _act(arr: np.ndarray, act: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    return t if act == F32 else t.to(torch.bfloat16)


def make_workload(name: str, dims: Dims, seqlens: List[int], has_past: List[int],
                  num_blocks: int, seed: int, block_idx: Optional[List[int]] = None,
                  slow_decay: bool = False, channel_gate: bool = False) -> Workload:
    """Draw one packed batch and the pool contents it runs against.

    ``block_idx`` defaults to a seeded random permutation of blocks
    1..num_blocks-1 (block 0 is the trash block); entries < 0 mark padding
    sequences.
    """
    rng = _rng(seed)
    N = len(seqlens)
    T = int(sum(seqlens))
    C = dims.C
    if block_idx is None:
        if N > num_blocks - 1:
            raise ValueError("more sequences than non-trash blocks")
        perm = rng.permutation(np.arange(1, num_blocks))
        block_idx = [int(v) for v in perm[:N]]
    x = _normal(rng, (T, C))
    a = _normal(rng, (T, dims.Hv, dims.dk) if channel_gate else (T, dims.Hv))
    b = _normal(rng, (T, dims.Hv))
    conv_w = _normal(rng, (C, dims.K), 0.5)
    gshape = (dims.Hv, dims.dk) if channel_gate else dims.Hv
    if slow_decay:
        A_log = np.log(rng.uniform(0.01, 0.1, dims.Hv))
        dt_bias = np.full(gshape, -8.0)
    else:
        A_log = np.log(rng.uniform(1.0, 16.0, dims.Hv))
        dt_bias = rng.standard_normal(gshape) * 0.1

    ref = sorted({0} | {int(v) for v in block_idx if 0 <= int(v) < num_blocks})
    pos = {blk: i for i, blk in enumerate(ref)}
    R = len(ref)
    conv_state = np.zeros((R, dims.K - 1, C), dtype=np.float32)
    rec_state = np.zeros((R, dims.Hv, dims.dk, dims.dv), dtype=np.float32)
    for s in range(N):
        blk = int(block_idx[s])
        if blk <= 0 or blk >= num_blocks:
            continue
        i = pos[blk]
        if has_past[s]:
            conv_state[i] = _normal(rng, (dims.K - 1, C))
            rec_state[i] = _normal(rng, (dims.Hv, dims.dk, dims.dv), 0.02)
        else:
            conv_state[i] = np.nan
            rec_state[i] = np.nan

    cu = np.zeros(N + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64))
    return Workload(
        name=name, dims=dims, num_blocks=num_blocks,
        x=_act(x, dims.act), a=_act(a, dims.act), b=_act(b, dims.act),
        conv_w=_act(conv_w, dims.act),
        A_log=torch.from_numpy(A_log.astype(np.float32)),
        dt_bias=torch.from_numpy(dt_bias.astype(np.float32)),
        cu_seqlens=torch.from_numpy(cu),
        block_idx=torch.tensor(block_idx, dtype=torch.int32),
        has_past=torch.tensor([1 if p else 0 for p in has_past], dtype=torch.uint8),
        ref_blocks=torch.tensor(ref, dtype=torch.int64),
        conv_state=_act(conv_state, dims.act),
        rec_state=torch.from_numpy(rec_state),
        fill_seed=seed + 1000,
    )


# --------------------------------------------------------------------------
# The five standard cases.

TINY_DIMS = Dims(Hk=2, Hv=4, dk=32, dv=32, K=4, act=F32)
FULL_DIMS = Dims(Hk=16, Hv=32, dk=128, dv=128, K=4, act=BF16)


def tiny_packed(seed: int = 0, slow_decay: bool = False) -> Workload:
    """3 sequences of lengths {5, 1, 9}; the length-1 one is a decode with a
    past, the others start from the trash block.  2 k-heads, 4 v-heads,
    d_k = d_v = 32, K = 4, fp32 everywhere, 8 pool blocks."""
    return make_workload("tiny_packed_fp32", TINY_DIMS, [5, 1, 9], [0, 1, 0], 8, seed,
                         slow_decay=slow_decay)


def decode_batch(seed: int = 1, n_req: int = 256, num_blocks: int = 512,
                 dims: Dims = FULL_DIMS, slow_decay: bool = False) -> Workload:
    """256 requests with one new token each, all with a past, mapped to a
    random permutation of blocks 1..511 of a 512-block pool."""
    return make_workload(f"decode_{n_req}req", dims, [1] * n_req, [1] * n_req, num_blocks, seed,
                         slow_decay=slow_decay)


def prefill_lengths(seed: int = 2, n: int = 8, lo: int = 512, hi: int = 4096,
                    total_lo: int = 15360, total_hi: int = 17408) -> List[int]:
    """n lengths uniform in [lo, hi], redrawn until the total is ~16k tokens."""
    rng = _rng(seed)
    while True:
        lens = rng.integers(lo, hi + 1, n)
        if total_lo <= int(lens.sum()) <= total_hi:
            return [int(v) for v in lens]


def packed_prefill(seed: int = 2, num_blocks: int = 64, dims: Dims = FULL_DIMS,
                   slow_decay: bool = False) -> Workload:
    """8 sequences, lengths U[512, 4096] totalling ~16k tokens, no past."""
    lens = prefill_lengths(seed)
    return make_workload("prefill_8seq_16k", dims, lens, [0] * len(lens), num_blocks, seed,
                         slow_decay=slow_decay)


def mixed_lengths(seed: int = 3, n_dec: int = 64, n_pre: int = 6, lo: int = 256, hi: int = 2048,
                  total: int = 8192):
    """64 decode tokens plus 6 prefill continuations U[256, 2048] summing to
    8192 tokens (the last prefill length is set by the total and redrawn until
    in range).  Returns (lengths, order) with the 70 sequences shuffled."""
    rng = _rng(seed)
    want = total - n_dec
    while True:
        first = rng.integers(lo, hi + 1, n_pre - 1)
        last = want - int(first.sum())
        if lo <= last <= hi:
            break
    pre = [int(v) for v in first] + [last]
    lens = [1] * n_dec + pre
    order = rng.permutation(len(lens))
    return [lens[i] for i in order]


def mixed_batch(seed: int = 3, num_blocks: int = 1024, dims: Dims = FULL_DIMS,
                slow_decay: bool = False) -> Workload:
    """64 decode requests + 6 chunked-prefill continuations, all with past,
    8192 tokens, 1024-block pool with random block assignment."""
    lens = mixed_lengths(seed)
    return make_workload("mixed_64dec_6pre_8k", dims, lens, [1] * len(lens), num_blocks, seed,
                         slow_decay=slow_decay)


def long_context(seed: int = 4, n: int = 4, first: int = 32768, cont: int = 4096,
                 dims: Dims = FULL_DIMS, slow_decay: bool = False):
    """4 sequences of 32768 tokens with no past, then 4096 more tokens each
    continued from the saved states; also the single 36864-token pass over
    the same tokens.  Returns (first_call, continuation_call, single_pass),
    three workloads sharing x, weights and block assignment; the
    continuation's pool contents are whatever the first call leaves, so only
    its x/a/b/cu_seqlens/has_past are meaningful."""
    total = first + cont
    whole = make_workload("long_single_pass", dims, [total] * n, [0] * n, 2 * n + 1, seed,
                          slow_decay=slow_decay)
    C = dims.C
    xs = whole.x.view(n, total, C)
    as_ = whole.a.view(n, total, dims.Hv)
    bs = whole.b.view(n, total, dims.Hv)

    def part(lo, hi, past, name):
        L = hi - lo
        cu = torch.arange(n + 1, dtype=torch.int32) * L
        return dataclasses.replace(
            whole, name=name,
            x=xs[:, lo:hi].reshape(n * L, C).contiguous(),
            a=as_[:, lo:hi].reshape(n * L, dims.Hv).contiguous(),
            b=bs[:, lo:hi].reshape(n * L, dims.Hv).contiguous(),
            cu_seqlens=cu, has_past=torch.full((n,), past, dtype=torch.uint8))

    return part(0, first, 0, "long_first_32k"), part(first, total, 1, "long_cont_4k"), whole


def row_split(wl: Workload, cuts: List[int]):
    """Split every sequence of ``wl`` at its own cut (tokens of the first
    part; 0 < cut < length) into two consecutive calls on the same blocks: the
    first with the workload's own has_past, the second continuing from the
    states the first leaves (has_past = 1).  Only the batch description and
    x/a/b change; weights, blocks and the pool contents are the workload's."""
    cu = wl.cu_seqlens.tolist()
    parts = []
    for first in (True, False):
        rows, lens = [], []
        for s in range(wl.N):
            lo, hi = cu[s], cu[s + 1]
            mid = lo + cuts[s]
            r = range(lo, mid) if first else range(mid, hi)
            rows.extend(r)
            lens.append(len(r))
        idx = torch.tensor(rows, dtype=torch.int64)
        ncu = np.zeros(wl.N + 1, dtype=np.int32)
        ncu[1:] = np.cumsum(lens)
        hp = wl.has_past.clone() if first else torch.ones(wl.N, dtype=torch.uint8)
        parts.append(dataclasses.replace(
            wl, name=wl.name + ("_first" if first else "_cont"), x=wl.x[idx].contiguous(),
            a=wl.a[idx].contiguous(), b=wl.b[idx].contiguous(),
            cu_seqlens=torch.from_numpy(ncu), has_past=hp))
    return parts[0], parts[1]


def standard_cases():
    """Name -> builder for the five standard cases."""
    return {
        "tiny": tiny_packed,
        "decode": decode_batch,
        "prefill": packed_prefill,
        "mixed": mixed_batch,
        "long": long_context,
    }


# --------------------------------------------------------------------------
# Mamba2 mixer workloads (conv over x | B | C, then the selective scan).

@dataclasses.dataclass
class SsdDims:
    H: int   # heads
    P: int   # head dim
    N: int   # state size
    G: int   # groups sharing B and C
    K: int   # conv width
    act: str

    @property
    def C(self) -> int:
        """Conv channels: x | B | C."""
        return self.H * self.P + 2 * self.G * self.N


@dataclasses.dataclass
class SsdWorkload:
    name: str
    dims: SsdDims
    num_blocks: int
    xbc: torch.Tensor  # [T][C] act
    dt: torch.Tensor  # [T][H] act
    conv_w: torch.Tensor  # [C][K] act
    A_log: torch.Tensor  # [H] f32
    dt_bias: torch.Tensor  # [H] f32
    D: torch.Tensor  # [H] f32
    cu_seqlens: torch.Tensor  # [N+1] int32
    block_idx: torch.Tensor  # [N] int32
    has_past: torch.Tensor  # [N] uint8
    ref_blocks: torch.Tensor  # [R] int64, ref_blocks[0] == 0
    conv_state: torch.Tensor  # [R][K-1][C] act
    ssm_state: torch.Tensor  # [R][H][P][N] f32

    @property
    def T(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def N(self) -> int:
        return int(self.block_idx.numel())


def make_ssd_workload(name: str, dims: SsdDims, seqlens: List[int], has_past: List[int],
                      num_blocks: int, seed: int, block_idx: Optional[List[int]] = None,
                      slow_decay: bool = False) -> SsdWorkload:
    """One packed batch for a Mamba2 mixer and the pool contents it runs
    against.  Recipe: xbc, dt ~ N(0, 1); conv weight ~ N(0, 0.5);
    A_log = log U(1, 16); dt_bias = softplus^-1 of log-uniform [1e-3, 1e-1]
    (the usual Mamba2 time-step range); D ~ N(1, 0.1); past conv states
    ~ N(0, 1), past SSM states ~ N(0, 0.02); blocks written by requests with
    no past hold NaN.  Slow decay: A_log = log U(0.01, 0.1) and dt = -4
    (small, slowly forgetting time steps)."""
    rng = _rng(seed)
    N = len(seqlens)
    T = int(sum(seqlens))
    C = dims.C
    if block_idx is None:
        if N > num_blocks - 1:
            raise ValueError("more sequences than non-trash blocks")
        perm = rng.permutation(np.arange(1, num_blocks))
        block_idx = [int(v) for v in perm[:N]]
    xbc = _normal(rng, (T, C))
    dt = _normal(rng, (T, dims.H))
    conv_w = _normal(rng, (C, dims.K), 0.5)
    step = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), dims.H))
    dt_bias = step + np.log(-np.expm1(-step))  # softplus(dt_bias) = step
    if slow_decay:
        A_log = np.log(rng.uniform(0.01, 0.1, dims.H))
        dt[:] = -4.0
    else:
        A_log = np.log(rng.uniform(1.0, 16.0, dims.H))
    D = 1.0 + 0.1 * rng.standard_normal(dims.H)
    ref = sorted({0} | {int(v) for v in block_idx if 0 <= int(v) < num_blocks})
    pos = {blk: i for i, blk in enumerate(ref)}
    R = len(ref)
    conv_state = np.zeros((R, dims.K - 1, C), dtype=np.float32)
    ssm_state = np.zeros((R, dims.H, dims.P, dims.N), dtype=np.float32)
    for s in range(N):
        blk = int(block_idx[s])
        if blk <= 0 or blk >= num_blocks:
            continue
        i = pos[blk]
        if has_past[s]:
            conv_state[i] = _normal(rng, (dims.K - 1, C))
            ssm_state[i] = _normal(rng, (dims.H, dims.P, dims.N), 0.02)
        else:
            conv_state[i] = np.nan
            ssm_state[i] = np.nan
    cu = np.zeros(N + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64))
    return SsdWorkload(
        name=name, dims=dims, num_blocks=num_blocks,
        xbc=_act(xbc, dims.act), dt=_act(dt, dims.act), conv_w=_act(conv_w, dims.act),
        A_log=torch.from_numpy(A_log.astype(np.float32)),
        dt_bias=torch.from_numpy(dt_bias.astype(np.float32)),
        D=torch.from_numpy(D.astype(np.float32)),
        cu_seqlens=torch.from_numpy(cu),
        block_idx=torch.tensor(block_idx, dtype=torch.int32),
        has_past=torch.tensor([1 if p else 0 for p in has_past], dtype=torch.uint8),
        ref_blocks=torch.tensor(ref, dtype=torch.int64),
        conv_state=_act(conv_state, dims.act),
        ssm_state=torch.from_numpy(ssm_state),
    )


# --------------------------------------------------------------------------
# The dense neighbours of the forward (input projection, gated norm, output
# projection), with random-init weights of a hybrid model's gated-delta-net
# layer: d_model = 2048 with the full head dims (16 k-heads, 32 v-heads,
# d = 128) is the size class of the Qwen3-Next gated-delta-net layers.

@dataclasses.dataclass
class LayerWeights:
    d_model: int
    w_qkv: torch.Tensor   # [C][d_model] bf16, rows q | k | v
    w_z: torch.Tensor     # [Hv*dv][d_model] bf16
    w_b: torch.Tensor     # [Hv][d_model] bf16
    w_a: torch.Tensor     # [Hv][d_model] bf16
    w_out: torch.Tensor   # [d_model][Hv*dv] bf16
    norm_w: torch.Tensor  # [dv] f32
    eps: float = 1e-6


def layer_weights(dims: Dims, d_model: int = 2048, seed: int = 31) -> LayerWeights:
    """Projection weights ~ N(0, 1/fan_in) (so every output is ~N(0, 1) for
    unit inputs), norm weight ~ 1 + N(0, 0.1); bf16 except the norm weight."""
    rng = _rng(seed)
    C, HV = dims.C, dims.Hv * dims.dv

    def w(n_out, n_in):
        return _act(_normal(rng, (n_out, n_in), 1.0 / np.sqrt(n_in)), BF16)

    return LayerWeights(d_model=d_model, w_qkv=w(C, d_model), w_z=w(HV, d_model),
                        w_b=w(dims.Hv, d_model), w_a=w(dims.Hv, d_model), w_out=w(d_model, HV),
                        norm_w=torch.from_numpy(1.0 + _normal(rng, (dims.dv,), 0.1)))


def hidden_states(T: int, d_model: int = 2048, seed: int = 32) -> torch.Tensor:
    """Layer inputs [T][d_model] ~ N(0, 1), bf16."""
    return _act(_normal(_rng(seed), (T, d_model)), BF16)

"""fp64 CPU oracle for the varlen gated-delta-net layer forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA path (no kernels, headers, helpers, layout code or constants); the
only thing both sides use is the seeded input generator, which holds none of
the layer's arithmetic.

Contents:
  * ``forward``      -- the plain token-by-token fp64 forward (C, gdn_oracle.c),
                        on the referenced blocks of a workload; workloads with
                        one gate per key channel run the KDA rule;
  * ``gdn_rule_head`` / ``kda_rule_head`` -- the two rules on one chain;
  * ``data_errors``  -- which sequences the rules for bad input skip;
  * ``pool_layout``  -- the state-pool byte layout as the boundary states it
                        (conv sub-state at 0, recurrent sub-state at the next
                        128-byte boundary, block stride rounded up);
  * ``read_pool_states`` -- decode a pool byte image with that layout;
  * ``ssd_scan_head`` / ``ssd_forward`` -- the Mamba2 mixer's selective scan
                        (C, ssd_oracle.c) on one chain and on a packed batch;
  * ``in_proj`` / ``gated_rmsnorm`` / ``out_proj`` -- the dense neighbours
                        of the forward in the layer (the projections around it
                        and the gated output norm), fp64;
  * ``product_form_final_state`` / ``chunked_wy_forward`` and their KDA
    counterparts ``kda_product_form_final_state`` / ``kda_chunked_forward``
    -- independent restatements of the recurrences used only to pin the token
    loops (numpy); ``ssd_quadratic_form`` / ``ssd_chunked_forward`` the same
    for the scan.

Every function cites the passage it follows; the readings taken where the
sources are silent are listed in the module docstring of gdn_oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_SRCS = [os.path.join(_HERE, "gdn_oracle.c"), os.path.join(_HERE, "ssd_oracle.c")]
_lock = threading.Lock()
_lib = None

L2_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile the oracle's C sources with gcc (OpenMP if the compiler has it)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(f) for f in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", "-o", tmp] + _SRCS + ["-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_gdn_forward.restype = I
            lib.oracle_gdn_forward.argtypes = [I] * 8 + [P] * 13 + [I]
            lib.oracle_kda_forward.restype = I
            lib.oracle_kda_forward.argtypes = [I] * 8 + [P] * 13 + [I]
            lib.oracle_conv_silu_seq.restype = None
            lib.oracle_conv_silu_seq.argtypes = [I, I, I, P, P, P, I, I, P]
            lib.oracle_gdn_rule_head.restype = None
            lib.oracle_gdn_rule_head.argtypes = [I, I, I, P, P, P, P, P,
                                                 ctypes.c_double, ctypes.c_double, P, P]
            lib.oracle_ssd_forward.restype = I
            lib.oracle_ssd_forward.argtypes = [I] * 8 + [P] * 13 + [I]
            lib.oracle_ssd_scan_head.restype = None
            lib.oracle_ssd_scan_head.argtypes = [I, I, I, P, P, P, P, ctypes.c_double,
                                                 ctypes.c_double, ctypes.c_double, P, P]
            lib.oracle_kda_rule_head.restype = None
            lib.oracle_kda_rule_head.argtypes = [I, I, I, P, P, P, P, P,
                                                 ctypes.c_double, P, P, P]
            _lib = lib
    return _lib


def _p(arr: np.ndarray):
    return arr.ctypes.data_as(ctypes.c_void_p)


def _f64(t) -> np.ndarray:
    """CPU tensor or array (fp32/bf16/fp64) -> contiguous fp64 numpy."""
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        if str(t.dtype) == "torch.bfloat16":
            t = t.float()
        t = t.numpy()
    return np.ascontiguousarray(t, dtype=np.float64)


# ---------------------------------------------------------------------------
# Elementary steps, exposed for the pins.

def conv_silu_seq(x, tail, w, ch0=0, nch=None):
    """Varlen causal depthwise conv1d + SiLU of one sequence continued from its
    conv state ("Continuous batching for linear attention layers": a varlen
    causal convolution continues every sequence from its own conv state).
    x: [L][C], tail: [K-1][C], w: [C][K] -> [L][nch] fp64."""
    x, tail, w = _f64(x), _f64(tail), _f64(w)
    L, C = x.shape
    K = w.shape[1]
    nch = C - ch0 if nch is None else nch
    y = np.zeros((L, nch))
    _load().oracle_conv_silu_seq(L, C, K, _p(x), _p(tail), _p(w), ch0, nch, _p(y))
    return y


def gdn_rule_head(q, k, v, a, b, A_log, dt_bias, S0):
    """Gated delta rule over one chain, token by token (Gated Delta Networks,
    the gated delta rule; normalisations and gates as stated in gdn_oracle.c).
    q,k: [L][dk] raw, v: [L][dv], a,b: [L], S0: [dv][dk] -> (o [L][dv], S_L)."""
    q, k, v, a, b = (_f64(t) for t in (q, k, v, a, b))
    S = _f64(S0).copy()
    L, dk = q.shape
    dv = v.shape[1]
    o = np.zeros((L, dv))
    _load().oracle_gdn_rule_head(L, dk, dv, _p(q), _p(k), _p(v), _p(a), _p(b),
                                 float(A_log), float(dt_bias), _p(S), _p(o))
    return o, S


def kda_rule_head(q, k, v, a, b, A_log, dt_bias, S0):
    """KDA rule over one chain, token by token (Kimi Linear, the KDA
    recurrence: the gated delta rule with one decay per key channel).
    q,k: [L][dk] raw, v: [L][dv], a: [L][dk], b: [L], dt_bias: [dk],
    S0: [dv][dk] -> (o [L][dv], S_L)."""
    q, k, v, a, b, dt_bias = (_f64(t) for t in (q, k, v, a, b, dt_bias))
    S = _f64(S0).copy()
    L, dk = q.shape
    dv = v.shape[1]
    if a.shape != (L, dk) or dt_bias.shape != (dk,):
        raise ValueError("per-channel gates: a [L][dk], dt_bias [dk]")
    o = np.zeros((L, dv))
    _load().oracle_kda_rule_head(L, dk, dv, _p(q), _p(k), _p(v), _p(a), _p(b),
                                 float(A_log), _p(dt_bias), _p(S), _p(o))
    return o, S


def ssd_scan_head(x, B, C, dt, A_log, dt_bias, Dskip, h0):
    """Mamba2 selective scan over one chain, token by token (Transformers are
    SSMs, the SSD recurrence; see ssd_oracle.c).  x: [L][P], B, C: [L][N],
    dt: [L] raw, h0: [P][N] -> (y [L][P], h_L)."""
    x, B, C, dt = (_f64(t) for t in (x, B, C, dt))
    h = _f64(h0).copy()
    L, P = x.shape
    N = B.shape[1]
    y = np.zeros((L, P))
    _load().oracle_ssd_scan_head(L, P, N, _p(x), _p(B), _p(C), _p(dt), float(A_log),
                                 float(dt_bias), float(Dskip), _p(h), _p(y))
    return y, h


# ---------------------------------------------------------------------------
# Bad-input rules.

ERR_SEQLENS = 1 << 0
ERR_BLOCK_RANGE = 1 << 1
ERR_TRASH_WRITE = 1 << 2
ERR_DUPLICATE = 1 << 3


def data_errors(cu_seqlens, block_idx, num_blocks, T):
    """Which sequences are skipped, and the error flags raised.

    The pool gives a request one block for its whole life, never shared, and
    block 0 is the trash block that is only ever read ("Continuous batching for
    linear attention layers").  A sequence is active when its block index is
    >= 0 and its length > 0 (index < 0 is a padding entry, as graph padding
    produces in the engine's batch preparation).  Active sequences whose index
    is out of range, equal to 0, or shared with another active sequence are
    skipped and flagged; cu_seqlens that do not start at 0, decrease or do not
    end at T skip the whole batch.
    """
    cu = [int(v) for v in cu_seqlens]
    blk = [int(v) for v in block_idx]
    N = len(blk)
    flags = 0
    skip = [False] * N
    ok = cu[0] == 0 and cu[-1] == T and all(cu[i + 1] >= cu[i] for i in range(N))
    if not ok:
        return [True] * N, ERR_SEQLENS
    active = [blk[s] >= 0 and cu[s + 1] > cu[s] for s in range(N)]
    seen = {}
    for s in range(N):
        if not active[s]:
            continue
        if blk[s] >= num_blocks:
            skip[s] = True
            flags |= ERR_BLOCK_RANGE
        elif blk[s] == 0:
            skip[s] = True
            flags |= ERR_TRASH_WRITE
        else:
            seen.setdefault(blk[s], []).append(s)
    for b, ss in seen.items():
        if len(ss) > 1:
            flags |= ERR_DUPLICATE
            for s in ss:
                skip[s] = True
    return skip, flags


# ---------------------------------------------------------------------------
# The whole forward.

def forward(wl, nthreads: int = 0, out_init=None):
    """Run the packed forward of workload ``wl`` (see the generator module) in
    fp64, with the KDA rule when ``wl`` has one gate per key channel.
    Returns a dict with
      out        [T][Hv][dv] fp64 (rows of skipped sequences: ``out_init`` or NaN)
      conv_state [R][K-1][C] fp64 and rec_state [R][Hv][dk][dv] fp64 (k-major,
                 like the pool), for the workload's referenced blocks after the
                 call
      skip, flags, threads.
    """
    d = wl.dims
    T, N = wl.T, wl.N
    ref = [int(v) for v in wl.ref_blocks]
    pos = {b: i for i, b in enumerate(ref)}
    skip, flags = data_errors(wl.cu_seqlens, wl.block_idx, wl.num_blocks, T)
    blk_local = np.array([pos.get(int(b), -1) if not skip[s] else -1
                          for s, b in enumerate(wl.block_idx.tolist())], dtype=np.int32)
    x = _f64(wl.x)
    a = _f64(wl.a)
    b = _f64(wl.b)
    w = _f64(wl.conv_w)
    A_log = _f64(wl.A_log)
    dt_bias = _f64(wl.dt_bias)
    cu = np.ascontiguousarray(wl.cu_seqlens.numpy(), dtype=np.int32)
    has_past = np.ascontiguousarray(wl.has_past.numpy(), dtype=np.uint8)
    skip_arr = np.array(skip, dtype=np.uint8)
    conv = _f64(wl.conv_state)
    # pool orientation [k][v] -> the oracle's S[v][k]
    rec = np.ascontiguousarray(np.swapaxes(_f64(wl.rec_state), 2, 3))
    if out_init is None:
        out = np.full((T, d.Hv, d.dv), np.nan)
    else:
        out = _f64(out_init).reshape(T, d.Hv, d.dv).copy()
    if wl.channel_gate and (a.shape != (T, d.Hv, d.dk) or dt_bias.shape != (d.Hv, d.dk)):
        raise ValueError("per-channel gates: a [T][Hv][dk], dt_bias [Hv][dk]")
    run = _load().oracle_kda_forward if wl.channel_gate else _load().oracle_gdn_forward
    if flags & ERR_SEQLENS:
        used = 0
    else:
        used = run(
            T, N, d.Hk, d.Hv, d.dk, d.dv, d.K, len(ref),
            _p(x), _p(a), _p(b), _p(cu), _p(blk_local), _p(has_past), _p(skip_arr),
            _p(w), _p(A_log), _p(dt_bias), _p(conv), _p(rec), _p(out), int(nthreads))
    return {
        "out": out,
        "conv_state": conv,
        "rec_state": np.ascontiguousarray(np.swapaxes(rec, 2, 3)),
        "skip": skip,
        "flags": flags,
        "threads": used,
    }


def ssd_forward(wl, nthreads: int = 0, out_init=None):
    """Packed forward of a Mamba2 mixer workload (``synth.SsdWorkload``) in
    fp64, with the same skip rules as ``forward``.  Returns a dict with
    ``y`` [T][H][P], ``conv_state`` [R][K-1][C], ``ssm_state`` [R][H][P][N]
    (the referenced blocks after the call), ``skip``, ``flags``, ``threads``."""
    d = wl.dims
    T, Nseq = wl.T, wl.N
    ref = [int(v) for v in wl.ref_blocks]
    pos = {b: i for i, b in enumerate(ref)}
    skip, flags = data_errors(wl.cu_seqlens, wl.block_idx, wl.num_blocks, T)
    blk_local = np.array([pos.get(int(b), -1) if not skip[s] else -1
                          for s, b in enumerate(wl.block_idx.tolist())], dtype=np.int32)
    xbc, dt, w = _f64(wl.xbc), _f64(wl.dt), _f64(wl.conv_w)
    A_log, dt_bias, Dskip = _f64(wl.A_log), _f64(wl.dt_bias), _f64(wl.D)
    cu = np.ascontiguousarray(wl.cu_seqlens.numpy(), dtype=np.int32)
    has_past = np.ascontiguousarray(wl.has_past.numpy(), dtype=np.uint8)
    skip_arr = np.array(skip, dtype=np.uint8)
    conv = _f64(wl.conv_state)
    ssm = _f64(wl.ssm_state).copy()
    if out_init is None:
        y = np.full((T, d.H, d.P), np.nan)
    else:
        y = _f64(out_init).reshape(T, d.H, d.P).copy()
    used = 0
    if not flags & ERR_SEQLENS:
        used = _load().oracle_ssd_forward(
            T, Nseq, d.H, d.P, d.N, d.G, d.K, len(ref), _p(xbc), _p(dt), _p(cu), _p(blk_local),
            _p(has_past), _p(skip_arr), _p(w), _p(A_log), _p(dt_bias), _p(Dskip), _p(conv),
            _p(ssm), _p(y), int(nthreads))
    return {"y": y, "conv_state": conv, "ssm_state": ssm, "skip": skip, "flags": flags,
            "threads": used}


# ---------------------------------------------------------------------------
# Pool byte layout as the boundary states it.

def _roundup(v, m):
    return (v + m - 1) // m * m


def pool_layout(num_blocks, num_layers, Hk, Hv, dk, dv, K, act_bytes, block_align=0):
    """Byte layout of the state pool.

    The allocator packs the declared per-request states of a layer into one
    block, each state on a 128-byte boundary ("Continuous batching for linear
    attention layers", the commit that makes the layers declare their states).
    Here: conv state [K-1][C] in the activation dtype at offset 0, recurrent
    state [Hv][dk][dv] fp32 at the next 128-byte boundary, block stride rounded
    up to max(128, block_align); block b of layer l starts at
    (l * num_blocks + b) * stride.
    """
    C = 2 * Hk * dk + Hv * dv
    conv_bytes = (K - 1) * C * act_bytes
    rec_off = _roundup(conv_bytes, 128)
    rec_bytes = Hv * dk * dv * 4
    stride = _roundup(rec_off + rec_bytes, max(128, block_align))
    return {"stride": stride, "conv_off": 0, "conv_bytes": conv_bytes, "rec_off": rec_off,
            "rec_bytes": rec_bytes, "total": stride * num_blocks * num_layers}


def read_pool_states(pool_bytes: np.ndarray, layer, blocks, dims, num_blocks, num_layers,
                     block_align=0):
    """Decode the conv and recurrent sub-states of ``blocks`` from a pool byte
    image (uint8 array) with the layout above.  Returns fp64
    (conv [B][K-1][C], rec [B][Hv][dk][dv])."""
    act_bytes = 4 if dims.act == "f32" else 2
    lay = pool_layout(num_blocks, num_layers, dims.Hk, dims.Hv, dims.dk, dims.dv, dims.K,
                      act_bytes, block_align)
    C = dims.C
    convs, recs = [], []
    for blk in blocks:
        base = (layer * num_blocks + int(blk)) * lay["stride"]
        cb = pool_bytes[base: base + lay["conv_bytes"]]
        if act_bytes == 4:
            conv = cb.view(np.float32).astype(np.float64)
        else:
            conv = (cb.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        rb = pool_bytes[base + lay["rec_off"]: base + lay["rec_off"] + lay["rec_bytes"]]
        convs.append(conv.reshape(dims.K - 1, C))
        recs.append(rb.view(np.float32).astype(np.float64).reshape(dims.Hv, dims.dk, dims.dv))
    return np.stack(convs), np.stack(recs)


def ssd_pool_layout(num_blocks, num_layers, H, P, N, G, K, act_bytes, block_align=0):
    """Byte layout of a Mamba2 state pool: the same per-request block as the
    gated delta net's, with the mixer's two declared states each on a 128-byte
    boundary ("Continuous batching for linear attention layers", the commit
    that makes the layers declare their states): conv state [K-1][C]
    (C = H*P + 2*G*N, activation dtype) at 0, SSM state [H][P][N] fp32 at the
    next 128-byte boundary, stride rounded up to max(128, block_align)."""
    C = H * P + 2 * G * N
    conv_bytes = (K - 1) * C * act_bytes
    ssm_off = _roundup(conv_bytes, 128)
    ssm_bytes = H * P * N * 4
    stride = _roundup(ssm_off + ssm_bytes, max(128, block_align))
    return {"stride": stride, "conv_off": 0, "conv_bytes": conv_bytes, "ssm_off": ssm_off,
            "ssm_bytes": ssm_bytes, "total": stride * num_blocks * num_layers}


def read_ssd_pool_states(pool_bytes: np.ndarray, layer, blocks, dims, num_blocks, num_layers,
                         block_align=0):
    """Decode the conv and SSM sub-states of ``blocks`` from a Mamba2 pool byte
    image.  Returns fp64 (conv [B][K-1][C], ssm [B][H][P][N])."""
    act_bytes = 4 if dims.act == "f32" else 2
    lay = ssd_pool_layout(num_blocks, num_layers, dims.H, dims.P, dims.N, dims.G, dims.K,
                          act_bytes, block_align)
    convs, ssms = [], []
    for blk in blocks:
        base = (layer * num_blocks + int(blk)) * lay["stride"]
        cb = pool_bytes[base: base + lay["conv_bytes"]]
        if act_bytes == 4:
            conv = cb.view(np.float32).astype(np.float64)
        else:
            conv = (cb.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        sb = pool_bytes[base + lay["ssm_off"]: base + lay["ssm_off"] + lay["ssm_bytes"]]
        convs.append(conv.reshape(dims.K - 1, dims.C))
        ssms.append(sb.view(np.float32).astype(np.float64).reshape(dims.H, dims.P, dims.N))
    return np.stack(convs), np.stack(ssms)


# ---------------------------------------------------------------------------
# Independent restatements used only as pins (numpy, fp64).

def product_form_final_state(k, v, g, beta, S0):
    """Closed product form of the gated delta rule.  Writing the update as
    S_t = S_{t-1} M_t + beta_t v_t k_t^T with M_t = e^{g_t} (I - beta_t k_t k_t^T),
    unrolling gives
        S_L = S_0 M_1 ... M_L + sum_t beta_t v_t k_t^T M_{t+1} ... M_L.
    k: [L][dk] (normalised), v: [L][dv], g, beta: [L], S0: [dv][dk]."""
    L, dk = k.shape
    I = np.eye(dk)
    Ms = [np.exp(g[t]) * (I - beta[t] * np.outer(k[t], k[t])) for t in range(L)]
    suffix = [None] * (L + 1)
    suffix[L] = I
    for t in range(L - 1, -1, -1):
        suffix[t] = Ms[t] @ suffix[t + 1]
    S = S0 @ suffix[0]
    for t in range(L):
        S = S + beta[t] * np.outer(v[t], k[t]) @ suffix[t + 1]
    return S


def chunked_wy_forward(q, k, v, g, beta, S0, chunk=64):
    """Chunked (WY / UT-transform) evaluation of the same recurrence, fp64.

    Within a chunk with inclusive cumulative gate G_i, the per-token update
    vectors u_i (S_i = e^{G_i} S_0 + sum_{j<=i} e^{G_i-G_j} u_j k_j^T) solve
    (I + A) U = diag(beta) V - diag(beta e^G) K S_0^T with
    A_ij = beta_i e^{G_i-G_j} k_i.k_j (j < i); then
      O = diag(e^G) Q S_0^T + ((Q K^T) o M) U,  M_ij = e^{G_i-G_j} (j <= i),
      S_C = e^{G_C} S_0 + U^T diag(e^{G_C-G_j}) K.
    Only non-positive exponents appear.  q, k normalised [L][dk]; v [L][dv];
    S0 [dv][dk].  Returns (O [L][dv], S_L)."""
    L = q.shape[0]
    S = S0.copy()
    outs = []
    for c0 in range(0, L, chunk):
        Q, Kc, V = q[c0:c0 + chunk], k[c0:c0 + chunk], v[c0:c0 + chunk]
        gc, bc = g[c0:c0 + chunk], beta[c0:c0 + chunk]
        n = Q.shape[0]
        G = np.cumsum(gc)
        diff = G[:, None] - G[None, :]
        lower = np.tril(np.ones((n, n), dtype=bool), -1)
        A = np.where(lower, bc[:, None] * np.exp(np.where(lower, diff, 0.0)) * (Kc @ Kc.T), 0.0)
        Tm = np.linalg.inv(np.eye(n) + A)
        W = Tm @ (bc[:, None] * np.exp(G)[:, None] * Kc)
        U = Tm @ (bc[:, None] * V) - W @ S.T
        incl = np.tril(np.ones((n, n), dtype=bool))
        M = np.where(incl, np.exp(np.where(incl, diff, 0.0)), 0.0)
        O = np.exp(G)[:, None] * (Q @ S.T) + ((Q @ Kc.T) * M) @ U
        S = np.exp(G[-1]) * S + U.T @ (np.exp(G[-1] - G)[:, None] * Kc)
        outs.append(O)
    return np.concatenate(outs, axis=0), S


def kda_product_form_final_state(k, v, g, beta, S0):
    """Closed product form of the KDA rule.  The token update is
    S_t = S_{t-1} D_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T with
    D_t = Diag(e^{g_t}) (one decay per key channel), so with
    M_t = D_t (I - beta_t k_t k_t^T)
        S_L = S_0 M_1 ... M_L + sum_t beta_t v_t k_t^T M_{t+1} ... M_L.
    k: [L][dk] (normalised), v: [L][dv], g: [L][dk], beta: [L], S0: [dv][dk]."""
    L, dk = k.shape
    I = np.eye(dk)
    Ms = [np.diag(np.exp(g[t])) @ (I - beta[t] * np.outer(k[t], k[t])) for t in range(L)]
    suffix = [None] * (L + 1)
    suffix[L] = I
    for t in range(L - 1, -1, -1):
        suffix[t] = Ms[t] @ suffix[t + 1]
    S = S0 @ suffix[0]
    for t in range(L):
        S = S + beta[t] * np.outer(v[t], k[t]) @ suffix[t + 1]
    return S


def kda_chunked_forward(q, k, v, g, beta, S0, chunk=64):
    """Chunked (WY / UT-transform) evaluation of the KDA rule, fp64.

    With Gam_i = sum_{s<=i} g_s (a vector per token, cumulative within the
    chunk), the state after token i of a chunk is
        S_i = S_0 Diag(e^{Gam_i}) + sum_{j<=i} u_j (k_j o e^{Gam_i - Gam_j})^T,
    and the update vectors solve
        (I + A) U = diag(beta) V - diag(beta) (K o e^{Gam}) S_0^T,
        A_ij = beta_i sum_c k_ic k_jc e^{Gam_ic - Gam_jc}   (j < i);
    then
        O = (Q o e^{Gam}) S_0^T + P U,  P_ij = sum_c q_ic k_jc e^{Gam_ic - Gam_jc} (j <= i),
        S_C = S_0 Diag(e^{Gam_C}) + U^T (K o e^{Gam_C - Gam}).
    Every pairwise factor is formed directly, so only non-positive exponents
    appear.  q, k normalised [L][dk]; v [L][dv]; g [L][dk]; beta [L];
    S0 [dv][dk].  Returns (O [L][dv], S_L)."""
    L = q.shape[0]
    S = S0.copy()
    outs = []
    for c0 in range(0, L, chunk):
        Q, Kc, V = q[c0:c0 + chunk], k[c0:c0 + chunk], v[c0:c0 + chunk]
        gc, bc = g[c0:c0 + chunk], beta[c0:c0 + chunk]
        n = Q.shape[0]
        Gam = np.cumsum(gc, axis=0)  # [n][dk]
        A = np.zeros((n, n))
        P = np.zeros((n, n))
        for i in range(n):
            for j in range(i + 1):
                f = np.exp(Gam[i] - Gam[j])
                P[i, j] = np.sum(Q[i] * Kc[j] * f)
                if j < i:
                    A[i, j] = bc[i] * np.sum(Kc[i] * Kc[j] * f)
        Tm = np.linalg.inv(np.eye(n) + A)
        U = Tm @ (bc[:, None] * V) - Tm @ (bc[:, None] * (Kc * np.exp(Gam))) @ S.T
        O = (Q * np.exp(Gam)) @ S.T + P @ U
        S = S * np.exp(Gam[-1])[None, :] + U.T @ (Kc * np.exp(Gam[-1] - Gam))
        outs.append(O)
    return np.concatenate(outs, axis=0), S


def ssd_quadratic_form(x, B, C, dt, a_log_decay, Dskip, h0):
    """The scan written as one matrix product (the "attention" side of state
    space duality).  With per-token time steps dt_t (after softplus), decays
    log a_t = a_log_decay[t] and the segment sums
    Lam_ts = sum_{r=s+1..t} log a_r (s <= t):
        y_t = sum_{s<=t} e^{Lam_ts} (C_t . B_s) dt_s x_s
              + e^{sum_{r<=t} log a_r} h_0 C_t + D x_t,
        h_L = e^{sum_r log a_r} h_0 + sum_s e^{Lam_Ls} dt_s x_s B_s^T.
    x: [L][P], B, C: [L][N], dt, a_log_decay: [L], h0: [P][N]."""
    L = x.shape[0]
    cum = np.cumsum(a_log_decay)
    seg = cum[:, None] - cum[None, :]  # Lam_ts for s <= t
    causal = np.tril(np.ones((L, L), dtype=bool))
    M = np.where(causal, np.exp(np.where(causal, seg, 0.0)), 0.0) * (C @ B.T)
    y = M @ (dt[:, None] * x) + np.exp(cum)[:, None] * (C @ h0.T) + Dskip * x
    h = np.exp(cum[-1]) * h0 + (np.exp(cum[-1] - cum)[:, None] * dt[:, None] * x).T @ B
    return y, h


def ssd_chunked_forward(x, B, C, dt, a_log_decay, Dskip, h0, chunk=64):
    """Chunked evaluation of the scan: inside a chunk the quadratic form, and
    between chunks only the state is passed,
        h_end = e^{A_c} h_start + sum_s e^{A_c - A_s} dt_s x_s B_s^T
    (A_s the within-chunk cumulative log decay).  Same arguments as
    ``ssd_quadratic_form``."""
    h = h0.copy()
    ys = []
    for c0 in range(0, x.shape[0], chunk):
        sl = slice(c0, c0 + chunk)
        y, h = ssd_quadratic_form(x[sl], B[sl], C[sl], dt[sl], a_log_decay[sl], Dskip, h)
        ys.append(y)
    return np.concatenate(ys, axis=0), h


# ---------------------------------------------------------------------------
# The dense neighbours of the forward in a hybrid model's gated-delta-net layer
# (the pages name the layer; its projections are the plainest reading of what
# surrounds the varlen forward).  A matmul is the library primitive here.

def in_proj(hidden, w_qkv, w_z, w_b, w_a):
    """Input projection, token by token: x_qkv = W_qkv h, z = W_z h, b = W_b h,
    a = W_a h (weights [out][in]).  fp64.  Returns (x_qkv, z, b, a) as
    [T][C], [T][Hv*d_v], [T][Hv], [T][Hv]."""
    h = _f64(hidden)
    return tuple(h @ _f64(w).T for w in (w_qkv, w_z, w_b, w_a))


def gated_rmsnorm(o, z, norm_w, eps):
    """Gated RMS norm of the layer's output, per token and v-head over its d_v
    channels: o / sqrt(mean(o^2) + eps) * norm_w * silu(z), silu(z) =
    z / (1 + e^{-z}).  o, z: [T][Hv][d_v]; norm_w: [d_v].  fp64."""
    o = _f64(o)
    z = _f64(z)
    rs = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    with np.errstate(over="ignore"):
        silu = z / (1.0 + np.exp(-z))
    return o * rs * _f64(norm_w) * silu


def out_proj(o_norm, w_out):
    """Output projection, token by token: y = W_out o_norm (o_norm flattened over
    its heads; W_out [d_model][Hv*d_v]).  fp64."""
    o = _f64(o_norm)
    return o.reshape(o.shape[0], -1) @ _f64(w_out).T

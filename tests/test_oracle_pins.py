"""Pins of the fp64 oracle against facts other than itself (CPU only).

Each test checks the oracle against a library routine, a closed form, an
invariant the method fixes, or an independent restatement, chosen so that a
plausible slip (a dropped term, a wrong sign, a transposed operand, a wrong
head map, a wrong tap orientation) fails at least one of them.
"""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from continuous_linear_attention_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------
# Convolution: torch's depthwise conv1d is the library special case.

@pytest.mark.parametrize("L,C,K", [(9, 12, 4), (1, 5, 4), (2, 7, 3), (30, 16, 2)])
def test_conv_no_past_equals_torch_conv1d(L, C, K):
    rng = _rng(L * 100 + C)
    x = rng.standard_normal((L, C))
    w = rng.standard_normal((C, K)) * 0.5
    tail = np.zeros((K - 1, C))
    got = oracle.conv_silu_seq(x, tail, w)
    xt = torch.from_numpy(x).T[None]  # [1][C][L]
    ref = F.conv1d(xt, torch.from_numpy(w)[:, None, :], groups=C, padding=K - 1)[0, :, :L]
    ref = F.silu(ref).T.numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("L", [1, 2, 3, 11])
def test_conv_with_past_equals_conv_over_concatenation(L):
    C, K = 10, 4
    rng = _rng(L)
    x = rng.standard_normal((L, C))
    tail = rng.standard_normal((K - 1, C))
    w = rng.standard_normal((C, K))
    got = oracle.conv_silu_seq(x, tail, w)
    cat = torch.from_numpy(np.concatenate([tail, x])).T[None]
    ref = F.silu(F.conv1d(cat, torch.from_numpy(w)[:, None, :], groups=C)[0]).T.numpy()
    assert ref.shape == (L, C)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_conv_channel_subset_matches_full():
    rng = _rng(7)
    x = rng.standard_normal((6, 20))
    tail = rng.standard_normal((3, 20))
    w = rng.standard_normal((20, 4))
    full = oracle.conv_silu_seq(x, tail, w)
    np.testing.assert_array_equal(oracle.conv_silu_seq(x, tail, w, 5, 7), full[:, 5:12])


# ----------------------------------------------------------------------------
# Recurrence: the closed product form and the chunked WY form.

def _normalised_inputs(L, dk, dv, seed, big=1e4, slow=False):
    """Raw q, k scaled so that the L2-norm epsilon is negligible (relative
    1e-14): then the library's F.normalize gives the normalised vectors."""
    rng = _rng(seed)
    q = rng.standard_normal((L, dk)) * big
    k = rng.standard_normal((L, dk)) * big
    v = rng.standard_normal((L, dv))
    a = rng.standard_normal(L)
    b = rng.standard_normal(L)
    A_log = math.log(rng.uniform(0.01, 0.1) if slow else rng.uniform(1, 16))
    dt_bias = -8.0 if slow else float(rng.standard_normal() * 0.1)
    qn = F.normalize(torch.from_numpy(q), dim=-1).numpy() / math.sqrt(dk)
    kn = F.normalize(torch.from_numpy(k), dim=-1).numpy()
    g = (-math.exp(A_log) * F.softplus(torch.from_numpy(a + dt_bias))).numpy()
    beta = torch.sigmoid(torch.from_numpy(b)).numpy()
    return dict(q=q, k=k, v=v, a=a, b=b, A_log=A_log, dt_bias=dt_bias,
                qn=qn, kn=kn, g=g, beta=beta)


@pytest.mark.parametrize("slow", [False, True])
def test_rule_matches_closed_product_form(slow):
    L, dk, dv = 7, 5, 3
    d = _normalised_inputs(L, dk, dv, 11, slow=slow)
    S0 = _rng(12).standard_normal((dv, dk)) * 0.3
    o, S = oracle.gdn_rule_head(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"],
                                d["dt_bias"], S0)
    for t in range(L):
        St = oracle.product_form_final_state(d["kn"][:t + 1], d["v"][:t + 1], d["g"][:t + 1],
                                             d["beta"][:t + 1], S0)
        np.testing.assert_allclose(o[t], St @ d["qn"][t], rtol=0, atol=1e-12)
    S_ref = oracle.product_form_final_state(d["kn"], d["v"], d["g"], d["beta"], S0)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("L", [1, 63, 64, 65, 150])
def test_rule_matches_chunked_wy_form(L):
    dk, dv = 16, 12
    d = _normalised_inputs(L, dk, dv, L, slow=True)
    S0 = _rng(L + 1).standard_normal((dv, dk)) * 0.1
    o, S = oracle.gdn_rule_head(d["q"], d["k"], d["v"], d["a"], d["b"], d["A_log"],
                                d["dt_bias"], S0)
    o2, S2 = oracle.chunked_wy_forward(d["qn"], d["kn"], d["v"], d["g"], d["beta"], S0)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-10)
    np.testing.assert_allclose(S, S2, rtol=0, atol=1e-10)


def test_beta_zero_only_decays():
    """b = -1000 makes sigmoid exactly 0: S_t = e^{g_t} S_{t-1}, o_t = S_t q_t."""
    L, dk, dv = 6, 8, 4
    d = _normalised_inputs(L, dk, dv, 21)
    b = np.full(L, -1000.0)
    S0 = _rng(22).standard_normal((dv, dk))
    o, S = oracle.gdn_rule_head(d["q"], d["k"], d["v"], d["a"], b, d["A_log"], d["dt_bias"], S0)
    G = np.cumsum(d["g"])
    for t in range(L):
        np.testing.assert_allclose(o[t], math.exp(G[t]) * (S0 @ d["qn"][t]), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(S, math.exp(G[-1]) * S0, rtol=1e-12)


def test_huge_gate_forgets_state():
    """a + dt_bias = 800: softplus = 800 (its large-argument branch), e^g
    underflows to exactly 0, so S_1 = beta v k^T regardless of S_0."""
    dk, dv = 4, 3
    rng = _rng(5)
    q = rng.standard_normal((1, dk)) * 1e4
    k = rng.standard_normal((1, dk)) * 1e4
    v = rng.standard_normal((1, dv))
    S0 = rng.standard_normal((dv, dk))
    o, S = oracle.gdn_rule_head(q, k, v, [800.0], [0.3], 0.0, 0.0, S0)
    kn = F.normalize(torch.from_numpy(k[0]), dim=0).numpy()
    qn = F.normalize(torch.from_numpy(q[0]), dim=0).numpy() / 2.0
    beta = 1.0 / (1.0 + math.exp(-0.3))
    np.testing.assert_allclose(S, beta * np.outer(v[0], kn), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(o[0], S @ qn, rtol=1e-13, atol=1e-15)


# ----------------------------------------------------------------------------
# Whole forward: closed form with orthonormal keys (golden fixture), head map,
# state orientation in the pool.

def _fixture_workload(fx):
    dims = synth.Dims(Hk=fx["Hk"], Hv=fx["Hv"], dk=fx["dk"], dv=fx["dv"], K=fx["K"], act="f32")
    C = dims.C
    L = fx["L"]
    x = np.zeros((L, C), dtype=np.float32)
    a = np.full((L, dims.Hv), fx["a_all"], dtype=np.float32)
    b = np.full((L, dims.Hv), fx["b_write"], dtype=np.float32)
    b[L - 1, :] = fx["b_last"]
    for t in range(L):
        for kh in range(dims.Hk):
            x[t, kh * dims.dk + fx["q_index"][t]] = fx["qk_scale"]
            x[t, dims.Hk * dims.dk + kh * dims.dk + fx["key_index"][kh][t]] = fx["qk_scale"]
        for h in range(dims.Hv):
            x[t, 2 * dims.Hk * dims.dk + h * dims.dv:2 * dims.Hk * dims.dk + (h + 1) * dims.dv] = \
                fx["v_rows"][h][t]
    w = np.zeros((C, dims.K), dtype=np.float32)
    w[:, dims.K - 1] = 1.0
    wl = synth.make_workload("golden", dims, [L], [0], 2, 0, block_idx=[1])
    return dataclasses.replace(
        wl, x=torch.from_numpy(x), a=torch.from_numpy(a), b=torch.from_numpy(b),
        conv_w=torch.from_numpy(w), A_log=torch.zeros(dims.Hv), dt_bias=torch.zeros(dims.Hv))


def test_golden_orthonormal_keys():
    with open(os.path.join(GOLDEN, "orthonormal_keys.json")) as f:
        fx = json.load(f)
    wl = _fixture_workload(fx)
    res = oracle.forward(wl)
    d = wl.dims
    out = res["out"]
    for h in range(d.Hv):
        np.testing.assert_allclose(out[fx["L"] - 1, h], fx["expected_last_out"][h], rtol=1e-12)
    blk = [int(v) for v in wl.ref_blocks].index(1)
    rec = res["rec_state"][blk]  # [Hv][dk][dv], element S[v][k] at [h][k][v]
    for h in range(d.Hv):
        np.testing.assert_allclose(rec[h], fx["expected_state_kv"][h], rtol=1e-12, atol=1e-12)
    # new conv tail = the last K-1 input rows
    np.testing.assert_array_equal(res["conv_state"][blk], wl.x.numpy()[-(d.K - 1):])


# ----------------------------------------------------------------------------
# Invariants the pages fix.

def _slice_workload(wl, seqs):
    """The sub-batch made of sequences ``seqs`` of ``wl`` (same pool)."""
    cu = wl.cu_seqlens.tolist()
    rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs]).astype(np.int64)
    lens = [cu[s + 1] - cu[s] for s in seqs]
    ncu = np.zeros(len(seqs) + 1, dtype=np.int32)
    ncu[1:] = np.cumsum(lens)
    idx = torch.from_numpy(rows)
    return dataclasses.replace(
        wl, x=wl.x[idx], a=wl.a[idx], b=wl.b[idx], cu_seqlens=torch.from_numpy(ncu),
        block_idx=wl.block_idx[list(seqs)], has_past=wl.has_past[list(seqs)])


def test_packed_equals_each_alone():
    wl = synth.tiny_packed(0)
    full = oracle.forward(wl)
    cu = wl.cu_seqlens.tolist()
    for s in range(wl.N):
        one = oracle.forward(_slice_workload(wl, [s]))
        np.testing.assert_array_equal(full["out"][cu[s]:cu[s + 1]], one["out"])
        r = [int(v) for v in wl.ref_blocks].index(int(wl.block_idx[s]))
        np.testing.assert_array_equal(full["rec_state"][r], one["rec_state"][r])
        np.testing.assert_array_equal(full["conv_state"][r], one["conv_state"][r])


def test_no_past_reads_only_the_trash_block():
    wl = synth.tiny_packed(0)
    res = oracle.forward(wl)
    assert np.isfinite(res["out"]).all()  # the NaN-filled write blocks were never read
    assert not res["conv_state"][0].any() and not res["rec_state"][0].any()
    # equals a run where the same sequences have a past made of zeros
    z = dataclasses.replace(wl, has_past=torch.ones_like(wl.has_past),
                            conv_state=wl.conv_state.clone(), rec_state=wl.rec_state.clone())
    ref = [int(v) for v in wl.ref_blocks]
    for s in range(wl.N):
        if not wl.has_past[s]:
            r = ref.index(int(wl.block_idx[s]))
            z.conv_state[r] = 0
            z.rec_state[r] = 0
    res2 = oracle.forward(z)
    np.testing.assert_array_equal(res["out"], res2["out"])
    np.testing.assert_array_equal(res["rec_state"], res2["rec_state"])


@pytest.mark.parametrize("cut", [1, 2, 3, 17, 63, 64, 65])
def test_split_anywhere_equals_one_pass(cut):
    dims = synth.Dims(Hk=1, Hv=2, dk=8, dv=8, K=4, act="f32")
    L = 80
    whole = synth.make_workload("w", dims, [L], [0], 2, 3, block_idx=[1], slow_decay=True)
    one = oracle.forward(whole)
    first = _slice_rows(whole, 0, cut, past=0)
    r1 = oracle.forward(first)
    # the continuation starts from the first part's fp64 states, unrounded
    second = dataclasses.replace(_slice_rows(whole, cut, L, past=1),
                                 conv_state=torch.from_numpy(r1["conv_state"]),
                                 rec_state=torch.from_numpy(r1["rec_state"]))
    r2 = oracle.forward(second)
    np.testing.assert_allclose(np.concatenate([r1["out"], r2["out"]]), one["out"],
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(r2["rec_state"], one["rec_state"], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(r2["conv_state"], one["conv_state"])


def _slice_rows(wl, lo, hi, past):
    return dataclasses.replace(
        wl, x=wl.x[lo:hi], a=wl.a[lo:hi], b=wl.b[lo:hi],
        cu_seqlens=torch.tensor([0, hi - lo], dtype=torch.int32),
        has_past=torch.tensor([past], dtype=torch.uint8))


def test_tail_update_short_sequences_shift():
    """len < K-1: the new tail is the old tail shifted up by len rows."""
    dims = synth.Dims(Hk=1, Hv=1, dk=4, dv=4, K=4, act="f32")
    wl = synth.make_workload("t", dims, [1, 2], [1, 1], 4, 9, block_idx=[2, 3])
    res = oracle.forward(wl)
    ref = [int(v) for v in wl.ref_blocks]
    x = wl.x.numpy()
    for s, (lo, hi) in enumerate([(0, 1), (1, 3)]):
        r = ref.index(int(wl.block_idx[s]))
        old = wl.conv_state[r].numpy()
        expect = np.concatenate([old, x[lo:hi]])[-3:]
        np.testing.assert_array_equal(res["conv_state"][r], expect)


def test_skipped_sequences_leave_out_and_blocks_untouched():
    dims = synth.Dims(Hk=1, Hv=2, dk=4, dv=4, K=4, act="f32")
    wl = synth.make_workload("s", dims, [3, 2, 0, 4], [1, 1, 0, 1], 6, 4,
                             block_idx=[2, -1, 3, 4])
    init = np.full((wl.T, dims.Hv, dims.dv), 7.25)
    res = oracle.forward(wl, out_init=init)
    assert (res["out"][3:5] == 7.25).all()  # padding sequence rows untouched
    ref = [int(v) for v in wl.ref_blocks]
    r3 = ref.index(3)  # zero-length sequence: its block keeps its contents (NaN)
    assert np.isnan(res["rec_state"][r3]).all()


def test_data_error_rules():
    cu = [0, 2, 3, 5, 5]
    skip, flags = oracle.data_errors(cu, [1, 1, 4, 9], 8, 5)
    assert flags == oracle.ERR_DUPLICATE and skip == [True, True, False, False]
    skip, flags = oracle.data_errors(cu, [0, 2, 9, 3], 8, 5)
    assert flags == oracle.ERR_TRASH_WRITE | oracle.ERR_BLOCK_RANGE
    assert skip == [True, False, True, False]
    skip, flags = oracle.data_errors([0, 3, 2], [1, 2], 8, 2)
    assert flags == oracle.ERR_SEQLENS and skip == [True, True]
    skip, flags = oracle.data_errors([0, 2, 4], [1, 2], 8, 5)
    assert flags == oracle.ERR_SEQLENS


def test_pool_layout_formula():
    lay = oracle.pool_layout(512, 1, 16, 32, 128, 128, 4, 2)
    assert lay["conv_bytes"] == 3 * 8192 * 2 and lay["rec_off"] == 49152
    assert lay["stride"] == 49152 + 32 * 128 * 128 * 4
    lay = oracle.pool_layout(8, 1, 2, 4, 32, 32, 4, 4)
    assert (lay["conv_bytes"], lay["rec_off"], lay["stride"]) == (3072, 3072, 3072 + 16384)
    lay = oracle.pool_layout(4, 2, 1, 1, 8, 8, 4, 2, block_align=4096)
    assert lay["conv_bytes"] == 144 and lay["rec_off"] == 256 and lay["stride"] == 4096
    assert lay["total"] == 4096 * 8


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_read_pool_states_round_trips_a_hand_built_image(act):
    """The pool decoder reads back a byte image written element by element in
    the stated layout ("Continuous batching for linear attention layers": one
    block per request, each declared state on a 128-byte boundary): conv state
    [K-1][C] at offset 0, oldest row first; recurrent state at the next
    128-byte boundary with S_h[v][k] at ((h*d_k + k)*d_v + v)*4; block b of
    layer l at (l*num_blocks + b)*stride.  The offsets below are worked out
    by hand for Hk = 1, Hv = 2, d = 8, K = 3 (C = 2*8 + 2*8 = 32 channels):
    bf16 conv 2*32*2 = 128 bytes -> rec at 128, rec 2*8*8*4 = 512 bytes,
    block 640 -> stride 1024 with a 1024-byte alignment; f32 conv 256 bytes ->
    rec at 256, block 768 -> stride 1024.  Every value encodes its own indices
    (exact in bf16 and fp32), so a transposed state, a swapped row order or a
    wrong block or layer offset reads a different number."""
    import struct
    dims = synth.Dims(Hk=1, Hv=2, dk=8, dv=8, K=3, act=act)
    nb, nl, align = 3, 2, 1024
    stride, rec_off = 1024, (128 if act == "bf16" else 256)
    img = bytearray(stride * nb * nl)

    def conv_val(l, b, r, c):
        return float(l * 128 + b * 64 + r * 32 + c - 200)

    def rec_val(l, b, h, v, k):
        return l * 10000.0 + b * 1000.0 + h * 100.0 + v * 10.0 + k + 0.25

    for l in range(nl):
        for b in range(nb):
            base = (l * nb + b) * stride
            for r in range(2):
                for c in range(32):
                    val = conv_val(l, b, r, c)
                    if act == "bf16":
                        raw = struct.unpack("<I", struct.pack("<f", val))[0] >> 16
                        struct.pack_into("<H", img, base + (r * 32 + c) * 2, raw)
                    else:
                        struct.pack_into("<f", img, base + (r * 32 + c) * 4, val)
            for h in range(2):
                for k in range(8):
                    for v in range(8):
                        off = base + rec_off + ((h * 8 + k) * 8 + v) * 4
                        struct.pack_into("<f", img, off, rec_val(l, b, h, v, k))
    pool = np.frombuffer(bytes(img), dtype=np.uint8)
    for layer in range(nl):
        conv, rec = oracle.read_pool_states(pool, layer, [2, 0, 1], dims, nb, nl,
                                            block_align=align)
        for i, b in enumerate([2, 0, 1]):
            for r in range(2):
                for c in range(32):
                    assert conv[i, r, c] == conv_val(layer, b, r, c)
            for h in range(2):
                for k in range(8):
                    for v in range(8):
                        # rec is returned as [h][k][v] = S_h[v][k]
                        assert rec[i, h, k, v] == rec_val(layer, b, h, v, k)

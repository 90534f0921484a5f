"""Pins of the oracle's per-channel-decay rule (KDA) against facts other than
itself (CPU only).

The rule differs from the gated delta rule only in its gate: one decay per
key channel.  So it is pinned by its reduction to the already pinned scalar
rule when every channel has the same gate, by the closed product form with
diagonal decays (which fixes the side the decay multiplies), by the chunked
WY form a tensor-core kernel would evaluate, by exact closed forms with
beta = 0, and by the invariants of the packed forward (packed = alone,
split = whole, no past reads only the trash block) on per-channel-gate
workloads.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import kernel_forms
import oracle
from continuous_linear_attention_gb300 import synth


def _rng(seed):
    return np.random.default_rng(seed)


def _inputs(L, dk, dv, seed, slow=False, big=1e4):
    """Raw q, k scaled so that the L2-norm epsilon is negligible; gates from
    torch's softplus and sigmoid (library routines)."""
    rng = _rng(seed)
    q = rng.standard_normal((L, dk)) * big
    k = rng.standard_normal((L, dk)) * big
    v = rng.standard_normal((L, dv))
    a = rng.standard_normal((L, dk))
    b = rng.standard_normal(L)
    A_log = math.log(rng.uniform(0.01, 0.1) if slow else rng.uniform(1, 16))
    dt_bias = np.full(dk, -8.0) if slow else rng.standard_normal(dk) * 0.1
    qn = F.normalize(torch.from_numpy(q), dim=-1).numpy() / math.sqrt(dk)
    kn = F.normalize(torch.from_numpy(k), dim=-1).numpy()
    g = (-math.exp(A_log) * F.softplus(torch.from_numpy(a + dt_bias[None, :]))).numpy()
    beta = torch.sigmoid(torch.from_numpy(b)).numpy()
    return dict(q=q, k=k, v=v, a=a, b=b, A_log=A_log, dt_bias=dt_bias,
                qn=qn, kn=kn, g=g, beta=beta)


def _run(d, S0, a=None, b=None):
    return oracle.kda_rule_head(d["q"], d["k"], d["v"], d["a"] if a is None else a,
                                d["b"] if b is None else b, d["A_log"], d["dt_bias"], S0)


# ----------------------------------------------------------------------------
# One chain.

@pytest.mark.parametrize("slow", [False, True])
def test_equal_channel_gates_reduce_to_the_scalar_rule(slow):
    """Every key channel with the same gate is the gated delta rule."""
    L, dk, dv = 9, 6, 5
    d = _inputs(L, dk, dv, 3, slow=slow)
    a1 = d["a"][:, 0]
    db = float(d["dt_bias"][0])
    S0 = _rng(4).standard_normal((dv, dk)) * 0.2
    o, S = oracle.kda_rule_head(d["q"], d["k"], d["v"], np.repeat(a1[:, None], dk, axis=1),
                                d["b"], d["A_log"], np.full(dk, db), S0)
    o_ref, S_ref = oracle.gdn_rule_head(d["q"], d["k"], d["v"], a1, d["b"], d["A_log"], db, S0)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-14)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-14)


@pytest.mark.parametrize("slow", [False, True])
def test_rule_matches_closed_product_form(slow):
    """S_L = S_0 M_1..M_L + sum_t beta_t v_t k_t^T M_{t+1}..M_L with
    M_t = Diag(e^{g_t}) (I - beta_t k_t k_t^T), and o_t = S_t q_t, at every
    token: a decay applied to the wrong side (rows, i.e. v, instead of key
    columns) or after the delta step fails here."""
    L, dk, dv = 7, 5, 3
    d = _inputs(L, dk, dv, 11, slow=slow)
    S0 = _rng(12).standard_normal((dv, dk)) * 0.3
    o, S = _run(d, S0)
    for t in range(L):
        St = oracle.kda_product_form_final_state(d["kn"][:t + 1], d["v"][:t + 1], d["g"][:t + 1],
                                                 d["beta"][:t + 1], S0)
        np.testing.assert_allclose(o[t], St @ d["qn"][t], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, oracle.kda_product_form_final_state(
        d["kn"], d["v"], d["g"], d["beta"], S0), rtol=0, atol=1e-12)


@pytest.mark.parametrize("L", [1, 17, 64, 65, 130])
def test_rule_matches_chunked_wy_form(L):
    dk, dv = 8, 6
    d = _inputs(L, dk, dv, 100 + L, slow=True)
    S0 = _rng(L).standard_normal((dv, dk)) * 0.1
    o, S = _run(d, S0)
    o2, S2 = oracle.kda_chunked_forward(d["qn"], d["kn"], d["v"], d["g"], d["beta"], S0)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-10)
    np.testing.assert_allclose(S, S2, rtol=0, atol=1e-10)


def test_chunked_form_with_fast_decay_and_a_short_chunk():
    """Default (fast) gates, chunk 16: the chunked form stays exact where
    whole-chunk exponent factors would overflow."""
    L, dk, dv = 40, 8, 4
    d = _inputs(L, dk, dv, 7)
    d["a"] = d["a"] + 3.0  # g about -3 .. -50 per token and channel
    d["g"] = (-math.exp(d["A_log"]) * F.softplus(torch.from_numpy(d["a"] + d["dt_bias"]))).numpy()
    S0 = _rng(8).standard_normal((dv, dk))
    o, S = _run(d, S0)
    o2, S2 = oracle.kda_chunked_forward(d["qn"], d["kn"], d["v"], d["g"], d["beta"], S0, chunk=16)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, S2, rtol=0, atol=1e-12)


def test_beta_zero_decays_each_key_channel_by_its_own_gate():
    """sigmoid(-1000) is exactly 0: S_t[v][c] = S_0[v][c] e^{sum_{s<=t} g_s[c]}
    and o_t = S_t q_t."""
    L, dk, dv = 6, 8, 4
    d = _inputs(L, dk, dv, 21, slow=True)
    S0 = _rng(22).standard_normal((dv, dk))
    o, S = _run(d, S0, b=np.full(L, -1000.0))
    Gam = np.cumsum(d["g"], axis=0)
    for t in range(L):
        np.testing.assert_allclose(o[t], (S0 * np.exp(Gam[t])[None, :]) @ d["qn"][t], rtol=1e-12)
    np.testing.assert_allclose(S, S0 * np.exp(Gam[-1])[None, :], rtol=1e-12)


def test_channel_selective_forgetting_is_exact():
    """A gate of 800 on some key channels zeroes exactly those state columns
    (e^{-800 e^0} underflows to 0); a gate of -1e4 on the others keeps them
    exactly (softplus(-1e4) = 0)."""
    dk, dv = 6, 3
    rng = _rng(5)
    q = rng.standard_normal((1, dk))
    k = rng.standard_normal((1, dk))
    v = rng.standard_normal((1, dv))
    S0 = rng.standard_normal((dv, dk))
    forget = np.array([True, False, True, False, False, True])
    a = np.where(forget, 800.0, -1e4)[None, :]
    o, S = oracle.kda_rule_head(q, k, v, a, [-1000.0], 0.0, np.zeros(dk), S0)
    np.testing.assert_array_equal(S[:, forget], 0.0)
    np.testing.assert_array_equal(S[:, ~forget], S0[:, ~forget])


def test_one_token_from_zero_state_is_the_outer_product():
    """From S_0 = 0 the decay has nothing to act on: S_1 = beta v k^T."""
    dk, dv = 5, 4
    d = _inputs(1, dk, dv, 31)
    o, S = _run(d, np.zeros((dv, dk)))
    np.testing.assert_allclose(S, d["beta"][0] * np.outer(d["v"][0], d["kn"][0]), rtol=1e-13)
    np.testing.assert_allclose(o[0], S @ d["qn"][0], rtol=1e-13)


# ----------------------------------------------------------------------------
# Whole packed forward with per-channel gates.

KDA_TINY = synth.Dims(Hk=2, Hv=4, dk=8, dv=8, K=4, act="f32")


def _kda_workload(seed=0, seqlens=(5, 1, 9), past=(0, 1, 0), slow=False, dims=KDA_TINY):
    return synth.make_workload("kda_tiny", dims, list(seqlens), list(past), 8, seed,
                               slow_decay=slow, channel_gate=True)


def test_forward_reads_the_gates_in_their_stated_layout():
    """Per chain, the forward equals the single-chain rule fed with the
    conv+SiLU rows of its heads and the gate rows a[t][h][:] and dt_bias[h][:];
    v-head h reads k-head h // (Hv/Hk)."""
    wl = _kda_workload(1)
    d = wl.dims
    res = oracle.forward(wl)
    x = wl.x.numpy().astype(np.float64)
    w = wl.conv_w.numpy().astype(np.float64)
    a = wl.a.numpy().astype(np.float64)
    b = wl.b.numpy().astype(np.float64)
    ref_blocks = [int(v) for v in wl.ref_blocks]
    cu = wl.cu_seqlens.tolist()
    ratio = d.Hv // d.Hk
    for s in range(wl.N):
        src = ref_blocks.index(int(wl.block_idx[s]) if wl.has_past[s] else 0)
        tail = wl.conv_state[src].numpy().astype(np.float64)
        y = oracle.conv_silu_seq(x[cu[s]:cu[s + 1]], tail, w)
        for h in range(d.Hv):
            kh = h // ratio
            q = y[:, kh * d.dk:(kh + 1) * d.dk]
            k = y[:, d.Hk * d.dk + kh * d.dk:d.Hk * d.dk + (kh + 1) * d.dk]
            v = y[:, 2 * d.Hk * d.dk + h * d.dv:2 * d.Hk * d.dk + (h + 1) * d.dv]
            S0 = wl.rec_state[src, h].numpy().astype(np.float64).T  # [k][v] -> S[v][k]
            o, S = oracle.kda_rule_head(q, k, v, a[cu[s]:cu[s + 1], h], b[cu[s]:cu[s + 1], h],
                                        float(wl.A_log[h]), wl.dt_bias[h].numpy(), S0)
            np.testing.assert_array_equal(res["out"][cu[s]:cu[s + 1], h], o)
            r = ref_blocks.index(int(wl.block_idx[s]))
            np.testing.assert_array_equal(res["rec_state"][r, h], S.T)


def test_forward_with_equal_channel_gates_equals_the_scalar_forward():
    wl = _kda_workload(2, slow=True)
    d = wl.dims
    a1 = wl.a[:, :, 0]
    db = wl.dt_bias[:, 0]
    kda = dataclasses.replace(wl, a=a1[:, :, None].expand(-1, -1, d.dk).contiguous(),
                              dt_bias=db[:, None].expand(-1, d.dk).contiguous())
    gdn = dataclasses.replace(wl, a=a1.contiguous(), dt_bias=db.contiguous())
    r1, r2 = oracle.forward(kda), oracle.forward(gdn)
    np.testing.assert_allclose(r1["out"], r2["out"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(r1["rec_state"], r2["rec_state"], rtol=0, atol=1e-14)
    np.testing.assert_array_equal(r1["conv_state"], r2["conv_state"])


def test_packed_equals_each_alone():
    wl = _kda_workload(0)
    full = oracle.forward(wl)
    cu = wl.cu_seqlens.tolist()
    refb = [int(v) for v in wl.ref_blocks]
    for s in range(wl.N):
        rows = torch.arange(cu[s], cu[s + 1])
        one = dataclasses.replace(
            wl, x=wl.x[rows], a=wl.a[rows], b=wl.b[rows],
            cu_seqlens=torch.tensor([0, cu[s + 1] - cu[s]], dtype=torch.int32),
            block_idx=wl.block_idx[s:s + 1], has_past=wl.has_past[s:s + 1])
        r = oracle.forward(one)
        np.testing.assert_array_equal(full["out"][cu[s]:cu[s + 1]], r["out"])
        i = refb.index(int(wl.block_idx[s]))
        np.testing.assert_array_equal(full["rec_state"][i], r["rec_state"][i])


def test_no_past_reads_only_the_trash_block():
    wl = _kda_workload(0)
    res = oracle.forward(wl)
    assert np.isfinite(res["out"]).all()  # the NaN-filled write blocks were never read


@pytest.mark.parametrize("cut", [1, 3, 64, 65])
def test_split_anywhere_equals_one_pass(cut):
    dims = synth.Dims(Hk=1, Hv=2, dk=8, dv=8, K=4, act="f32")
    L = 80
    whole = synth.make_workload("w", dims, [L], [0], 2, 3, block_idx=[1], slow_decay=True,
                                channel_gate=True)
    one = oracle.forward(whole)

    def part(lo, hi, past):
        return dataclasses.replace(
            whole, x=whole.x[lo:hi], a=whole.a[lo:hi], b=whole.b[lo:hi],
            cu_seqlens=torch.tensor([0, hi - lo], dtype=torch.int32),
            has_past=torch.tensor([past], dtype=torch.uint8))

    r1 = oracle.forward(part(0, cut, 0))
    second = dataclasses.replace(part(cut, L, 1), conv_state=torch.from_numpy(r1["conv_state"]),
                                 rec_state=torch.from_numpy(r1["rec_state"]))
    r2 = oracle.forward(second)
    np.testing.assert_allclose(np.concatenate([r1["out"], r2["out"]]), one["out"],
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(r2["rec_state"], one["rec_state"], rtol=0, atol=1e-12)


def test_gate_shapes_are_checked():
    wl = _kda_workload(0)
    bad = dataclasses.replace(wl, dt_bias=wl.dt_bias[:, :1].contiguous())
    with pytest.raises(ValueError):
        oracle.forward(bad)


@pytest.mark.parametrize("sub,split", [(16, 8), (16, 16), (32, 8)])
def test_referenced_intra_blocks_equal_the_pairwise_ones(sub, split):
    """The operand-rescaling form of A and P (references between sub-chunks
    and between the halves of a sub-chunk) equals the pairwise definition, on
    gates strong enough that one whole-chunk factorisation overflows."""
    n, dk = 64, 16
    d = _inputs(n, dk, 4, 41)
    g = d["g"] * 8.0  # about -30 per token and channel: e^{-Gam} overflows fp64 by the end
    Gam = np.cumsum(g, axis=0)
    A, P = kernel_forms.kda_intra_blocks(d["qn"], d["kn"], Gam, d["beta"], sub=sub, split=split)
    Aref = np.zeros((n, n))
    Pref = np.zeros((n, n))
    for i in range(n):
        for j in range(i + 1):
            f = np.exp(Gam[i] - Gam[j])
            Pref[i, j] = np.sum(d["qn"][i] * d["kn"][j] * f)
            if j < i:
                Aref[i, j] = d["beta"][i] * np.sum(d["kn"][i] * d["kn"][j] * f)
    np.testing.assert_allclose(A, Aref, rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(P, Pref, rtol=1e-12, atol=1e-300)
    with np.errstate(over="ignore", invalid="ignore"):
        whole = (d["kn"] * np.exp(Gam)) @ (d["kn"] * np.exp(-Gam)).T
    assert not np.isfinite(whole).all()

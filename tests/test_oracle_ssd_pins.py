"""Pins of the oracle's Mamba2 selective scan against facts other than itself
(CPU only).

The token loop is pinned by the other side of state space duality (the scan
written as one causal matrix product), by chunked state passing, by exact
closed forms with no decay and with total decay, and by the invariants of
the packed forward (packed = alone, split = whole, no past reads only the
trash block, the stated channel order and head-to-group map).  The
convolution is the gated delta net oracle's, pinned there against torch's
conv1d.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from continuous_linear_attention_gb300 import synth


def _rng(seed):
    return np.random.default_rng(seed)


def _chain(L, P, N, seed, slow=False):
    rng = _rng(seed)
    x = rng.standard_normal((L, P))
    B = rng.standard_normal((L, N))
    C = rng.standard_normal((L, N))
    dt = np.full(L, -4.0) if slow else rng.standard_normal(L)
    A_log = math.log(rng.uniform(0.01, 0.1) if slow else rng.uniform(1, 16))
    dt_bias = float(rng.standard_normal() * 0.5)
    Dskip = float(1 + 0.1 * rng.standard_normal())
    h0 = rng.standard_normal((P, N)) * 0.2
    step = F.softplus(torch.from_numpy(dt + dt_bias)).numpy()  # library softplus
    return dict(x=x, B=B, C=C, dt=dt, A_log=A_log, dt_bias=dt_bias, D=Dskip, h0=h0,
                step=step, logdecay=-math.exp(A_log) * step)


def _scan(c, **over):
    c = {**c, **over}
    return oracle.ssd_scan_head(c["x"], c["B"], c["C"], c["dt"], c["A_log"], c["dt_bias"],
                                c["D"], c["h0"])


@pytest.mark.parametrize("slow", [False, True])
@pytest.mark.parametrize("L", [1, 9, 40])
def test_scan_equals_the_quadratic_form(L, slow):
    """y = (causal decay mask o C B^T) (dt x) + decayed h_0 C + D x at every
    token, and the final state: a transposed B/C, a missing dt on the input,
    a decay applied after the input, or a dropped skip term fails here."""
    c = _chain(L, 6, 5, L * 7 + slow, slow=slow)
    y, h = _scan(c)
    y2, h2 = oracle.ssd_quadratic_form(c["x"], c["B"], c["C"], c["step"], c["logdecay"], c["D"],
                                       c["h0"])
    np.testing.assert_allclose(y, y2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(h, h2, rtol=0, atol=1e-12)


@pytest.mark.parametrize("L", [1, 63, 64, 65, 150])
def test_scan_equals_chunked_state_passing(L):
    c = _chain(L, 4, 8, 100 + L, slow=True)
    y, h = _scan(c)
    y2, h2 = oracle.ssd_chunked_forward(c["x"], c["B"], c["C"], c["step"], c["logdecay"], c["D"],
                                        c["h0"])
    np.testing.assert_allclose(y, y2, rtol=0, atol=1e-11)
    np.testing.assert_allclose(h, h2, rtol=0, atol=1e-11)


def test_no_decay_is_a_running_sum():
    """A_log = -1e4: exp(A_log) = 0 exactly, so a_t = 1 and
    h_t = h_0 + sum_{s<=t} dt_s x_s B_s^T, y_t = h_t C_t + D x_t."""
    c = _chain(7, 3, 4, 5)
    y, h = _scan(c, A_log=-1e4)
    run = c["h0"].copy()
    for t in range(7):
        run = run + c["step"][t] * np.outer(c["x"][t], c["B"][t])
        np.testing.assert_allclose(y[t], run @ c["C"][t] + c["D"] * c["x"][t], rtol=1e-12,
                                   atol=1e-14)
    np.testing.assert_allclose(h, run, rtol=1e-12, atol=1e-14)


def test_total_decay_forgets_the_state():
    """A_log = 800: exp(800) overflows to inf, a_t = e^{-inf} = 0, so each
    token's state is its own input alone."""
    c = _chain(3, 3, 4, 6)
    y, h = _scan(c, A_log=800.0)
    last = c["step"][2] * np.outer(c["x"][2], c["B"][2])
    np.testing.assert_allclose(h, last, rtol=1e-13, atol=0)  # dt: torch's softplus, to rounding
    np.testing.assert_allclose(y[2], last @ c["C"][2] + c["D"] * c["x"][2], rtol=1e-13)


# ----------------------------------------------------------------------------
# Whole packed forward.

TINY = synth.SsdDims(H=4, P=8, N=6, G=2, K=4, act="f32")


def _wl(seed=0, lens=(5, 1, 9), past=(0, 1, 0), slow=False):
    return synth.make_ssd_workload("ssd_tiny", TINY, list(lens), list(past), 8, seed,
                                   slow_decay=slow)


def test_forward_reads_channels_and_groups_as_stated():
    """Per chain: x channels of head h, B and C of group h // (H/G), in the
    order x | B | C; the conv continues from the block the sequence reads."""
    wl = _wl(1)
    d = wl.dims
    res = oracle.ssd_forward(wl)
    xbc = wl.xbc.numpy().astype(np.float64)
    w = wl.conv_w.numpy().astype(np.float64)
    dt = wl.dt.numpy().astype(np.float64)
    refb = [int(v) for v in wl.ref_blocks]
    cu = wl.cu_seqlens.tolist()
    for s in range(wl.N):
        src = refb.index(int(wl.block_idx[s]) if wl.has_past[s] else 0)
        y = oracle.conv_silu_seq(xbc[cu[s]:cu[s + 1]], wl.conv_state[src].numpy(), w)
        for hd in range(d.H):
            g = hd // (d.H // d.G)
            xs = y[:, hd * d.P:(hd + 1) * d.P]
            Bs = y[:, d.H * d.P + g * d.N:d.H * d.P + (g + 1) * d.N]
            Cs = y[:, d.H * d.P + d.G * d.N + g * d.N:d.H * d.P + d.G * d.N + (g + 1) * d.N]
            ys, hs = oracle.ssd_scan_head(xs, Bs, Cs, dt[cu[s]:cu[s + 1], hd], float(wl.A_log[hd]),
                                          float(wl.dt_bias[hd]), float(wl.D[hd]),
                                          wl.ssm_state[src, hd].numpy())
            np.testing.assert_array_equal(res["y"][cu[s]:cu[s + 1], hd], ys)
            r = refb.index(int(wl.block_idx[s]))
            np.testing.assert_array_equal(res["ssm_state"][r, hd], hs)


def test_packed_equals_each_alone_and_no_past_reads_only_trash():
    wl = _wl(0)
    full = oracle.ssd_forward(wl)
    assert np.isfinite(full["y"]).all()  # NaN-filled write blocks never read
    cu = wl.cu_seqlens.tolist()
    refb = [int(v) for v in wl.ref_blocks]
    for s in range(wl.N):
        rows = torch.arange(cu[s], cu[s + 1])
        one = dataclasses.replace(
            wl, xbc=wl.xbc[rows], dt=wl.dt[rows],
            cu_seqlens=torch.tensor([0, cu[s + 1] - cu[s]], dtype=torch.int32),
            block_idx=wl.block_idx[s:s + 1], has_past=wl.has_past[s:s + 1])
        r = oracle.ssd_forward(one)
        np.testing.assert_array_equal(full["y"][cu[s]:cu[s + 1]], r["y"])
        i = refb.index(int(wl.block_idx[s]))
        np.testing.assert_array_equal(full["ssm_state"][i], r["ssm_state"][i])
        np.testing.assert_array_equal(full["conv_state"][i], r["conv_state"][i])
    assert not full["conv_state"][0].any() and not full["ssm_state"][0].any()


@pytest.mark.parametrize("cut", [1, 2, 3, 64, 65])
def test_split_anywhere_equals_one_pass(cut):
    L = 80
    whole = synth.make_ssd_workload("w", TINY, [L], [0], 2, 3, block_idx=[1], slow_decay=True)
    one = oracle.ssd_forward(whole)

    def part(lo, hi, past):
        return dataclasses.replace(
            whole, xbc=whole.xbc[lo:hi], dt=whole.dt[lo:hi],
            cu_seqlens=torch.tensor([0, hi - lo], dtype=torch.int32),
            has_past=torch.tensor([past], dtype=torch.uint8))

    r1 = oracle.ssd_forward(part(0, cut, 0))
    second = dataclasses.replace(part(cut, L, 1), conv_state=torch.from_numpy(r1["conv_state"]),
                                 ssm_state=torch.from_numpy(r1["ssm_state"]))
    r2 = oracle.ssd_forward(second)
    np.testing.assert_allclose(np.concatenate([r1["y"], r2["y"]]), one["y"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r2["ssm_state"], one["ssm_state"], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(r2["conv_state"], one["conv_state"])


def test_skipped_sequences_and_new_conv_tails():
    wl = synth.make_ssd_workload("s", TINY, [2, 3, 0, 4], [1, 1, 0, 1], 6, 4,
                                 block_idx=[2, -1, 3, 4])
    init = np.full((wl.T, TINY.H, TINY.P), 7.25)
    res = oracle.ssd_forward(wl, out_init=init)
    assert (res["y"][2:5] == 7.25).all()  # padding sequence rows untouched
    refb = [int(v) for v in wl.ref_blocks]
    assert np.isnan(res["ssm_state"][refb.index(3)]).all()  # zero-length: block untouched
    xbc = wl.xbc.numpy()
    for s, (lo, hi) in [(0, (0, 2)), (3, (5, 9))]:
        r = refb.index(int(wl.block_idx[s]))
        old = wl.conv_state[r].numpy()
        np.testing.assert_array_equal(res["conv_state"][r], np.concatenate([old, xbc[lo:hi]])[-3:])


def test_pool_image_round_trip_through_the_stated_layout():
    """States packed into a byte image at the stated offsets (bf16 conv state,
    fp32 SSM state) decode back exactly: the decoder the GPU checks use reads
    the layout the boundary states."""
    dims = synth.SsdDims(H=4, P=32, N=32, G=2, K=4, act="bf16")
    nb, align = 5, 4096
    lay = oracle.ssd_pool_layout(nb, 1, dims.H, dims.P, dims.N, dims.G, dims.K, 2, align)
    img = np.zeros(lay["total"], dtype=np.uint8)
    rng = _rng(9)
    conv = torch.from_numpy(rng.standard_normal((nb, dims.K - 1, dims.C)).astype(np.float32))
    conv = conv.to(torch.bfloat16)
    ssm = rng.standard_normal((nb, dims.H, dims.P, dims.N)).astype(np.float32)
    for b in range(nb):
        o = b * lay["stride"]
        img[o:o + lay["conv_bytes"]] = conv[b].reshape(-1).view(torch.uint8).numpy()
        img[o + lay["ssm_off"]:o + lay["ssm_off"] + lay["ssm_bytes"]] = ssm[b].reshape(-1).view(np.uint8)
    c2, s2 = oracle.read_ssd_pool_states(img, 0, [3, 1], dims, nb, 1, block_align=align)
    np.testing.assert_array_equal(c2, conv.float().numpy()[[3, 1]].astype(np.float64))
    np.testing.assert_array_equal(s2, ssm[[3, 1]].astype(np.float64))
    assert lay["ssm_off"] % 128 == 0 and lay["stride"] % align == 0

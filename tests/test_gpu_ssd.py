"""GPU parity of the Mamba2 mixer forward (gdn_ssd_varlen_forward) against the
fp64 oracle, through the C ABI: packed batches of decodes and prefills with
and without a past, head dims 32 and 64, state sizes 32 to 128, fp32 and bf16
activations, padding and bad block indices."""
import pytest

from continuous_linear_attention_gb300 import synth

from gpu_check import check_ssd_against_oracle

pytestmark = pytest.mark.gpu

TINY = synth.SsdDims(H=4, P=32, N=32, G=2, K=4, act="f32")


def test_tiny_packed_fp32():
    check_ssd_against_oracle(synth.make_ssd_workload("ssd_tiny", TINY, [5, 1, 9], [0, 1, 0], 8,
                                                     0))


def test_tiny_packed_fp32_slow_decay():
    check_ssd_against_oracle(synth.make_ssd_workload("ssd_tiny_slow", TINY, [5, 1, 70],
                                                     [0, 1, 1], 8, 0, slow_decay=True))


@pytest.mark.parametrize("P,N", [(32, 64), (64, 32), (64, 128)])
def test_bf16_mixed_lengths(P, N):
    dims = synth.SsdDims(H=8, P=P, N=N, G=2, K=4, act="bf16")
    wl = synth.make_ssd_workload("ssd_mixed", dims, [70, 1, 1, 129, 3], [1, 1, 0, 0, 1], 16, 5)
    check_ssd_against_oracle(wl)


def test_decode_batch_large_heads():
    """128 heads of 64, state 128, 8 groups (the size class of the hybrid
    families' Mamba2 mixers): 64 decodes with a past, on the decode kernel."""
    dims = synth.SsdDims(H=128, P=64, N=128, G=8, K=4, act="bf16")
    wl = synth.make_ssd_workload("ssd_decode", dims, [1] * 64, [1] * 64, 128, 1)
    check_ssd_against_oracle(wl)


def test_decode_kernel_with_longer_sequences():
    """Decode kernel (H/G = 8) for the length-1 sequences and the token-serial
    kernel for the others, in one call."""
    dims = synth.SsdDims(H=16, P=64, N=128, G=2, K=4, act="bf16")
    lens = [1] * 24 + [65, 130, 3]
    wl = synth.make_ssd_workload("ssd_mixed_dec", dims, lens, [1] * 20 + [0] * 4 + [1, 0, 1], 40,
                                 2)
    check_ssd_against_oracle(wl)


def test_padding_and_bad_blocks_are_skipped():
    dims = synth.SsdDims(H=4, P=32, N=32, G=1, K=3, act="f32")
    wl = synth.make_ssd_workload("ssd_pad", dims, [3, 2, 0, 4], [1, 1, 0, 1], 6, 4,
                                 block_idx=[2, -1, 3, 4])
    check_ssd_against_oracle(wl)


def test_graph_replay_matches_eager():
    """Decodes and one prefill, captured once in a CUDA graph and replayed
    from the same pool contents: bit-identical to the eager call."""
    import torch

    from continuous_linear_attention_gb300 import harness
    dims = synth.SsdDims(H=16, P=64, N=128, G=2, K=4, act="bf16")
    wl = synth.make_ssd_workload("ssd_graph", dims, [1] * 8 + [40], [1] * 9, 16, 3)
    run = harness.SsdDeviceRun(wl)
    pool0 = run.mem.clone()
    run.run()
    torch.cuda.synchronize()
    y_eager = run.y.clone()
    g = torch.cuda.CUDAGraph()
    run.mem.copy_(pool0)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        run.run(torch.cuda.current_stream())
    run.mem.copy_(pool0)
    run.y.fill_(harness.OUT_SENTINEL)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(run.y, y_eager)
    assert run.pool.error_flags() == 0
    run.close()


@pytest.mark.parametrize("blocks,flag", [([3, 9, 5], 0x2), ([3, 0, 5], 0x4), ([3, 5, 5], 0x8)])
def test_bad_block_indices_are_flagged_and_skipped(blocks, flag):
    wl = synth.make_ssd_workload("ssd_bad", TINY, [4, 1, 3], [1, 1, 0], 8, 2, block_idx=blocks)
    check_ssd_against_oracle(wl, expect_flags=flag)


FULL = synth.SsdDims(H=16, P=64, N=128, G=2, K=4, act="bf16")


@pytest.mark.parametrize("lens,past", [
    ([128], [0]),                     # exactly one chunk
    ([129, 1, 40], [1, 1, 0]),        # a second chunk of one token, a decode, a short prefill
    ([300, 257], [0, 1]),             # three chunks with a partial last one, with a past
])
def test_chunked_scan_matches_the_oracle(lens, past):
    """At P = 64, N = 128, bf16 the prefills run as the chunked tensor-core
    scan (the scratch grows on the first call)."""
    wl = synth.make_ssd_workload("ssd_chunked", FULL, lens, past, 16, 11)
    check_ssd_against_oracle(wl)


def test_chunked_and_token_serial_scans_agree():
    import torch

    from continuous_linear_attention_gb300 import harness
    wl = synth.make_ssd_workload("ssd_both", FULL, [200, 1, 70], [1, 1, 0], 8, 12)
    a = harness.SsdDeviceRun(wl)
    b = harness.SsdDeviceRun(wl)
    b.pool.reserve(0)  # no scratch: token-serial kernel for the prefills
    a.run()
    b.run()
    torch.cuda.synchronize()
    err = (a.y.float() - b.y.float()).norm() / b.y.float().norm()
    assert float(err) <= 5e-3
    assert a.pool.error_flags() == 0 and b.pool.error_flags() == 0
    a.close()
    b.close()


@pytest.mark.parametrize("K", [2, 3, 4])
def test_chunked_scan_conv_widths_and_short_sequences(K):
    """The chunked scan's token-parallel conv at every conv width: sequences
    of two and three tokens whose window reaches into the past conv state,
    lengths on and next to the conv's 64-token chunks, with and without past."""
    dims = synth.SsdDims(H=16, P=64, N=128, G=2, K=K, act="bf16")
    lens = [2, 3, 63, 64, 65, 191, 1, 130]
    past = [1, 1, 1, 0, 1, 1, 1, 0]
    wl = synth.make_ssd_workload("ssd_conv_widths", dims, lens, past, 16, 13 + K)
    check_ssd_against_oracle(wl)


@pytest.mark.parametrize("slow", [False, True])
def test_chunked_scan_multi_chunk_chains(slow):
    """Chains of two to eight 128-token chunks (the X tile and the first
    head's masked matrix swap shared-memory regions every chunk and the next
    chunk's tiles load one chunk ahead), lengths on and next to two and three
    chunks, with and without a past; with slow decay the state carried from
    chunk to chunk dominates the outputs."""
    lens = [256, 257, 383, 384, 385, 1000, 2, 1]
    past = [1, 0, 1, 1, 0, 1, 1, 1]
    wl = synth.make_ssd_workload("ssd_multi_chunk", FULL, lens, past, 16, 17, slow_decay=slow)
    check_ssd_against_oracle(wl)

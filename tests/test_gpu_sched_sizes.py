"""The device scheduler over batch sizes past one sequence per thread: it
classifies up to four sequences per thread before its wait on the previous
kernel (list positions kept in registers) and falls back to classifying after
the wait for larger batches.  Both paths, with decodes, prefills, padding
entries, empty sequences and one duplicated block (flagged, both users
skipped), against the oracle at small head dims (token-serial kernels)."""
import numpy as np
import pytest

from continuous_linear_attention_gb300 import binding, synth

from gpu_check import check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_req", [3000, 5000])
def test_scheduler_classifies_large_batches(n_req):
    rng = np.random.default_rng(n_req)
    lens = np.where(rng.random(n_req) < 0.9, 1, rng.integers(0, 9, size=n_req)).tolist()
    has_past = rng.integers(0, 2, size=n_req).tolist()
    num_blocks = n_req + 8
    blocks = (rng.permutation(num_blocks - 1)[:n_req] + 1).tolist()
    for s in rng.choice(n_req, size=20, replace=False):
        blocks[s] = -1  # padding entries
    # one block named twice by requests with tokens: both are flagged and skipped
    users = [s for s in range(n_req) if blocks[s] > 0 and lens[s] > 0]
    blocks[users[1]] = blocks[users[0]]
    wl = synth.make_workload(f"sched_{n_req}", synth.TINY_DIMS, lens, has_past, num_blocks,
                             n_req, block_idx=blocks)
    check_against_oracle(wl, expect_flags=binding.FLAG_DUPLICATE)

"""Cycles per tcgen05.mma (kind::f16, M = 128, K = 16) as seen by the issuing
thread, for several N, with A in shared or in tensor memory.  The chunked
prefill kernels issue their products from one thread, so this per-instruction
cost bounds how fast a chain of small products can run.

    python -m continuous_linear_attention_gb300.diag_mma [--reps 64]
"""
import argparse
import json

import torch

from . import binding, build


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--reps", type=int, default=64, help="MMAs per measurement (multiple of 8)")
    args = ap.parse_args()
    build.build()
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    rows = []
    for a_tmem in (False, True):
        for N in (16, 32, 64, 128, 256):
            binding.diag_umma_issue_timing(N, a_tmem, args.reps, out)
            torch.cuda.synchronize()
            issue, total, ok = (int(v) for v in out.cpu())
            rows.append({"A": "tmem" if a_tmem else "smem", "N": N, "reps": args.reps,
                         "issue_cycles_per_mma": issue / args.reps,
                         "cycles_per_mma_to_completion": total / args.reps, "completed": bool(ok)})
    for r in rows:
        print(json.dumps(r))


if __name__ == "__main__":
    main()

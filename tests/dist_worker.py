"""One rank of the two-process gloo test (run by tests/test_dist_gloo.py, not collected)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import oracle  # noqa: E402
from sparse_mixture_experts_70_b300 import dist as D  # noqa: E402
from sparse_mixture_experts_70_b300 import workloads as wl  # noqa: E402


def main() -> None:
    rank, world, _ = D.env()
    D.init("gloo")
    w = wl.small(T=96, d=32, f=64, E=6, k=2, router_bias_var=1.0, seed=41)
    inp = wl.generate_router_inputs(w)
    lo, hi = rank * w.T // world, (rank + 1) * w.T // world
    # this rank's share of the batch, routed by the oracle (the GPU path's counts and psum
    # columns have the same meaning)
    z, p = oracle.router(inp["h"][lo:hi], inp["W_r"], inp["b_r"])
    idx, _, _ = oracle.topk(z, w.k)
    counts, *_ = oracle.dispatch(idx, w.E)
    aux = D.global_aux(torch.from_numpy(counts), torch.from_numpy(p.sum(0)), hi - lo, w.k)
    zl = D.global_zloss(oracle.zloss(z) * (hi - lo), hi - lo)
    slowest = D.max_over_ranks([float(rank + 1), 10.0 - rank])
    value = D.job_tokens_per_s(hi - lo, world, slowest[0])
    D.barrier()
    print(json.dumps({"rank": rank, "aux": aux, "zloss": zl, "slowest": slowest, "value": value}),
          flush=True)
    D.shutdown()


if __name__ == "__main__":
    main()

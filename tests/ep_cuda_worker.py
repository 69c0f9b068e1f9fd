"""One rank of the two-process expert-parallel test with the CUDA compute steps (run by
tests/test_gpu_ep_gloo.py, not collected). Both ranks share the one GPU of the machine, each in
its own process and CUDA context; the exchange is ep.forward's own all_to_all over gloo (rows
staged through host memory), so no kernel of one rank waits on the other."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from sparse_mixture_experts_70_b300 import binding as B  # noqa: E402
from sparse_mixture_experts_70_b300 import dist as D  # noqa: E402
from sparse_mixture_experts_70_b300 import ep  # noqa: E402
from sparse_mixture_experts_70_b300 import workloads as wl  # noqa: E402

CASES = {
    # name: (workload of the whole batch, tokens of rank 0)
    "swiglu_k2": (wl.small(T=700, d=256, f=320, E=6, k=2, seed=81), 420),
    "top1_gelu": (wl.small(T=900, d=128, f=256, E=16, k=1, act=wl.ACT_GELU_TANH,
                           gate=wl.GATE_RAW_PROB, seed=82), 300),
    "f32_bias_capacity": (wl.small(T=260, d=128, f=192, E=5, k=2, act=wl.ACT_GELU_TANH,
                                   dtype="f32", has_bias=True, capacity_factor=1.0,
                                   router_bias_var=1.0, seed=83), 130),
    # enough rows per expert for the CTA-pair GEMM on each rank's slice
    "pair_rows": (wl.small(T=2048, d=256, f=512, E=4, k=2, seed=84), 1024),
    "empty_rank": (wl.small(T=120, d=128, f=128, E=3, k=2, seed=85), 120),
}


def inputs_of(w):
    inputs = wl.generate(w)
    if w.has_bias:
        inputs = wl.random_biases(w, inputs, seed=w.seed + 100)
    return inputs


def main() -> None:
    rank, world, _ = D.env()
    D.init("gloo")
    torch.cuda.set_device(0)
    w, t0 = CASES[sys.argv[1]]
    inputs = inputs_of(w)
    dev = {k: (v.cuda().contiguous() if v is not None else None) for k, v in inputs.items()}
    lo_t, hi_t = (0, t0) if rank == 0 else (t0, w.T)
    mine = w.with_(T=hi_t - lo_t)
    backend = ep.LibmoeBackend(B.config_for(mine), dev, world)
    out = ep.forward(backend, dev["h"][lo_t:hi_t].contiguous(), w.E, world)
    torch.cuda.synchronize()
    status = B.moe_device_status(backend.ws)
    aux = D.global_aux(out["counts"], out["psum"], hi_t - lo_t, w.k)
    zl = D.global_zloss(out["lse2"], hi_t - lo_t)
    D.barrier()
    torch.save({"rank": rank, "tokens": (lo_t, hi_t), "experts": ep.expert_range(rank, world, w.E),
                "y": out["y"].cpu(), "idx": out["idx"].cpu(), "counts": out["counts"].cpu(),
                "recv_counts": out["recv_counts"], "aux": aux, "zloss": zl, "status": status},
               sys.argv[2])
    D.shutdown()


if __name__ == "__main__":
    main()

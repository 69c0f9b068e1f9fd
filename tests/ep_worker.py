"""One rank of the two-process expert-parallel test (run by tests/test_dist_ep_gloo.py, not
collected). Every compute step of the exchange runs in the double-precision oracle; the rank
holds only its own experts' weights."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from sparse_mixture_experts_70_b300 import dist as D  # noqa: E402
from sparse_mixture_experts_70_b300 import ep  # noqa: E402
from sparse_mixture_experts_70_b300 import workloads as wl  # noqa: E402

CASES = {
    # name: (workload of the whole batch, tokens of rank 0)
    "swiglu": (wl.small(T=67, d=32, f=64, E=5, k=2, seed=71), 40),
    "gelu_cap": (wl.small(T=90, d=32, f=64, E=4, k=1, act=wl.ACT_GELU_TANH, gate=wl.GATE_RAW_PROB,
                          has_bias=True, router_bias_var=1.0, capacity_factor=1.0, seed=72), 61),
    "empty_rank": (wl.small(T=30, d=32, f=64, E=3, k=2, seed=73), 30),
}


class OracleBackend:
    """route / dispatch / local_ffn / combine of one rank in the oracle (float64 rows)."""

    def __init__(self, w, inputs, lo, hi):
        self.w, self.inp = w, inputs
        sl = slice(lo, hi)
        self.W1, self.W2 = inputs["W1"][sl], inputs["W2"][sl]
        self.W3 = None if inputs.get("W3") is None else inputs["W3"][sl]
        self.b1 = None if inputs.get("b1") is None else inputs["b1"][sl]
        self.b2 = None if inputs.get("b2") is None else inputs["b2"][sl]

    def route(self, h):
        r = oracle.route(self.w, dict(self.inp, h=h))
        self.r = r
        T = h.shape[0]
        part = np.append(r["p"].sum(0), r["zloss"] * T).reshape(1, -1)
        return torch.from_numpy(r["idx"]), torch.from_numpy(r["g"]), torch.from_numpy(part)

    def dispatch(self, idx, h):
        r = self.r
        kept = int(r["offsets"][-1])
        x_perm = torch.zeros((idx.numel(), h.shape[1]), dtype=torch.float64)
        x_perm[:kept] = h.double()[torch.from_numpy(r["sorted_token"][:kept]).long()]
        return (torch.from_numpy(r["counts"]), torch.from_numpy(r["offsets"]),
                torch.from_numpy(r["slot_of"]), x_perm)

    def local_ffn(self, rows, local, lo, hi):
        y = oracle.expert_ffn(rows.numpy(), local.numpy(), self.W1, self.W3, self.W2, self.b1,
                              self.b2, oracle.act_code(self.w))
        return torch.from_numpy(y)

    def combine(self, y_perm, slot_of, gates):
        T, k = gates.shape
        s = slot_of.numpy().reshape(T, k)
        yslot = np.zeros((T, k, y_perm.shape[1]))
        yslot[s >= 0] = y_perm.numpy()[s[s >= 0]]
        return torch.from_numpy(oracle.combine(gates.numpy(), yslot))


def main() -> None:
    rank, world, _ = D.env()
    D.init("gloo")
    w, t0 = CASES[sys.argv[1]]
    inputs = wl.generate(w)
    lo_t, hi_t = (0, t0) if rank == 0 else (t0, w.T)
    mine = w.with_(T=hi_t - lo_t)
    lo, hi = ep.expert_range(rank, world, w.E)
    out = ep.forward(OracleBackend(mine, inputs, lo, hi), inputs["h"][lo_t:hi_t].contiguous(),
                     w.E, world)
    aux = D.global_aux(out["counts"], out["psum"], hi_t - lo_t, w.k)
    zl = D.global_zloss(out["lse2"], hi_t - lo_t)
    D.barrier()
    print(json.dumps({"rank": rank, "tokens": [lo_t, hi_t], "experts": [lo, hi],
                      "y": out["y"].tolist(), "recv_counts": out["recv_counts"].tolist(),
                      "counts": out["counts"].tolist(), "aux": aux, "zloss": zl}), flush=True)
    D.shutdown()


if __name__ == "__main__":
    main()

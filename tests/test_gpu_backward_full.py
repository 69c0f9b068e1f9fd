"""Backward parity at the full benchmark shapes (Mixtral, many-small, Switch, decode), in the
launch configuration bench.py times: sampled entries -- dh rows of a token sample and, for a few
(expert, hidden unit) pairs, rows of dW1 / dW3 and columns of dW2 -- against the oracle's sampled
backward, which evaluates exactly those entries. The oracle differentiates at its own routing;
where its top-k boundary or in-set margin is below 1e-4 the GPU's choice may differ and is used
instead (the reading the forward parity tests take)."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import workloads as wl

from parity import BF16_REL_L2, NEAR_TIE, to_dev

pytestmark = pytest.mark.gpu

AUX_W, Z_W = 0.01, 0.001


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b)) / max(float(np.linalg.norm(b)), 1e-30)


@pytest.mark.parametrize("name", ["mixtral", "many_small", "switch", "decode"])
def test_backward_full_size_sampled(name):
    w = wl.WORKLOADS[name]
    inputs = wl.generate(w)
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 1000)
    dy = torch.randn((w.T, w.d), generator=g).to(torch.bfloat16)
    dev = to_dev(inputs)
    cfg = B.config_for(w)
    layer = B.Layer(cfg, dev)
    layer.forward(dev["h"])
    grads = layer.backward(dev["h"], dy.cuda(), AUX_W, Z_W)
    torch.cuda.synchronize()
    assert B.moe_device_status(layer.ws) == B.MOE_OK
    idx_g = layer.topk_idx.cpu().numpy()
    got = {k: (v.float().cpu().numpy() if v is not None else None) for k, v in grads.items()}
    del layer, dev, grads
    torch.cuda.empty_cache()

    r = oracle.route(w, inputs)
    idx = r["idx"].copy()
    differ = np.nonzero((idx != idx_g).any(axis=1))[0]
    for t in differ:  # only near-ties may differ; there the GPU's choice is taken
        assert min(r["boundary"][t], r["inset"][t]) < NEAR_TIE, t
        assert sorted(idx_g[t]) == sorted(set(idx_g[t])) and (idx_g[t] < w.E).all()
        idx[t] = idx_g[t]
    assert len(differ) <= max(2, w.T // 1000)

    rng = np.random.default_rng(w.seed)
    toks = np.unique(np.concatenate([[0, w.T - 1], rng.choice(w.T, 10, replace=False)]))
    counts = np.bincount(idx.ravel(), minlength=w.E)
    hit = np.nonzero(counts)[0]
    # the first and last experts with slots and a random one; two hidden units each (the first /
    # last unit of an N tile, and a random one), so every operand's edge and interior are read
    experts = [hit[0], hit[-1], rng.choice(hit)]
    units = [0, w.f - 1, 255 % w.f, 256 % w.f, int(rng.integers(w.f)), int(rng.integers(w.f))]
    cols = [(int(e), int(units[2 * i + j])) for i, e in enumerate(experts) for j in range(2)]
    ref = oracle.backward_sampled(inputs["h"], inputs["W_r"], inputs.get("b_r"), inputs["W1"],
                                  inputs.get("W3"), inputs["W2"], inputs.get("b1"),
                                  inputs.get("b2"), idx, dy, oracle.act_code(w),
                                  oracle.gate_code(w), toks, cols, aux_weight=AUX_W,
                                  zloss_weight=Z_W)
    assert _rel_l2(got["dh"][toks], ref["dh"]) <= BF16_REL_L2
    e_idx = [e for e, _ in cols]
    n_idx = [n for _, n in cols]
    assert _rel_l2(got["dW1"][e_idx, n_idx], ref["dW1"]) <= BF16_REL_L2
    assert _rel_l2(got["dW2"][e_idx, :, n_idx], ref["dW2"]) <= BF16_REL_L2
    if ref["dW3"] is not None:
        assert _rel_l2(got["dW3"][e_idx, n_idx], ref["dW3"]) <= BF16_REL_L2
    # experts that received no slot have zero weight gradients
    for e in np.nonzero(counts == 0)[0][:4]:
        assert not got["dW1"][e].any() and not got["dW2"][e].any()

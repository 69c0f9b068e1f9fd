"""Expert parallelism with the C-ABI compute steps on one GPU.

With one rank the exchange is a copy, the regroup by local expert is the identity and the
k = 1 combine with gate 1 an exact copy: the layer output must equal the five step calls' bit for
bit. Two ranks are emulated in one process (each rank's buffers and weights slices are its own;
the all_to_all is done by hand on the device), and each rank's output is compared with the oracle
layer over that rank's tokens."""
import pytest
import torch

import oracle
from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import ep
from sparse_mixture_experts_70_b300 import workloads as wl

from parity import check_layer_output, rel_l2, run_steps, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    wl.small("ep_swiglu_k2", T=700, d=256, f=320, E=6, k=2),
    wl.small("ep_top1_gelu", T=900, d=128, f=256, E=16, k=1, act=wl.ACT_GELU_TANH,
             gate=wl.GATE_RAW_PROB),
    wl.small("ep_f32_bias", T=130, d=128, f=192, E=5, k=2, act=wl.ACT_GELU_TANH, dtype="f32",
             has_bias=True),
    wl.small("ep_capacity", T=600, d=128, f=256, E=8, k=2, capacity_factor=1.0, seed=5),
    # enough rows per expert for the CTA-pair GEMM, on the whole layer and on each rank's slice
    wl.small("ep_pair", T=2048, d=256, f=512, E=4, k=2, seed=9),
]


def _inputs(w):
    inputs = wl.generate(w)
    if w.has_bias:
        inputs = wl.random_biases(w, inputs, seed=w.seed + 100)
    return inputs


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_one_rank_equals_the_step_calls(w):
    inputs = _inputs(w)
    dev = to_dev(inputs)
    out = ep.forward(ep.LibmoeBackend(B.config_for(w), dev, 1), dev["h"], w.E, 1)
    torch.cuda.synchronize()
    steps = run_steps(w, inputs, dev)
    assert torch.equal(out["idx"].cpu(), steps["idx"])
    assert torch.equal(out["counts"].cpu(), steps["counts"])
    assert torch.equal(out["y"].cpu(), steps["y"])
    ref = oracle.reference(w, inputs)
    check_layer_output(w, ref, out["y"].cpu())


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_two_emulated_ranks_match_the_oracle(w):
    inputs = _inputs(w)
    dev = to_dev(inputs)
    world = 2
    cut = w.T * 3 // 5
    spans = [(0, cut), (cut, w.T)]
    ranges = [ep.expert_range(r, world, w.E) for r in range(world)]
    back = []
    routed = []
    for r, (a, b) in enumerate(spans):
        mine = w.with_(T=b - a)
        be = ep.LibmoeBackend(B.config_for(mine), dev, world)
        h = dev["h"][a:b].contiguous()
        idx, gates, psum = be.route(h)
        counts, offsets, slot_of, x_perm = be.dispatch(idx, h)
        off = offsets.cpu().long()
        routed.append(dict(be=be, idx=idx, gates=gates, slot_of=slot_of, x_perm=x_perm,
                           off=off, y_perm=torch.empty_like(x_perm)))
    # every owner: rows from each source in rank order, experts ascending within a source
    for q, (lo, hi) in enumerate(ranges):
        blocks, local, spans_q = [], [], []
        for s in routed:
            rlo, rhi = int(s["off"][lo]), int(s["off"][hi])
            blocks.append(s["x_perm"][rlo:rhi])
            for e in range(lo, hi):
                local += [e - lo] * int(s["off"][e + 1] - s["off"][e])
            spans_q.append((rlo, rhi))
        rows = torch.cat(blocks)
        loc = torch.tensor(local, dtype=torch.int32, device="cuda")
        y_in = routed[q]["be"].local_ffn(rows, loc, lo, hi) if rows.shape[0] else rows
        at = 0
        for s, (rlo, rhi) in zip(routed, spans_q):
            s["y_perm"][rlo:rhi] = y_in[at:at + rhi - rlo]
            at += rhi - rlo
    for r, ((a, b), s) in enumerate(zip(spans, routed)):
        y = s["be"].combine(s["y_perm"], s["slot_of"], s["gates"])
        torch.cuda.synchronize()
        mine = w.with_(T=b - a)
        sub = dict(inputs, h=inputs["h"][a:b].contiguous())
        ref = oracle.reference(mine, sub)
        check_layer_output(mine, ref, y.cpu())
        # a rank's layer output is also the one-GPU layer's over the same tokens (up to the
        # rounding of GEMM variants: the expert slices hold other row counts than the whole layer)
        steps = run_steps(mine, sub, to_dev(sub))
        assert rel_l2(y.cpu().double().numpy(), steps["y"].double().numpy()) <= 1e-3

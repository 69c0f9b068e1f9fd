"""Parity of moe_backward (through the C ABI) with the oracle's double-precision backward, on the
GPU's own routing (the expert choice is held fixed in the backward, so the oracle differentiates
at the GPU's idx). Cases span several row tiles with ragged tails, N and M tiles that are not
multiples of the tile, capacity drops, a router bias and a selection-only bias, top-1 Switch
gates with biases, the fused gather (no permuted copy), the tensor-core router, and an expert
that receives no slot. Every gradient is compared by relative L2 norm against the bf16 bound;
the auxiliary and z-loss terms are checked on their own with dy = 0."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import workloads as wl

from parity import BF16_REL_L2, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("dh", "dW_r", "db_r", "dW1", "dW3", "dW2", "db1", "db2")


def _case(w, bias_seed=None, zero_expert=False):
    inputs = wl.generate(w)
    if bias_seed is not None:
        inputs = wl.random_biases(w, inputs, bias_seed)
    if zero_expert:
        # expert 0 is never chosen: a large negative router bias on its logit
        b_r = inputs["b_r"].clone() if inputs.get("b_r") is not None else torch.zeros(w.E)
        b_r[0] = -60.0
        inputs["b_r"] = b_r
    return inputs


def _dy(w, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn((w.T, w.d), generator=g).to(torch.bfloat16)


def _run(w, inputs, dy, aux_weight, zloss_weight, train=False):
    dev = to_dev(inputs)
    cfg = B.config_for(w)
    layer = B.Layer(cfg, dev)
    # poison the backward workspace: every pad and partial must be written before it is read
    layer.bws = torch.full((max(B.moe_backward_workspace_size(cfg), 16),), 255, dtype=torch.uint8,
                           device="cuda")
    if train:
        layer.forward_train(dev["h"])  # keeps the pre-activations in bws
    else:
        layer.forward(dev["h"])
    g = layer.backward(dev["h"], dy.cuda(), aux_weight, zloss_weight)
    torch.cuda.synchronize()
    assert B.moe_device_status(layer.ws) == B.MOE_OK
    idx = layer.topk_idx.cpu().numpy()
    return {k: (v.float().cpu().numpy() if v is not None else None) for k, v in g.items()}, idx


def _oracle(w, inputs, idx, dy, aux_weight, zloss_weight):
    keep = None
    if w.capacity_factor > 0:
        C = oracle.capacity(w.capacity_factor, w.T, w.k, w.E)
        _, _, _, slot_of = oracle.dispatch_capacity(idx, w.E, C)
        keep = (slot_of >= 0).reshape(w.T, w.k)
    return oracle.backward(inputs["h"], inputs["W_r"], inputs.get("b_r"), inputs["W1"],
                           inputs.get("W3"), inputs["W2"], inputs.get("b1"), inputs.get("b2"),
                           idx, dy, oracle.act_code(w), oracle.gate_code(w), keep=keep,
                           aux_weight=aux_weight, zloss_weight=zloss_weight)


def _rel_l2(a, b):
    den = float(np.linalg.norm(b))
    return float(np.linalg.norm(a - b)) / max(den, 1e-30)


def _compare(got, ref, bound=BF16_REL_L2, names=GRADS):
    for name in names:
        if ref[name] is None:
            assert got[name] is None, name
            continue
        assert got[name].shape == ref[name].shape, name
        assert np.isfinite(got[name]).all(), name
        err = _rel_l2(got[name], ref[name])
        assert err <= bound, (name, err)


CASES = [
    (wl.small("bwd_swiglu_renorm", T=600, d=256, f=384, E=4, k=2, seed=21), {}, 0.0, 0.0),
    (wl.small("bwd_gelu_bias_raw_top1", T=700, d=192, f=256, E=5, k=1, act=wl.ACT_GELU_TANH,
              gate=wl.GATE_RAW_PROB, has_bias=True, router_bias_var=1.0, seed=22),
     dict(bias_seed=5), 0.3, 0.05),
    (wl.small("bwd_capacity", T=512, d=128, f=256, E=8, k=2, capacity_factor=1.0, seed=23), {},
     0.2, 0.0),
    (wl.small("bwd_selbias_top4", T=400, d=128, f=192, E=16, k=4, sel_bias_std=0.5,
              router_bias_var=0.5, seed=24), {}, 0.1, 0.1),
    (wl.small("bwd_gather", T=500, d=128, f=256, E=6, k=2, fuse_gather=True, seed=25), {}, 0.0,
     0.0),
    (wl.small("bwd_tc_router", T=3000, d=256, f=256, E=8, k=2, seed=26), {}, 0.05, 0.02),
    (wl.small("bwd_zero_expert", T=300, d=128, f=128, E=6, k=2, seed=27), dict(zero_expert=True),
     0.0, 0.0),
    # experts of at least four row tiles: the data-gradient GEMMs take the CTA-pair kernel
    (wl.small("bwd_pair", T=1100, d=128, f=320, E=2, k=2, seed=29), {}, 0.0, 0.0),
    # experts of one to six row tiles (skewed routing) on the single-CTA kernels, forward and
    # data-gradient GEMMs (W2 and W1 / W3 read MN-major)
    (wl.small("bwd_multi_tile", T=1000, d=256, f=384, E=6, k=2, router_bias_var=1.0,
              seed=30), {}, 0.05, 0.01),
]


@pytest.mark.parametrize("w,opts,aux_w,z_w", CASES, ids=lambda c: getattr(c, "name", ""))
def test_backward_matches_oracle(w, opts, aux_w, z_w):
    inputs = _case(w, **opts)
    dy = _dy(w, w.seed + 100)
    got, idx = _run(w, inputs, dy, aux_w, z_w)
    ref = _oracle(w, inputs, idx, dy, aux_w, z_w)
    _compare(got, ref)
    if opts.get("zero_expert"):
        assert not (idx == 0).any()
        for name in ("dW1", "dW3", "dW2"):
            if got[name] is not None:
                assert (got[name][0] == 0).all(), name


@pytest.mark.parametrize("aux_w,z_w", [(1.0, 0.0), (0.0, 1.0)])
def test_auxiliary_and_zloss_gradients_alone(aux_w, z_w):
    """dy = 0: only the auxiliary term (through P_i) or only the z-loss reaches the router, and
    the expert weights get no gradient."""
    w = wl.small("bwd_aux_only", T=640, d=128, f=128, E=8, k=2, router_bias_var=0.5, seed=28)
    inputs = _case(w)
    dy = torch.zeros((w.T, w.d), dtype=torch.bfloat16)
    got, idx = _run(w, inputs, dy, aux_w, z_w)
    ref = _oracle(w, inputs, idx, dy, aux_w, z_w)
    _compare(got, ref, names=("dh", "dW_r", "db_r"))
    for name in ("dW1", "dW3", "dW2"):
        assert (got[name] == 0).all(), name


@pytest.mark.parametrize("w,opts,aux_w,z_w", [CASES[0], CASES[1], CASES[2], CASES[4]],
                         ids=lambda c: getattr(c, "name", ""))
def test_training_forward_saves_what_the_backward_recomputes(w, opts, aux_w, z_w):
    """moe_forward_train + moe_backward(saved_preact = 1) against the oracle, and against the
    recomputing backward; the training forward's y equals moe_forward's bit for bit."""
    inputs = _case(w, **opts)
    dy = _dy(w, w.seed + 200)
    got, idx = _run(w, inputs, dy, aux_w, z_w, train=True)
    rec, idx2 = _run(w, inputs, dy, aux_w, z_w, train=False)
    assert np.array_equal(idx, idx2)
    _compare(got, _oracle(w, inputs, idx, dy, aux_w, z_w))
    for name in GRADS:
        if rec[name] is not None:
            assert _rel_l2(got[name], rec[name]) <= 1e-3, name
    dev = to_dev(inputs)
    cfg = B.config_for(w)
    a, b = B.Layer(cfg, dev), B.Layer(cfg, dev)
    ya = a.forward(dev["h"]).clone()
    yb = b.forward_train(dev["h"]).clone()
    torch.cuda.synchronize()
    assert torch.equal(ya, yb)
    assert torch.equal(a.aux, b.aux) and torch.equal(a.topk_idx, b.topk_idx)


@pytest.mark.parametrize("w", [
    wl.small("bwd_e256_k32", T=64, d=128, f=128, E=256, k=32, seed=31),
    wl.small("bwd_single_expert", T=300, d=128, f=192, E=1, k=1, act=wl.ACT_GELU_TANH,
             gate=wl.GATE_RAW_PROB, has_bias=True, seed=32),
], ids=lambda w: w.name)
def test_backward_at_the_limits(w):
    """E = 256 with k = 32 (every lane of the router warp holds a slot, 8 experts per lane) and a
    single expert (its gate is p = 1, so the router gets only the bias and aux terms)."""
    inputs = _case(w, bias_seed=7 if w.has_bias else None)
    dy = _dy(w, w.seed + 300)
    got, idx = _run(w, inputs, dy, 0.1, 0.05)
    _compare(got, _oracle(w, inputs, idx, dy, 0.1, 0.05))


def test_backward_is_deterministic_and_empty_batch_gives_zeros():
    w = wl.small("bwd_det", T=700, d=128, f=256, E=8, k=2, router_bias_var=0.5, seed=33)
    inputs = _case(w)
    dev = to_dev(inputs)
    cfg = B.config_for(w)
    layer = B.Layer(cfg, dev)
    layer.forward_train(dev["h"])
    dy = _dy(w, 5).cuda()
    first = {k: (v.clone() if v is not None else None)
             for k, v in layer.backward(dev["h"], dy, 0.1, 0.1).items()}
    for _ in range(3):
        again = layer.backward(dev["h"], dy, 0.1, 0.1)
        for k, v in first.items():
            if v is not None:
                assert torch.equal(v, again[k]), k  # no atomics: the same bits every call
    torch.cuda.synchronize()
    assert B.moe_device_status(layer.ws) == B.MOE_OK

    w0 = w.with_(T=0)
    dev0 = dict(dev)
    dev0["h"] = torch.empty((0, w.d), dtype=torch.bfloat16, device="cuda")
    layer0 = B.Layer(B.config_for(w0), dev0)
    layer0.forward(dev0["h"])
    # poison the outputs: an empty batch must overwrite every gradient with zeros
    layer0.grads = None
    g0 = layer0.backward(dev0["h"], torch.empty((0, w.d), dtype=torch.bfloat16, device="cuda"))
    for k in ("dW_r", "db_r", "dW1", "dW3", "dW2"):
        g0[k].fill_(7.0)
    g0 = layer0.backward(dev0["h"], torch.empty((0, w.d), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    for k in ("dW_r", "db_r", "dW1", "dW3", "dW2"):
        assert g0[k] is not None and not g0[k].any(), k


F32_CASES = [
    # the micro workload's shape: GELU with biases, f32 throughout, CUDA-core GEMMs
    (wl.small("bwd_f32_micro", T=256, d=128, f=512, E=8, k=2, act=wl.ACT_GELU_TANH, dtype="f32",
              has_bias=True, seed=41), dict(bias_seed=8), 0.2, 0.1),
    (wl.small("bwd_f32_swiglu_capacity", T=300, d=192, f=320, E=6, k=2, dtype="f32",
              capacity_factor=1.0, router_bias_var=0.5, seed=42), {}, 0.0, 0.05),
]
F32_REL_L2 = 2e-5  # f32 products and sums throughout (the oracle is double)


@pytest.mark.parametrize("w,opts,aux_w,z_w", F32_CASES, ids=lambda c: getattr(c, "name", ""))
def test_f32_backward_matches_oracle(w, opts, aux_w, z_w):
    inputs = _case(w, **opts)
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 100)
    dy = torch.randn((w.T, w.d), generator=g)
    got, idx = _run(w, inputs, dy, aux_w, z_w)
    _compare(got, _oracle(w, inputs, idx, dy, aux_w, z_w), bound=F32_REL_L2)


def test_backward_reads_the_routing_from_the_workspace():
    """moe_forward without topk_idx_out / counts_out keeps them in its workspace; moe_backward
    with NULL for both reads them there and gives the Layer path's bits."""
    w = wl.small("bwd_ws_routing", T=400, d=128, f=256, E=8, k=2, router_bias_var=0.5, seed=34)
    inputs = _case(w)
    dev = to_dev(inputs)
    cfg = B.config_for(w)
    dy = _dy(w, 9).cuda()
    layer = B.Layer(cfg, dev)
    layer.forward(dev["h"])
    want = {k: (v.clone() if v is not None else None)
            for k, v in layer.backward(dev["h"], dy, 0.1, 0.1).items()}
    ws = B.workspace(cfg)
    bws = torch.empty(B.moe_backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(layer.y)
    aux = torch.zeros(1, dtype=torch.float32, device="cuda")
    zl = torch.zeros(1, dtype=torch.float32, device="cuda")
    B.moe_forward(cfg, dev["h"], dev["W_r"], dev.get("b_r"), dev["W1"], None, dev.get("W3"),
                  dev["W2"], None, y, aux, None, None, ws, zloss_out=zl)
    got = {k: (torch.empty_like(v) if v is not None else None) for k, v in want.items()}
    B.moe_backward(cfg, dev["h"], dev["W_r"], dev.get("b_r"), dev["W1"], None, dev.get("W3"),
                   dev["W2"], None, None, None, dy, 0.1, 0.1, got["dh"], got["dW_r"], got["db_r"],
                   got["dW1"], None, got["dW3"], got["dW2"], None, ws, bws)
    torch.cuda.synchronize()
    assert B.moe_device_status(ws) == B.MOE_OK
    for k, v in want.items():
        if v is not None:
            assert torch.equal(v, got[k]), k


def test_training_step_replays_from_a_cuda_graph():
    """forward_train + backward recorded once in a CUDA graph (no host synchronisation inside)
    and replayed: the same bits as the eager calls."""
    w = wl.small("bwd_graph", T=900, d=256, f=256, E=8, k=2, seed=35)
    inputs = _case(w)
    dev = to_dev(inputs)
    layer = B.Layer(B.config_for(w), dev)
    dy = _dy(w, 11).cuda()
    h = dev["h"]
    layer.forward_train(h)
    eager = {k: (v.clone() if v is not None else None)
             for k, v in layer.backward(h, dy, 0.05, 0.02).items()}
    y_eager = layer.y.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # settles the library's one-time host queries
        layer.forward_train(h)
        layer.backward(h, dy, 0.05, 0.02)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward_train(h)
        layer.backward(h, dy, 0.05, 0.02)
    for k, v in layer.grads.items():
        if v is not None:
            v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert B.moe_device_status(layer.ws) == B.MOE_OK
    assert torch.equal(layer.y, y_eager)
    for k, v in eager.items():
        if v is not None:
            assert torch.equal(layer.grads[k], v), k

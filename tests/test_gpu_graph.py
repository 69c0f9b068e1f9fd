"""moe_forward recorded in a CUDA graph: replays give the eager call's bits, for the f32 path, a
bf16 layer with the cooperative (multi-chunk) dispatch and the paired GEMM, and a top-1 layer."""
import pytest
import torch

from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import workloads as wl

from parity import to_dev

pytestmark = pytest.mark.gpu

CASES = [
    wl.WORKLOADS["micro"],
    wl.small("graph_paired_coop", T=2600, d=256, f=384, E=4, k=2),
    wl.small("graph_top1", T=1500, d=128, f=256, E=16, k=1, act=wl.ACT_GELU_TANH,
             gate=wl.GATE_RAW_PROB),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_graph_replay_matches_eager(w):
    dev = to_dev(wl.generate(w))
    cfg = B.config_for(w)
    layer = B.Layer(cfg, dev)
    h = dev["h"].clone()
    layer.forward(h)
    torch.cuda.synchronize()
    expect = [t.clone() for t in (layer.y, layer.aux, layer.topk_idx, layer.counts)]
    graph = layer.capture(h)
    for t in (layer.y, layer.aux, layer.topk_idx, layer.counts):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    got = [layer.y, layer.aux, layer.topk_idx, layer.counts]
    for a, b in zip(expect, got):
        assert torch.equal(a, b)
    # new input in the captured buffer: the replay follows it
    h.copy_(torch.flip(dev["h"], dims=[0]))
    graph.replay()
    torch.cuda.synchronize()
    y_graph = layer.y.clone()
    layer.forward(h)
    torch.cuda.synchronize()
    assert torch.equal(y_graph, layer.y)
    assert B.moe_device_status(layer.ws) == B.MOE_OK

"""The kernel count moe_forward_launch_count reports against the kernels the CUDA profiler sees
in one moe_forward call, on configurations that take each launch plan: a small f32 layer
(dispatch and aux in one kernel, the first FFN kernel gathering from h, the second forming y), a
small bf16 layer (dispatch and aux in one kernel, permute, tensor-core GEMMs, combine), an f32
layer with more slots than one dispatch chunk and than the fused combine takes, the tensor-core
router (W_r split first), top-1 with the GEMM2 scatter (no combine), a capacity factor (combine
kept), the fused gather (no permute)."""
import json
import os
import tempfile

import pytest
import torch

from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import workloads as wl

from parity import to_dev

pytestmark = pytest.mark.gpu

OURS = ("router", "dispatch", "permute", "gemm", "ffn", "combine", "aux")

CASES = [
    wl.small("f32_gelu", T=200, d=128, f=256, E=8, k=2, act=wl.ACT_GELU_TANH, dtype="f32"),
    wl.small("bf16_single_chunk", T=100, d=128, f=256, E=8, k=2),
    wl.small("f32_many_slots", T=1200, d=128, f=256, E=8, k=2, act=wl.ACT_GELU_TANH,
             dtype="f32"),
    wl.small("tc_router_k2", T=3000, d=256, f=256, E=8, k=2),
    wl.small("top1_scatter", T=3000, d=128, f=256, E=16, k=1, act=wl.ACT_GELU_TANH,
             gate=wl.GATE_RAW_PROB),
    wl.small("top1_capacity", T=3000, d=128, f=256, E=16, k=1, act=wl.ACT_GELU_TANH,
             gate=wl.GATE_RAW_PROB, capacity_factor=1.25),
    wl.small("gather", T=500, d=128, f=256, E=6, k=2, fuse_gather=True),
]


def _kernels_in_trace(path: str) -> list[str]:
    with open(path) as fh:
        trace = json.load(fh)
    return [e["name"] for e in trace.get("traceEvents", []) if e.get("cat") == "kernel"]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_launch_count_matches_profiler(w):
    from torch.profiler import ProfilerActivity, profile
    dev = to_dev(wl.generate(w))
    cfg = B.config_for(w)
    layer = B.Layer(cfg, dev)
    layer.forward(dev["h"])
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        layer.forward(dev["h"])
        torch.cuda.synchronize()
    assert B.moe_device_status(layer.ws) == B.MOE_OK
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "trace.json")
        prof.export_chrome_trace(path)
        names = _kernels_in_trace(path)
    assert names, "the profiler recorded no kernels"
    assert all(any(o in n.lower() for o in OURS) for n in names), names
    assert len(names) == B.moe_forward_launch_count(cfg), names

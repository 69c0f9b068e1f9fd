"""moe_build_dispatch_static: dispatch for callers that cannot allocate device memory (a custom
operator handed only its inputs and outputs, a loop that must not call cudaMalloc). Its scratch is
a static device array inside libmoe, so its results must equal those of the workspace-based
moe_build_dispatch -- checked here through the C ABI on two calls in a row, the second on a
smaller problem, so that stale scratch left by the first call would show. This file is collected
last on purpose."""
import numpy as np
import pytest
import torch

from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import workloads as wl


def _dispatch_both(w, with_status=True):
    cfg = B.config_for(w)
    inp = wl.generate_router_inputs(w)
    h = inp["h"].cuda()
    W_r = inp["W_r"].cuda()
    b_r = inp["b_r"].cuda() if inp["b_r"] is not None else None
    T, k, E, d, P = w.T, w.k, w.E, w.d, w.P
    rows = B.moe_router_partials(cfg)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gates = torch.empty((T, k), dtype=torch.float32, device="cuda")
    psum = torch.empty((rows, E + 1), dtype=torch.float32, device="cuda")
    B.moe_router_topk(cfg, h, W_r, b_r, idx, gates, psum, B.workspace(cfg))
    outs = []
    for use_static in (False, True):
        counts = torch.full((E,), -3, dtype=torch.int32, device="cuda")
        offsets = torch.full((E + 1,), -3, dtype=torch.int32, device="cuda")
        st = torch.full((P,), -3, dtype=torch.int32, device="cuda")
        so = torch.full((P,), -3, dtype=torch.int32, device="cuda")
        xp = torch.zeros((P, d), dtype=w.torch_dtype, device="cuda")
        if use_static:
            status = torch.zeros(1, dtype=torch.int32, device="cuda") if with_status else None
            B.moe_build_dispatch_static(cfg, idx, h, counts, offsets, st, so, xp, status)
            torch.cuda.synchronize()
            assert status is None or status.item() == 0
        else:
            ws = B.workspace(cfg)
            B.moe_build_dispatch(cfg, idx, h, counts, offsets, st, so, xp, ws)
            assert B.moe_device_status(ws) == B.MOE_OK
        outs.append((counts.cpu(), offsets.cpu(), st.cpu(), so.cpu(), xp.cpu()))
    return idx.cpu(), outs


@pytest.mark.gpu
def test_static_scratch_dispatch_equals_workspace_dispatch_on_consecutive_calls():
    first = wl.small("static_a", T=9000, d=128, f=64, E=40, k=4, router_bias_var=2.0, seed=31)
    second = wl.small("static_b", T=700, d=64, f=64, E=40, k=4, router_bias_var=2.0, seed=32)
    for w in (first, second):
        idx, (ref, got) = _dispatch_both(w)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
        counts = ref[0].numpy()
        assert counts.sum() == w.P
        np.testing.assert_array_equal(counts, np.bincount(idx.numpy().ravel(), minlength=w.E))


@pytest.mark.gpu
def test_static_scratch_dispatch_without_a_status_word():
    """status = NULL: device-side failures are then not reported (they land in the array's
    header); the results are the same. Single-chunk (one block, no look-back) and multi-chunk
    shapes, one after the other."""
    for w in (wl.small("static_nostatus_a", T=300, d=64, f=64, E=12, k=3, seed=41),
              wl.small("static_nostatus_b", T=6000, d=64, f=64, E=24, k=2,
                       router_bias_var=1.0, seed=42)):
        idx, (ref, got) = _dispatch_both(w, with_status=False)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)


@pytest.mark.gpu
def test_static_scratch_rejects_shapes_beyond_its_capacity():
    # ceil(T k / 1024) * E = 257 * 256 > 65536 cells: refused before any launch
    cfg = B.config(T=257 * 1024 // 8, d=64, f=64, E=256, k=8)
    fake = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoEError) as err:
        B.moe_build_dispatch_static(cfg, fake, None, fake, fake, fake, fake, None)
    assert err.value.status == B.MOE_ERR_WORKSPACE

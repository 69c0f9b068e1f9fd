"""Failure detection without a GPU fault: the test hooks of include/moe_debug.h withhold one
signal with a short spin bound, so a bounded device-side wait runs out on purpose. The kernel must
record MOE_ERR_TIMEOUT, return within about the bound, and leave the context usable."""
import time

import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import workloads as wl

from parity import run_forward, to_dev

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000  # 20 ms


def _routing(w, dev, cfg, ws):
    rows = B.moe_router_partials(cfg)
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    gates = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    psum = torch.empty((rows, w.E + 1), dtype=torch.float32, device="cuda")
    B.moe_router_topk(cfg, dev["h"], dev["W_r"], dev["b_r"], idx, gates, psum, ws)
    return idx


def _assert_context_usable(w, inputs, dev):
    ref = oracle.route(w, inputs)
    fw = run_forward(w, dev)
    assert fw["status"] == B.MOE_OK
    np.testing.assert_array_equal(fw["counts"].numpy(), ref["counts"])


def test_dispatch_lookback_wait_runs_out_and_is_reported():
    w = wl.small("timeout_dispatch", T=3000, d=64, f=64, E=16, k=2, seed=51)
    inputs = wl.generate(w)
    dev = to_dev(inputs)
    cfg = B.config_for(w)
    ws = B.workspace(cfg)
    idx = _routing(w, dev, cfg, ws)
    counts = torch.empty(w.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(w.E + 1, dtype=torch.int32, device="cuda")
    st = torch.empty(w.P, dtype=torch.int32, device="cuda")
    so = torch.empty(w.P, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    B.moe_debug_dispatch_timeout(cfg, idx, counts, offsets, st, so, ws, LIMIT_NS)
    status = B.moe_device_status(ws)
    elapsed = time.perf_counter() - t0
    assert status == B.MOE_ERR_TIMEOUT
    assert elapsed < 5.0
    assert B.moe_device_status(ws) == B.MOE_OK  # read-and-clear
    _assert_context_usable(w, inputs, dev)


def test_expert_gemm_wait_runs_out_and_is_reported():
    w = wl.small("timeout_gemm", T=1000, d=256, f=256, E=4, k=2, seed=52)
    inputs = wl.generate(w)
    dev = to_dev(inputs)
    cfg = B.config_for(w)
    ws = B.workspace(cfg)
    idx = _routing(w, dev, cfg, ws)
    counts = torch.empty(w.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(w.E + 1, dtype=torch.int32, device="cuda")
    st = torch.empty(w.P, dtype=torch.int32, device="cuda")
    so = torch.empty(w.P, dtype=torch.int32, device="cuda")
    x_perm = torch.empty((w.P, w.d), dtype=torch.bfloat16, device="cuda")
    y_perm = torch.empty((w.P, w.d), dtype=torch.bfloat16, device="cuda")
    B.moe_build_dispatch(cfg, idx, dev["h"], counts, offsets, st, so, x_perm, ws)
    assert B.moe_device_status(ws) == B.MOE_OK
    t0 = time.perf_counter()
    B.moe_debug_expert_ffn_timeout(cfg, x_perm, offsets, dev["W1"], None, dev["W3"], dev["W2"],
                                   None, y_perm, ws, LIMIT_NS)
    status = B.moe_device_status(ws)
    elapsed = time.perf_counter() - t0
    assert status == B.MOE_ERR_TIMEOUT
    assert elapsed < 5.0
    # the same call without the hook succeeds right after
    B.moe_expert_ffn(cfg, x_perm, offsets, dev["W1"], None, dev["W3"], dev["W2"], None, y_perm, ws)
    assert B.moe_device_status(ws) == B.MOE_OK
    _assert_context_usable(w, inputs, dev)


def test_hooks_validate_their_arguments():
    cfg = B.config(T=100, d=64, f=64, E=4, k=2)   # 200 slots: a single dispatch chunk
    ws = B.workspace(cfg)
    t = torch.zeros(256, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoEError) as e:
        B.moe_debug_dispatch_timeout(cfg, t, t, t, t, t, ws, LIMIT_NS)
    assert e.value.status == B.MOE_ERR_INVALID_ARG
    cfg2 = B.config(T=3000, d=64, f=64, E=4, k=2)
    ws2 = B.workspace(cfg2)
    with pytest.raises(B.MoEError) as e:
        B.moe_debug_dispatch_timeout(cfg2, t, t, t, t, t, ws2, 10)  # bound below 1 ms
    assert e.value.status == B.MOE_ERR_INVALID_ARG

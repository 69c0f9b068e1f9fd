"""Helpers of the GPU parity tests: run libmoe through its C ABI on a workload's seeded inputs and
compare with the double-precision oracle (tests-only module)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_mixture_experts_70_b300 import binding as B

NEAR_TIE = 1e-4          # top-k decisions closer than this may differ between f32 and double
F32_MAX_ABS = 1e-4       # layer output bound for f32 workloads
BF16_REL_L2 = 1e-2       # layer output bound for bf16 workloads (f32 accumulation)
GATE_ABS = 2e-5          # f32 gates against the double gates
AUX_REL = 1e-4


def to_dev(inputs: dict, device="cuda") -> dict:
    return {k: (v.to(device).contiguous() if v is not None else None) for k, v in inputs.items()}


def run_steps(w, inputs: dict, dev: dict | None = None) -> dict:
    """Call the five step entry points one after another; return every intermediate on the host."""
    cfg = B.config_for(w)
    dev = dev or to_dev(inputs)
    T, k, E, d = w.T, w.k, w.E, w.d
    P = T * k
    dt = w.torch_dtype
    ws = B.workspace(cfg)
    rows = B.moe_router_partials(cfg)
    idx = torch.full((max(T, 1), k), -7, dtype=torch.int32, device="cuda")
    gates = torch.empty((max(T, 1), k), dtype=torch.float32, device="cuda")
    psum = torch.empty((max(rows, 1), E + 1), dtype=torch.float32, device="cuda")
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    sorted_token = torch.full((max(P, 1),), -7, dtype=torch.int32, device="cuda")
    slot_of = torch.full((max(P, 1),), -7, dtype=torch.int32, device="cuda")
    x_perm = torch.empty((max(P, 1), d), dtype=dt, device="cuda")
    y_perm = torch.empty((max(P, 1), d), dtype=dt, device="cuda")
    y = torch.empty((max(T, 1), d), dtype=dt, device="cuda")
    aux = torch.full((1,), -7.0, dtype=torch.float32, device="cuda")
    B.moe_router_topk(cfg, dev["h"], dev["W_r"], dev["b_r"], idx, gates, psum, ws,
                      sel_bias=dev.get("sel_bias"))
    B.moe_build_dispatch(cfg, idx, dev["h"], counts, offsets, sorted_token, slot_of, x_perm, ws)
    B.moe_expert_ffn(cfg, x_perm, offsets, dev["W1"], dev["b1"], dev["W3"], dev["W2"], dev["b2"],
                     y_perm, ws)
    B.moe_combine(cfg, y_perm, slot_of, gates, y)
    zloss = torch.full((1,), -7.0, dtype=torch.float32, device="cuda")
    B.moe_aux_loss(cfg, counts, psum, aux, zloss_out=zloss)
    status = B.moe_device_status(ws)
    torch.cuda.synchronize()
    out = dict(idx=idx[:T], gates=gates[:T], counts=counts, offsets=offsets,
               sorted_token=sorted_token[:P], slot_of=slot_of[:P], x_perm=x_perm[:P],
               y_perm=y_perm[:P], y=y[:T], aux=aux, zloss=zloss, status=status)
    return {k_: (v.cpu() if isinstance(v, torch.Tensor) else v) for k_, v in out.items()}


def run_forward(w, dev: dict, layer: B.Layer | None = None) -> dict:
    cfg = B.config_for(w)
    layer = layer or B.Layer(cfg, dev)
    layer.forward(dev["h"])
    status = B.moe_device_status(layer.ws)
    torch.cuda.synchronize()
    return dict(y=layer.y.cpu(), aux=layer.aux.cpu(), zloss=layer.zloss.cpu(),
                idx=layer.topk_idx.cpu(), counts=layer.counts.cpu(), status=status)


def routing_agreement(ref: dict, idx_gpu: np.ndarray) -> np.ndarray:
    """Tokens whose chosen experts differ from the oracle's. Each such token must be a near tie:
    a different set needs a boundary margin below NEAR_TIE, a different order an inset margin."""
    idx_ref = ref["idx"]
    diff = np.nonzero((idx_gpu != idx_ref).any(axis=1))[0]
    for t in diff:
        same_set = set(idx_gpu[t].tolist()) == set(idx_ref[t].tolist())
        margin = ref["inset"][t] if same_set else ref["boundary"][t]
        assert margin < NEAR_TIE, (t, idx_gpu[t], idx_ref[t], margin)
    return diff


def check_dispatch_valid(idx: np.ndarray, E: int, counts, offsets, sorted_token, slot_of,
                         C: int = -1) -> None:
    """The dispatch of routing `idx` (capacity C, -1 for none) is the stable counting sort that
    keeps the first C slots of every expert: checked by its properties."""
    T, k = idx.shape
    P = T * k
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    kept_counts = counts if C < 0 else np.minimum(counts, C)
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(kept_counts)]))
    kept = slot_of >= 0
    assert np.array_equal(np.sort(slot_of[kept]), np.arange(offsets[-1]))
    np.testing.assert_array_equal(sorted_token[slot_of[kept]], np.nonzero(kept)[0] // k)
    for e in range(E):
        slots = np.nonzero(flat == e)[0]            # token order
        lim = len(slots) if C < 0 else min(C, len(slots))
        np.testing.assert_array_equal(slot_of[slots[:lim]], np.arange(offsets[e], offsets[e] + lim))
        assert (slot_of[slots[lim:]] == -1).all()


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    num = np.linalg.norm((a - b).ravel())
    den = np.linalg.norm(b.ravel())
    return float(num / den) if den > 0 else float(num)


def check_layer_output(w, ref: dict, y_gpu: torch.Tensor, skip_tokens=()) -> dict:
    tokens = ref["tokens"]
    keep = np.array([t not in set(skip_tokens) for t in tokens])
    yg = y_gpu.float().numpy().astype(np.float64)[tokens[keep]]
    yr = ref["y"][keep]
    stats = dict(max_abs=float(np.abs(yg - yr).max()) if yg.size else 0.0, rel_l2=rel_l2(yg, yr))
    if w.dtype == "f32":
        assert stats["max_abs"] <= F32_MAX_ABS, stats
    else:
        assert stats["rel_l2"] <= BF16_REL_L2, stats
    assert np.isfinite(yg).all()
    return stats

"""Thin Python binding of libmoe's C ABI (include/moe.h), one function per entry point, same names.

Argument marshalling only: tensors are passed as device pointers (``data_ptr()``), the stream as
the current torch stream, and a non-OK status raises ``MoEError``. Every step of the layer runs in
libmoe's CUDA kernels; there is no CPU path. If libmoe.so is missing the import of the library
fails loudly (build it with ``python -m sparse_mixture_experts_70_b300.build``).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
INCLUDE_DIR = os.path.join(os.path.dirname(_HERE), "include")
HEADER_PATH = os.path.join(INCLUDE_DIR, "moe.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_INDEX = 4, 5, 6
MOE_F32, MOE_BF16 = 0, 1
MOE_ACT_GELU_TANH, MOE_ACT_SWIGLU = 0, 1
MOE_GATE_RENORM, MOE_GATE_RAW_PROB = 0, 1


class moe_config_t(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("f", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("act", ctypes.c_int32), ("gate", ctypes.c_int32), ("has_bias", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float),
                ("fuse_gather", ctypes.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


_lib = None
_P = ctypes.c_void_p
_CFG = ctypes.POINTER(moe_config_t)


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"{LIB_PATH} is missing: run `python -m sparse_mixture_experts_70_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        st = ctypes.c_int32
        sig = {
            "moe_workspace_size": [_CFG, ctypes.POINTER(ctypes.c_size_t)],
            "moe_workspace_init": [_P, ctypes.c_size_t, _P],
            "moe_router_partials": [_CFG, ctypes.POINTER(ctypes.c_int64)],
            "moe_router_topk": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
            "moe_build_dispatch": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
            "moe_build_dispatch_static": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P],
            "moe_expert_ffn": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
            "moe_combine": [_CFG, _P, _P, _P, _P, _P],
            "moe_aux_loss": [_CFG, _P, _P, _P, _P, _P],
            "moe_update_sel_bias": [_CFG, _P, _P, ctypes.c_float, _P],
            "moe_forward": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                            ctypes.c_size_t, _P],
            "moe_forward_events": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, ctypes.c_size_t, _P, _P, _P],
            "moe_device_status": [_P, _P],
            "moe_forward_launch_count": [_CFG, ctypes.POINTER(ctypes.c_int32)],
            "moe_pipeline_create": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    ctypes.POINTER(ctypes.c_void_p)],
            "moe_pipeline_submit": [_P, _P, _P, _P],
            "moe_pipeline_join": [_P, _P],
            "moe_pipeline_device_status": [_P],
            "moe_pipeline_destroy": [_P],
            "moe_fp32_ffma_probe": [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                    ctypes.POINTER(ctypes.c_double)],
            "moe_debug_dispatch_timeout": [_CFG, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                           ctypes.c_uint64, _P],
            "moe_debug_expert_ffn_timeout": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                             ctypes.c_size_t, ctypes.c_uint64, _P],
            "moe_backward_workspace_size": [_CFG, ctypes.POINTER(ctypes.c_size_t)],
            "moe_backward_launch_count": [_CFG, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)],
            "moe_backward": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_float,
                             ctypes.c_float, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                             _P, ctypes.c_size_t, ctypes.c_int32, _P],
            "moe_forward_train": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                  ctypes.c_size_t, _P, ctypes.c_size_t, _P],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = st
        L.moe_status_string.argtypes = [ctypes.c_int32]
        L.moe_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def header_symbols() -> list[str]:
    """Names of the functions the headers in include/ declare."""
    names = set()
    for fn in sorted(os.listdir(INCLUDE_DIR)):
        if fn.endswith(".h"):
            text = open(os.path.join(INCLUDE_DIR, fn)).read()
            names |= set(re.findall(r"^\s*(?:moe_status_t|const char\s*\*)\s*(moe_\w+)\s*\(",
                                    text, flags=re.M))
    return sorted(names)


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def config(T: int, d: int, f: int, E: int, k: int, dtype: int = MOE_BF16,
           act: int = MOE_ACT_SWIGLU, gate: int = MOE_GATE_RENORM, has_bias: bool = False,
           capacity_factor: float = 0.0, fuse_gather: bool = False) -> moe_config_t:
    return moe_config_t(T, d, f, E, k, dtype, act, gate, 1 if has_bias else 0, capacity_factor,
                        1 if fuse_gather else 0)


def config_for(w) -> moe_config_t:
    """The moe_config_t of a workloads.Workload."""
    return config(w.T, w.d, w.f, w.E, w.k, MOE_F32 if w.dtype == "f32" else MOE_BF16,
                  MOE_ACT_SWIGLU if w.act == "swiglu" else MOE_ACT_GELU_TANH,
                  MOE_GATE_RAW_PROB if w.gate == "raw_prob" else MOE_GATE_RENORM, w.has_bias,
                  getattr(w, "capacity_factor", 0.0), getattr(w, "fuse_gather", False))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoEError(status, where)


def moe_workspace_size(cfg: moe_config_t) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(lib().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_workspace_init")


def moe_router_partials(cfg: moe_config_t) -> int:
    n = ctypes.c_int64()
    _check(lib().moe_router_partials(ctypes.byref(cfg), ctypes.byref(n)), "moe_router_partials")
    return n.value


def moe_forward_launch_count(cfg: moe_config_t) -> int:
    """Kernels one moe_forward call with cfg launches (host-only)."""
    n = ctypes.c_int32()
    _check(lib().moe_forward_launch_count(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_forward_launch_count")
    return n.value


def workspace(cfg: moe_config_t, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of moe_workspace_size(cfg) bytes (PyTorch-owned device memory)."""
    return torch.zeros(max(moe_workspace_size(cfg), 1024), dtype=torch.uint8, device=device)


def moe_router_topk(cfg, h, W_r, b_r, topk_idx, gates, psum_part, ws, stream=None,
                    sel_bias=None) -> None:
    """psum_part: [moe_router_partials(cfg), E + 1] float; sel_bias: [E] float or None."""
    _check(lib().moe_router_topk(ctypes.byref(cfg), _ptr(h), _ptr(W_r), _ptr(b_r), _ptr(sel_bias),
                                 _ptr(topk_idx), _ptr(gates), _ptr(psum_part), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)),
           "moe_router_topk")


def moe_build_dispatch(cfg, topk_idx, h, counts, offsets, sorted_token, slot_of, x_perm, ws,
                       stream=None) -> None:
    _check(lib().moe_build_dispatch(ctypes.byref(cfg), _ptr(topk_idx), _ptr(h), _ptr(counts),
                                    _ptr(offsets), _ptr(sorted_token), _ptr(slot_of),
                                    _ptr(x_perm), _ptr(ws), ws.numel() * ws.element_size(),
                                    _stream(stream)), "moe_build_dispatch")


def moe_build_dispatch_static(cfg, topk_idx, h, counts, offsets, sorted_token, slot_of, x_perm,
                              status=None, stream=None) -> None:
    """moe_build_dispatch without a workspace (its scratch is a static array inside libmoe)."""
    _check(lib().moe_build_dispatch_static(ctypes.byref(cfg), _ptr(topk_idx), _ptr(h),
                                           _ptr(counts), _ptr(offsets), _ptr(sorted_token),
                                           _ptr(slot_of), _ptr(x_perm), _ptr(status),
                                           _stream(stream)), "moe_build_dispatch_static")


def moe_expert_ffn(cfg, x_perm, offsets, W1, b1, W3, W2, b2, y_perm, ws, stream=None) -> None:
    _check(lib().moe_expert_ffn(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(W1),
                                _ptr(b1), _ptr(W3), _ptr(W2), _ptr(b2), _ptr(y_perm), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream)), "moe_expert_ffn")


def moe_combine(cfg, y_perm, slot_of, gates, y, stream=None) -> None:
    _check(lib().moe_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(slot_of), _ptr(gates), _ptr(y),
                             _stream(stream)), "moe_combine")


def moe_aux_loss(cfg, counts, psum_part, aux_out, stream=None, zloss_out=None) -> None:
    _check(lib().moe_aux_loss(ctypes.byref(cfg), _ptr(counts), _ptr(psum_part), _ptr(aux_out),
                              _ptr(zloss_out), _stream(stream)), "moe_aux_loss")


def moe_update_sel_bias(cfg, counts, sel_bias, gamma: float, stream=None) -> None:
    """One step of the selection-only routing bias: +gamma below the mean load, -gamma above."""
    _check(lib().moe_update_sel_bias(ctypes.byref(cfg), _ptr(counts), _ptr(sel_bias),
                                     float(gamma), _stream(stream)), "moe_update_sel_bias")


def moe_forward(cfg, h, W_r, b_r, W1, b1, W3, W2, b2, y, aux_out, topk_idx_out, counts_out, ws,
                stream=None, sel_bias=None, zloss_out=None) -> None:
    _check(lib().moe_forward(ctypes.byref(cfg), _ptr(h), _ptr(W_r), _ptr(b_r), _ptr(sel_bias),
                             _ptr(W1), _ptr(b1), _ptr(W3), _ptr(W2), _ptr(b2), _ptr(y),
                             _ptr(aux_out), _ptr(zloss_out), _ptr(topk_idx_out),
                             _ptr(counts_out), _ptr(ws), ws.numel() * ws.element_size(),
                             _stream(stream)), "moe_forward")


def moe_fp32_ffma_probe(blocks: int, threads: int, iters: int, out, stream=None) -> float:
    """Launch the FP32 FFMA probe (include/moe_probe.h) on `stream`; returns its flop count."""
    flops = ctypes.c_double()
    _check(lib().moe_fp32_ffma_probe(int(blocks), int(threads), int(iters), _ptr(out),
                                     _stream(stream), ctypes.byref(flops)), "moe_fp32_ffma_probe")
    return flops.value


def moe_debug_dispatch_timeout(cfg, topk_idx, counts, offsets, sorted_token, slot_of, ws,
                               spin_limit_ns: int, stream=None) -> None:
    """Test hook (include/moe_debug.h): dispatch whose look-back wait runs out on purpose."""
    _check(lib().moe_debug_dispatch_timeout(ctypes.byref(cfg), _ptr(topk_idx), _ptr(counts),
                                            _ptr(offsets), _ptr(sorted_token), _ptr(slot_of),
                                            _ptr(ws), ws.numel() * ws.element_size(),
                                            int(spin_limit_ns), _stream(stream)),
           "moe_debug_dispatch_timeout")


def moe_debug_expert_ffn_timeout(cfg, x_perm, offsets, W1, b1, W3, W2, b2, y_perm, ws,
                                 spin_limit_ns: int, stream=None) -> None:
    """Test hook (include/moe_debug.h): expert GEMM whose first-stage wait runs out on purpose."""
    _check(lib().moe_debug_expert_ffn_timeout(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets),
                                              _ptr(W1), _ptr(b1), _ptr(W3), _ptr(W2), _ptr(b2),
                                              _ptr(y_perm), _ptr(ws),
                                              ws.numel() * ws.element_size(), int(spin_limit_ns),
                                              _stream(stream)), "moe_debug_expert_ffn_timeout")


def moe_forward_events(cfg, h, W_r, b_r, W1, b1, W3, W2, b2, y, aux_out, topk_idx_out,
                       counts_out, ws, ffn_begin, ffn_end, stream=None, sel_bias=None,
                       zloss_out=None) -> None:
    """moe_forward recording torch.cuda.Event ffn_begin / ffn_end around the expert FFN."""
    for ev in (ffn_begin, ffn_end):
        if not ev.cuda_event:  # torch creates the CUDA event on its first record
            ev.record(stream if isinstance(stream, torch.cuda.Stream)
                      else torch.cuda.current_stream())
    _check(lib().moe_forward_events(ctypes.byref(cfg), _ptr(h), _ptr(W_r), _ptr(b_r),
                                    _ptr(sel_bias), _ptr(W1), _ptr(b1), _ptr(W3), _ptr(W2),
                                    _ptr(b2), _ptr(y), _ptr(aux_out), _ptr(zloss_out),
                                    _ptr(topk_idx_out), _ptr(counts_out), _ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream),
                                    ffn_begin.cuda_event, ffn_end.cuda_event),
           "moe_forward_events")


def moe_backward_workspace_size(cfg: moe_config_t) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_backward_workspace_size")
    return n.value


def moe_backward_launch_count(cfg: moe_config_t, saved_preact: bool = False) -> int:
    n = ctypes.c_int32()
    _check(lib().moe_backward_launch_count(ctypes.byref(cfg), 1 if saved_preact else 0,
                                           ctypes.byref(n)), "moe_backward_launch_count")
    return n.value


def moe_forward_train(cfg, h, W_r, b_r, W1, b1, W3, W2, b2, y, aux_out, topk_idx_out, counts_out,
                      ws, bws, stream=None, sel_bias=None, zloss_out=None) -> None:
    _check(lib().moe_forward_train(ctypes.byref(cfg), _ptr(h), _ptr(W_r), _ptr(b_r),
                                   _ptr(sel_bias), _ptr(W1), _ptr(b1), _ptr(W3), _ptr(W2),
                                   _ptr(b2), _ptr(y), _ptr(aux_out), _ptr(zloss_out),
                                   _ptr(topk_idx_out), _ptr(counts_out), _ptr(ws),
                                   ws.numel() * ws.element_size(), _ptr(bws),
                                   bws.numel() * bws.element_size(), _stream(stream)),
           "moe_forward_train")


def moe_backward(cfg, h, W_r, b_r, W1, b1, W3, W2, b2, topk_idx, counts, dy, aux_weight,
                 zloss_weight, dh, dW_r, db_r, dW1, db1, dW3, dW2, db2, ws, bws,
                 stream=None, saved_preact: bool = False) -> None:
    _check(lib().moe_backward(ctypes.byref(cfg), _ptr(h), _ptr(W_r), _ptr(b_r), _ptr(W1),
                              _ptr(b1), _ptr(W3), _ptr(W2), _ptr(b2), _ptr(topk_idx),
                              _ptr(counts), _ptr(dy), float(aux_weight), float(zloss_weight),
                              _ptr(dh), _ptr(dW_r), _ptr(db_r), _ptr(dW1), _ptr(db1), _ptr(dW3),
                              _ptr(dW2), _ptr(db2), _ptr(ws), ws.numel() * ws.element_size(),
                              _ptr(bws), bws.numel() * bws.element_size(),
                              1 if saved_preact else 0, _stream(stream)),
           "moe_backward")


def moe_device_status(ws, stream=None) -> int:
    """Synchronise, read and clear the device status word; returns the status code."""
    return int(lib().moe_device_status(_ptr(ws), _stream(stream)))


# ----------------------------------------------------------------------------------------------
# convenience: the whole layer on tensors already on the device

class Layer:
    """Holds device copies of a layer's weights (and an optional "sel_bias" [E] float, the
    selection-only routing bias) and a workspace; ``forward(h)`` calls moe_forward, writing y,
    aux, zloss, topk_idx and counts."""

    def __init__(self, cfg: moe_config_t, weights: dict, device="cuda"):
        self.cfg = cfg
        dev = torch.device(device)
        self.w = {k: (v.to(dev).contiguous() if v is not None else None) for k, v in weights.items()
                  if k != "h"}
        self.ws = workspace(cfg, dev)
        dt = torch.bfloat16 if cfg.dtype == MOE_BF16 else torch.float32
        self.y = torch.empty((cfg.T, cfg.d), dtype=dt, device=dev)
        self.aux = torch.zeros(1, dtype=torch.float32, device=dev)
        self.zloss = torch.zeros(1, dtype=torch.float32, device=dev)
        self.topk_idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
        self.counts = torch.empty(cfg.E, dtype=torch.int32, device=dev)

    def forward(self, h: torch.Tensor, stream=None, ffn_events=None) -> torch.Tensor:
        """moe_forward on h; ffn_events = (begin, end) torch.cuda.Event to time the expert FFN."""
        w = self.w
        args = (self.cfg, h, w["W_r"], w.get("b_r"), w["W1"], w.get("b1"), w.get("W3"), w["W2"],
                w.get("b2"), self.y, self.aux, self.topk_idx, self.counts, self.ws)
        extra = dict(sel_bias=w.get("sel_bias"), zloss_out=self.zloss)
        self.saved_preact = False
        if ffn_events is None:
            moe_forward(*args, stream, **extra)
        else:
            moe_forward_events(*args, ffn_events[0], ffn_events[1], stream, **extra)
        return self.y

    def _bws(self, device) -> torch.Tensor:
        if getattr(self, "bws", None) is None:
            self.bws = torch.empty(max(moe_backward_workspace_size(self.cfg), 16),
                                   dtype=torch.uint8, device=device)
        return self.bws

    def forward_train(self, h: torch.Tensor, stream=None) -> torch.Tensor:
        """moe_forward_train on h: forward() that also keeps GEMM1's pre-activations in the
        backward workspace, so that the next backward() does not recompute them (bf16)."""
        w = self.w
        moe_forward_train(self.cfg, h, w["W_r"], w.get("b_r"), w["W1"], w.get("b1"), w.get("W3"),
                          w["W2"], w.get("b2"), self.y, self.aux, self.topk_idx, self.counts,
                          self.ws, self._bws(h.device), stream, sel_bias=w.get("sel_bias"),
                          zloss_out=self.zloss)
        self.saved_preact = True
        return self.y

    def backward(self, h: torch.Tensor, dy: torch.Tensor, aux_weight: float = 0.0,
                 zloss_weight: float = 0.0, stream=None) -> dict:
        """moe_backward after forward(h) or forward_train(h) (whose saved pre-activations it
        then uses): the gradients of sum(dy * y) + aux_weight * aux +
        zloss_weight * zloss (bf16 layers). Returns device tensors dh, dW_r, db_r, dW1, dW3,
        dW2, db1, db2 (None where the layer has no such parameter), owned by the Layer and
        overwritten by the next call."""
        cfg, w = self.cfg, self.w
        dev = h.device
        self._bws(dev)
        if getattr(self, "grads", None) is None:
            E, d, f = cfg.E, cfg.d, cfg.f
            bf = torch.bfloat16 if cfg.dtype == MOE_BF16 else torch.float32
            sw = cfg.act == MOE_ACT_SWIGLU
            self.grads = dict(
                dh=torch.empty((cfg.T, d), dtype=bf, device=dev),
                dW_r=torch.empty((d, E), dtype=torch.float32, device=dev),
                db_r=torch.empty(E, dtype=torch.float32, device=dev)
                if w.get("b_r") is not None else None,
                dW1=torch.empty((E, f, d), dtype=bf, device=dev),
                dW3=torch.empty((E, f, d), dtype=bf, device=dev) if sw else None,
                dW2=torch.empty((E, d, f), dtype=bf, device=dev),
                db1=torch.empty((E, f), dtype=torch.float32, device=dev) if cfg.has_bias else None,
                db2=torch.empty((E, d), dtype=torch.float32, device=dev) if cfg.has_bias else None)
        g = self.grads
        moe_backward(cfg, h, w["W_r"], w.get("b_r"), w["W1"], w.get("b1"), w.get("W3"), w["W2"],
                     w.get("b2"), self.topk_idx, self.counts, dy, aux_weight, zloss_weight,
                     g["dh"], g["dW_r"], g["db_r"], g["dW1"], g["db1"], g["dW3"], g["dW2"],
                     g["db2"], self.ws, self.bws, stream,
                     saved_preact=getattr(self, "saved_preact", False))
        return g

    def capture(self, h: torch.Tensor) -> "torch.cuda.CUDAGraph":
        """Record one moe_forward on the device tensor h into a CUDA graph. ``replay()`` reruns
        the layer on whatever h then holds (same buffer), writing self.y / aux / topk / counts.
        A forward on a side stream first settles the library's one-time host queries."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.forward(h)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.forward(h)
        return graph


class Pipeline:
    """moe_pipeline_*: batches of h in host memory through the layer, each batch's copy-in and
    copy-out overlapped with the neighbouring batches' computation (include/moe_pipeline.h).
    `weights` are device tensors (as for Layer); the layer runs on `stream` (default: the current
    stream at construction). Host tensors passed to submit() are kept alive until
    device_status() or close()."""

    def __init__(self, cfg: moe_config_t, weights: dict, stream=None):
        self.cfg = cfg
        self.w = {k: v for k, v in weights.items() if k != "h"}
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        w = self.w
        handle = ctypes.c_void_p()
        _check(lib().moe_pipeline_create(ctypes.byref(cfg), _ptr(w["W_r"]), _ptr(w.get("b_r")),
                                         _ptr(w.get("sel_bias")), _ptr(w["W1"]),
                                         _ptr(w.get("b1")), _ptr(w.get("W3")),
                                         _ptr(w["W2"]), _ptr(w.get("b2")), _stream(self.stream),
                                         ctypes.byref(handle)), "moe_pipeline_create")
        self._handle = handle
        self._pending = []
        self._dtype = torch.bfloat16 if cfg.dtype == MOE_BF16 else torch.float32

    def submit(self, h_host: torch.Tensor, y_host: torch.Tensor, aux_host: torch.Tensor) -> None:
        """Enqueue one batch: h_host [T, d] -> y_host [T, d], aux_host [1] (host tensors)."""
        shape = (self.cfg.T, self.cfg.d)
        for t in (h_host, y_host):
            if t.device.type != "cpu" or tuple(t.shape) != shape or t.dtype != self._dtype:
                raise ValueError(f"host tensors of shape {shape} and dtype {self._dtype} expected")
        if aux_host.device.type != "cpu" or aux_host.dtype != torch.float32 or aux_host.numel() < 1:
            raise ValueError("aux_host: a float32 host tensor")
        _check(lib().moe_pipeline_submit(self._handle, _ptr(h_host), _ptr(y_host), _ptr(aux_host)),
               "moe_pipeline_submit")
        self._pending.append((h_host, y_host, aux_host))

    def join(self, stream=None) -> None:
        """Make `stream` (default: the pipeline's stream) wait for every submitted batch."""
        _check(lib().moe_pipeline_join(self._handle, _stream(stream if stream is not None
                                                               else self.stream)),
               "moe_pipeline_join")

    def device_status(self) -> int:
        """Wait for all submitted batches; read and clear the device status word."""
        st = int(lib().moe_pipeline_device_status(self._handle))
        self._pending.clear()
        return st

    def close(self) -> None:
        if self._handle is not None and self._handle.value:
            lib().moe_pipeline_destroy(self._handle)
        self._handle = None
        self._pending.clear()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

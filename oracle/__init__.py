"""Double-precision CPU oracle of the top-k MoE FFN layer (forward and backward) -- TEST
INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this
package. The CUDA library and its Python binding never import, link or call it; the two share no
code. The arithmetic lives in ``moe_oracle.c`` (plain C, double, OpenMP over independent rows);
this module only builds it with gcc and marshals arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SO = os.path.join(_HERE, "libmoe_oracle.so")

F32, BF16 = 0, 1
GELU_TANH, SWIGLU = 0, 1
RENORM, RAW_PROB = 0, 1

_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/libmoe_oracle.so (gcc, -O2, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-fPIC", "-shared", _SRC, "-o", _SO + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_SO + ".tmp", _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        L.oracle_router.argtypes = [I64, I32, I32, P, I32, P, P, P, P]
        L.oracle_topk.argtypes = [I64, I32, I32, P, P, P, P]
        L.oracle_gates.argtypes = [I64, I32, I32, I32, P, P, P, P]
        L.oracle_dispatch.argtypes = [I64, I32, I32, P, P, P, P, P]
        L.oracle_expert_ffn.argtypes = [I64, I32, I32, I32, P, P, P, P, P, I32, P, P, P]
        L.oracle_combine.argtypes = [I64, I32, I32, P, P, P]
        L.oracle_forward_rows.argtypes = [I64, P, I32, I32, I32, I32, P, I32, P, P, P, P, P, I32,
                                          P, P, P]
        L.oracle_forward_rows_kept.argtypes = [I64, P, I32, I32, I32, I32, P, I32, P, P, P, P, P,
                                               I32, P, P, P, P]
        L.oracle_capacity.argtypes = [D, I64, I32, I32]
        L.oracle_capacity.restype = I64
        L.oracle_dispatch_capacity.argtypes = [I64, I32, I32, P, I64, P, P, P, P]
        L.oracle_aux_loss.argtypes = [I64, I32, I32, P, P]
        L.oracle_aux_loss.restype = D
        L.oracle_selection_keys.argtypes = [I64, I32, P, P, P]
        L.oracle_update_sel_bias.argtypes = [I64, I32, I32, P, D, P, P]
        L.oracle_zloss.argtypes = [I64, I32, P]
        L.oracle_zloss.restype = D
        L.oracle_param_count.argtypes = [I32, I64, I64, I32, I32, I32, I64, I64, I32, P, P]
        L.oracle_gelu_tanh.argtypes = [D]
        L.oracle_gelu_tanh.restype = D
        L.oracle_silu.argtypes = [D]
        L.oracle_silu.restype = D
        L.oracle_gelu_tanh_grad.argtypes = [D]
        L.oracle_gelu_tanh_grad.restype = D
        L.oracle_silu_grad.argtypes = [D]
        L.oracle_silu_grad.restype = D
        L.oracle_backward_sampled.argtypes = [I64, I32, I32, I32, I32, I32, I32, P, I32, P, P, P,
                                              P, P, I32, P, P, P, P, P, I32, D, D, I64, P, P,
                                              I64, P, P, P, P, P]
        L.oracle_backward.argtypes = [I64, I32, I32, I32, I32, I32, I32, P, I32, P, P, P, P, P,
                                      I32, P, P, P, P, P, I32, D, D, P, P, P, P, P, P, P, P, P]
        _lib = L
    return _lib


def set_threads(n: int) -> None:
    """Cap the OpenMP threads the oracle uses (takes effect for later parallel regions)."""
    try:
        omp = ctypes.CDLL("libgomp.so.1")
        omp.omp_set_num_threads(ctypes.c_int(int(n)))
    except OSError:
        os.environ["OMP_NUM_THREADS"] = str(n)


def max_threads() -> int:
    try:
        omp = ctypes.CDLL("libgomp.so.1")
        omp.omp_get_max_threads.restype = ctypes.c_int
        return int(omp.omp_get_max_threads())
    except OSError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------------------------
# marshalling helpers: torch CPU tensors are passed by pointer with their storage dtype code

def _stored(x) -> tuple[object, int]:
    """(contiguous CPU tensor/array kept alive, dtype code) for an f32 or bf16 input."""
    if isinstance(x, np.ndarray):
        x = torch.from_numpy(np.ascontiguousarray(x))
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x, BF16
    if x.dtype != torch.float32:
        x = x.to(torch.float32)
    return x, F32


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _f32(x):
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        x = torch.from_numpy(np.ascontiguousarray(x))
    return x.detach().cpu().to(torch.float32).contiguous()


def _np(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


# ----------------------------------------------------------------------------------------------
# one wrapper per oracle function

def router(h, W_r, b_r=None) -> tuple[np.ndarray, np.ndarray]:
    hs, hdt = _stored(h)
    T, d = hs.shape
    Wr = _f32(W_r)
    E = Wr.shape[1]
    br = _f32(b_r)
    z = np.empty((T, E), np.float64)
    p = np.empty((T, E), np.float64)
    lib().oracle_router(T, d, E, _ptr(hs), hdt, _ptr(Wr), _ptr(br), _ptr(z), _ptr(p))
    return z, p


def topk(z: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    z = _np(z, np.float64)
    T, E = z.shape
    idx = np.empty((T, k), np.int32)
    bnd = np.empty(T, np.float64)
    ins = np.empty(T, np.float64)
    lib().oracle_topk(T, E, k, _ptr(z), _ptr(idx), _ptr(bnd), _ptr(ins))
    return idx, bnd, ins


def gates(z: np.ndarray, p: np.ndarray, idx: np.ndarray, mode: int) -> np.ndarray:
    z = _np(z, np.float64)
    p = _np(p, np.float64)
    idx = _np(idx, np.int32)
    T, E = z.shape
    k = idx.shape[1]
    g = np.empty((T, k), np.float64)
    lib().oracle_gates(T, E, k, mode, _ptr(z), _ptr(p), _ptr(idx), _ptr(g))
    return g


def dispatch(idx: np.ndarray, E: int):
    idx = _np(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    sorted_token = np.empty(T * k, np.int32)
    slot_of = np.empty(T * k, np.int32)
    lib().oracle_dispatch(T, E, k, _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(sorted_token),
                          _ptr(slot_of))
    return counts, offsets, sorted_token, slot_of


def capacity(factor: float, T: int, k: int, E: int) -> int:
    return int(lib().oracle_capacity(float(factor), T, k, E))


def dispatch_capacity(idx: np.ndarray, E: int, C: int):
    """Dispatch with a per-expert capacity C (C < 0: no limit); slot_of is -1 for dropped slots."""
    idx = _np(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    sorted_token = np.full(T * k, -1, np.int32)
    slot_of = np.empty(T * k, np.int32)
    lib().oracle_dispatch_capacity(T, E, k, _ptr(idx), int(C), _ptr(counts), _ptr(offsets),
                                   _ptr(sorted_token), _ptr(slot_of))
    return counts, offsets, sorted_token, slot_of


def _weights(W1, W3, W2):
    w1, wdt = _stored(W1)
    w2, wdt2 = _stored(W2)
    assert wdt == wdt2
    w3 = None
    if W3 is not None:
        w3, wdt3 = _stored(W3)
        assert wdt3 == wdt
    return w1, w3, w2, wdt


def expert_ffn(x: np.ndarray, experts: np.ndarray, W1, W3, W2, b1=None, b2=None,
               act: int = SWIGLU) -> np.ndarray:
    x = _np(x, np.float64)
    experts = _np(experts, np.int32)
    n, d = x.shape
    w1, w3, w2, wdt = _weights(W1, W3, W2)
    f = w1.shape[1]
    b1c, b2c = _f32(b1), _f32(b2)
    y = np.empty((n, d), np.float64)
    lib().oracle_expert_ffn(n, d, f, act, _ptr(x), _ptr(experts), _ptr(w1), _ptr(w3), _ptr(w2),
                            wdt, _ptr(b1c), _ptr(b2c), _ptr(y))
    return y


def combine(g: np.ndarray, yslot: np.ndarray) -> np.ndarray:
    g = _np(g, np.float64)
    yslot = _np(yslot, np.float64)
    n, k = g.shape
    d = yslot.shape[-1]
    y = np.empty((n, d), np.float64)
    lib().oracle_combine(n, k, d, _ptr(g), _ptr(yslot), _ptr(y))
    return y


def forward_rows(tokens, h, idx, g, W1, W3, W2, b1=None, b2=None, act: int = SWIGLU,
                 keep=None):
    """Layer output rows of `tokens`; keep [T, k] (optional) marks the slots an expert processes."""
    tokens = _np(tokens, np.int64)
    hs, hdt = _stored(h)
    d = hs.shape[1]
    idx = _np(idx, np.int32)
    g = _np(g, np.float64)
    k = idx.shape[1]
    w1, w3, w2, wdt = _weights(W1, W3, W2)
    f = w1.shape[1]
    b1c, b2c = _f32(b1), _f32(b2)
    n = tokens.shape[0]
    y = np.empty((n, d), np.float64)
    if keep is None:
        lib().oracle_forward_rows(n, _ptr(tokens), d, f, k, act, _ptr(hs), hdt, _ptr(idx), _ptr(g),
                                  _ptr(w1), _ptr(w3), _ptr(w2), wdt, _ptr(b1c), _ptr(b2c), _ptr(y))
    else:
        kp = _np(keep, np.uint8)
        lib().oracle_forward_rows_kept(n, _ptr(tokens), d, f, k, act, _ptr(hs), hdt, _ptr(idx),
                                       _ptr(g), _ptr(w1), _ptr(w3), _ptr(w2), wdt, _ptr(b1c),
                                       _ptr(b2c), _ptr(kp), _ptr(y))
    return y


def aux_loss(counts: np.ndarray, p: np.ndarray, k: int) -> float:
    counts = _np(counts, np.int32)
    p = _np(p, np.float64)
    T, E = p.shape
    return float(lib().oracle_aux_loss(T, E, k, _ptr(counts), _ptr(p)))


def selection_keys(p: np.ndarray, b) -> np.ndarray:
    """Keys p + b of the selection-only routing bias (its top-k is the biased choice)."""
    p = _np(p, np.float64)
    T, E = p.shape
    b = _np(np.asarray(b, dtype=np.float64).reshape(E), np.float64)
    key = np.empty((T, E), np.float64)
    lib().oracle_selection_keys(T, E, _ptr(p), _ptr(b), _ptr(key))
    return key


def update_sel_bias(counts: np.ndarray, T: int, k: int, gamma: float, b) -> np.ndarray:
    """One step of the routing-bias update: +gamma below the mean load, -gamma above."""
    counts = _np(counts, np.int32)
    E = counts.shape[0]
    b = _np(np.asarray(b, dtype=np.float64).reshape(E), np.float64)
    out = np.empty(E, np.float64)
    lib().oracle_update_sel_bias(T, E, k, _ptr(counts), float(gamma), _ptr(b), _ptr(out))
    return out


def zloss(z: np.ndarray) -> float:
    """Router z-loss (1/T) sum_t (log sum_e exp z[t, e])^2."""
    z = _np(z, np.float64)
    T, E = z.shape
    return float(lib().oracle_zloss(T, E, _ptr(z)))


def param_count(n_layers, d, f, E, k, mats, shared_per_layer, shared_global, with_router=True):
    tot = ctypes.c_int64()
    act = ctypes.c_int64()
    lib().oracle_param_count(n_layers, d, f, E, k, mats, shared_per_layer, shared_global,
                             1 if with_router else 0, ctypes.byref(tot), ctypes.byref(act))
    return tot.value, act.value


def gelu_tanh(x: float) -> float:
    return float(lib().oracle_gelu_tanh(float(x)))


def silu(x: float) -> float:
    return float(lib().oracle_silu(float(x)))


def gelu_tanh_grad(x: float) -> float:
    return float(lib().oracle_gelu_tanh_grad(float(x)))


def silu_grad(x: float) -> float:
    return float(lib().oracle_silu_grad(float(x)))


def backward(h, W_r, b_r, W1, W3, W2, b1, b2, idx, dy, act: int, gate_mode: int, keep=None,
             aux_weight: float = 0.0, zloss_weight: float = 0.0) -> dict:
    """Gradients of sum(dy * y) + aux_weight * aux + zloss_weight * zloss for the routing idx
    (held fixed), all in double: dh, dW_r, db_r, dW1, dW3, dW2, db1, db2 (None where the layer
    has no such parameter) and dg, dL/dg of every slot [T, k]."""
    hs, hdt = _stored(h)
    T, d = hs.shape
    Wr = _f32(W_r)
    E = Wr.shape[1]
    br = _f32(b_r)
    idx = _np(idx, np.int32)
    k = idx.shape[1]
    w1, w3, w2, wdt = _weights(W1, W3, W2)
    f = w1.shape[1]
    b1c, b2c = _f32(b1), _f32(b2)
    dys, dydt = _stored(dy)
    kp = None if keep is None else _np(keep, np.uint8)
    out = dict(dh=np.empty((T, d)), dW_r=np.empty((d, E)), db_r=np.empty(E) if br is not None
               else None, dW1=np.empty((E, f, d)), dW3=np.empty((E, f, d)) if act == SWIGLU
               else None, dW2=np.empty((E, d, f)), db1=np.empty((E, f)) if b1c is not None
               else None, db2=np.empty((E, d)) if b2c is not None else None,
               dg=np.empty((T, k)))
    lib().oracle_backward(T, d, f, E, k, act, gate_mode, _ptr(hs), hdt, _ptr(Wr), _ptr(br),
                          _ptr(w1), _ptr(w3), _ptr(w2), wdt, _ptr(b1c), _ptr(b2c), _ptr(idx),
                          _ptr(kp), _ptr(dys), dydt, float(aux_weight), float(zloss_weight),
                          _ptr(out["dh"]), _ptr(out["dW_r"]), _ptr(out["db_r"]), _ptr(out["dW1"]),
                          _ptr(out["dW3"]), _ptr(out["dW2"]), _ptr(out["db1"]), _ptr(out["db2"]),
                          _ptr(out["dg"]))
    return out


def backward_sampled(h, W_r, b_r, W1, W3, W2, b1, b2, idx, dy, act: int, gate_mode: int,
                     tokens, cols, keep=None, aux_weight: float = 0.0,
                     zloss_weight: float = 0.0) -> dict:
    """Selected entries of backward() at any size: dh rows of `tokens`, and for each (e, n) in
    `cols` row n of dW1_e (and dW3_e) and column n of dW2_e, each as a length-d vector."""
    hs, hdt = _stored(h)
    T, d = hs.shape
    Wr = _f32(W_r)
    E = Wr.shape[1]
    br = _f32(b_r)
    idx = _np(idx, np.int32)
    k = idx.shape[1]
    w1, w3, w2, wdt = _weights(W1, W3, W2)
    f = w1.shape[1]
    b1c, b2c = _f32(b1), _f32(b2)
    dys, dydt = _stored(dy)
    kp = None if keep is None else _np(keep, np.uint8)
    tokens = _np(tokens, np.int64)
    cols = np.asarray(cols, dtype=np.int32).reshape(-1, 2)
    ce, cn = _np(cols[:, 0], np.int32), _np(cols[:, 1], np.int32)
    out = dict(dh=np.empty((len(tokens), d)), dW1=np.empty((len(cols), d)),
               dW3=np.empty((len(cols), d)) if act == SWIGLU else None,
               dW2=np.empty((len(cols), d)))
    lib().oracle_backward_sampled(T, d, f, E, k, act, gate_mode, _ptr(hs), hdt, _ptr(Wr), _ptr(br),
                                  _ptr(w1), _ptr(w3), _ptr(w2), wdt, _ptr(b1c), _ptr(b2c),
                                  _ptr(idx), _ptr(kp), _ptr(dys), dydt, float(aux_weight),
                                  float(zloss_weight), len(tokens), _ptr(tokens), _ptr(out["dh"]),
                                  len(cols), _ptr(ce), _ptr(cn), _ptr(out["dW1"]),
                                  _ptr(out["dW3"]), _ptr(out["dW2"]))
    return out


# ----------------------------------------------------------------------------------------------
# whole-layer reference for a workload

def act_code(w) -> int:
    return SWIGLU if w.act == "swiglu" else GELU_TANH


def gate_code(w) -> int:
    return RAW_PROB if w.gate == "raw_prob" else RENORM


def route(w, inputs) -> dict:
    """Router, top-k, gates, dispatch and auxiliary value over all T tokens of workload w
    (with the workload's capacity limit when it has one)."""
    z, p = router(inputs["h"], inputs["W_r"], inputs.get("b_r"))
    sel_bias = inputs.get("sel_bias")
    if sel_bias is not None:  # selection-only routing bias: choose by p + b, gate by p
        idx, bnd, ins = topk(selection_keys(p, sel_bias), w.k)
    else:
        idx, bnd, ins = topk(z, w.k)
    g = gates(z, p, idx, gate_code(w))
    factor = getattr(w, "capacity_factor", 0.0)
    if factor > 0:
        C = capacity(factor, w.T, w.k, w.E)
        counts, offsets, sorted_token, slot_of = dispatch_capacity(idx, w.E, C)
    else:
        C = -1
        counts, offsets, sorted_token, slot_of = dispatch(idx, w.E)
    aux = aux_loss(counts, p, w.k)
    return dict(z=z, p=p, idx=idx, boundary=bnd, inset=ins, g=g, counts=counts, offsets=offsets,
                sorted_token=sorted_token, slot_of=slot_of, aux=aux, zloss=zloss(z), capacity=C)


def reference(w, inputs, tokens=None) -> dict:
    """route() plus the layer output y (double) of the given tokens (all tokens when None)."""
    r = route(w, inputs)
    if tokens is None:
        tokens = np.arange(w.T, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    r["tokens"] = tokens
    keep = None if r["capacity"] < 0 else (r["slot_of"] >= 0).reshape(w.T, w.k)
    r["y"] = forward_rows(tokens, inputs["h"], r["idx"], r["g"], inputs["W1"], inputs.get("W3"),
                          inputs["W2"], inputs.get("b1"), inputs.get("b2"), act_code(w), keep=keep)
    return r


def sample_tokens(T: int, stride: int = 16, edge: int = 64) -> np.ndarray:
    """Deterministic token subset: every stride-th token plus the first and last `edge`."""
    s = set(range(0, T, stride)) | set(range(min(edge, T))) | set(range(max(0, T - edge), T))
    return np.array(sorted(s), dtype=np.int64)

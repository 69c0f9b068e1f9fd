"""The C-ABI library on the host: it loads, exports every function include/moe.h declares, and its
argument checks return the documented status codes before touching any device. CPU only."""
import ctypes
import subprocess

import pytest

from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import workloads as wl


def test_library_exports_every_declared_symbol():
    declared = B.header_symbols()
    assert len(declared) >= 11
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [s for s in declared if s not in exported]
    assert not missing, missing
    L = B.lib()
    for s in declared:
        assert getattr(L, s) is not None


def test_status_strings():
    for code, name in [(0, "MOE_OK"), (1, "MOE_ERR_INVALID_ARG"), (2, "MOE_ERR_UNSUPPORTED"),
                       (3, "MOE_ERR_WORKSPACE"), (4, "MOE_ERR_CUDA"), (5, "MOE_ERR_TIMEOUT"),
                       (6, "MOE_ERR_DEVICE_INDEX")]:
        assert B.status_string(code) == name


def _ws_size(cfg):
    n = ctypes.c_size_t()
    return B.lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), n.value


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workspace_sizes_of_the_workloads(name):
    w = wl.WORKLOADS[name]
    st, n = _ws_size(B.config_for(w))
    assert st == B.MOE_OK
    es = 4 if w.dtype == "f32" else 2
    # at least x_perm, H and y_perm
    assert n >= w.P * (2 * w.d + w.f) * es
    assert n < w.P * (2 * w.d + w.f) * es + 64 * 2**20


@pytest.mark.parametrize("kw,expect", [
    (dict(k=0), B.MOE_ERR_INVALID_ARG),
    (dict(k=9), B.MOE_ERR_INVALID_ARG),           # k > E
    (dict(E=0), B.MOE_ERR_INVALID_ARG),
    (dict(E=257, k=2), B.MOE_ERR_INVALID_ARG),
    (dict(d=100), B.MOE_ERR_INVALID_ARG),          # not a multiple of 64
    (dict(f=32), B.MOE_ERR_INVALID_ARG),
    (dict(T=-1), B.MOE_ERR_INVALID_ARG),
    (dict(T=2**30, k=2), B.MOE_ERR_INVALID_ARG),   # T k >= 2^31
    (dict(dtype=7), B.MOE_ERR_UNSUPPORTED),
    (dict(act=5), B.MOE_ERR_UNSUPPORTED),
    (dict(gate=3), B.MOE_ERR_UNSUPPORTED),
    (dict(E=64, k=33), B.MOE_ERR_UNSUPPORTED),     # k > 32 not built
    (dict(has_bias=True), B.MOE_ERR_UNSUPPORTED),  # SwiGLU has no biases
    (dict(capacity_factor=-1.0), B.MOE_ERR_INVALID_ARG),
    (dict(capacity_factor=float("nan")), B.MOE_ERR_INVALID_ARG),
    (dict(capacity_factor=float("inf")), B.MOE_ERR_INVALID_ARG),
])
def test_invalid_configs_are_rejected(kw, expect):
    base = dict(T=64, d=128, f=256, E=8, k=2, dtype=B.MOE_BF16, act=B.MOE_ACT_SWIGLU,
                gate=B.MOE_GATE_RENORM, has_bias=False)
    base.update(kw)
    cfg = B.config(**base)
    st, _ = _ws_size(cfg)
    assert st == expect
    L = B.lib()
    assert L.moe_forward(ctypes.byref(cfg), *([None] * 15), 0, None) == expect


def test_fuse_gather_flag():
    """fuse_gather takes 0 or 1; with bf16 it removes x_perm (P d 2 bytes, page-rounded) from the
    workspace, with f32 it changes nothing."""
    for dt in (B.MOE_BF16, B.MOE_F32):
        base = B.config(T=1000, d=256, f=512, E=8, k=2, dtype=dt)
        st0, n0 = _ws_size(base)
        fused = B.config(T=1000, d=256, f=512, E=8, k=2, dtype=dt, fuse_gather=True)
        st1, n1 = _ws_size(fused)
        assert st0 == st1 == B.MOE_OK
        if dt == B.MOE_BF16:
            assert n0 - n1 == 2000 * 256 * 2
        else:
            assert n0 == n1
    bad = B.config(T=64, d=128, f=256, E=8, k=2)
    bad.fuse_gather = 2
    assert _ws_size(bad)[0] == B.MOE_ERR_INVALID_ARG
    assert B.lib().moe_forward(ctypes.byref(bad), *([None] * 15), 0, None) == B.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("name,kw,expect", [
    # router, dispatch, aux, permute, GEMM1, GEMM2 (or the two f32 FFN launches), combine
    ("micro", {}, 4),                             # dispatch + aux in one kernel; f32: GEMM1
                                                  # gathers from h, GEMM2 forms y
    ("micro", {"dtype": "bf16"}, 6),              # dispatch + aux in one kernel
    ("micro", {"T": 2000}, 6),                    # two chunks; too many slots for the f32 combine
    ("decode", {}, 6),                            # dispatch + aux in one kernel
    ("mixtral", {}, 9),                           # tensor-core router: split, logits, select
    ("mixtral", {"fuse_gather": True}, 8),        # no permute
    ("switch", {}, 8),                            # top-1: GEMM2 scatters into y, no combine
    ("switch", {"capacity_factor": 1.0}, 9),      # drops possible: combine runs
    ("switch", {"fuse_gather": True}, 7),
    ("micro", {"T": 0}, 0),
])
def test_forward_launch_count(name, kw, expect):
    w = wl.WORKLOADS[name].with_(**kw)
    assert B.moe_forward_launch_count(B.config_for(w)) == expect


def test_pipeline_arguments_are_checked_before_any_cuda_call():
    L = B.lib()
    out = ctypes.c_void_p(123)
    bad = B.config(T=64, d=100, f=256, E=8, k=2)
    assert L.moe_pipeline_create(ctypes.byref(bad), *([None] * 9), ctypes.byref(out)) == \
        B.MOE_ERR_INVALID_ARG
    assert out.value is None  # *out cleared
    good = B.config(T=64, d=128, f=256, E=8, k=2)
    # NULL weights, misaligned weights, NULL out
    assert L.moe_pipeline_create(ctypes.byref(good), *([None] * 9), ctypes.byref(out)) == \
        B.MOE_ERR_INVALID_ARG
    assert L.moe_pipeline_create(ctypes.byref(good), 4, None, None, 18, None, 32, 64, None, None,
                                 ctypes.byref(out)) == B.MOE_ERR_INVALID_ARG
    assert L.moe_pipeline_create(ctypes.byref(good), 16, None, 18, 32, None, 48, 64, None, None,
                                 ctypes.byref(out)) == B.MOE_ERR_INVALID_ARG  # misaligned sel_bias
    assert L.moe_pipeline_create(ctypes.byref(good), 16, None, None, 32, None, 48, 64, None,
                                 None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_pipeline_submit(None, 16, 16, 16) == B.MOE_ERR_INVALID_ARG
    assert L.moe_pipeline_join(None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_pipeline_device_status(None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_pipeline_destroy(None) == B.MOE_OK


def test_null_and_misaligned_pointers_are_rejected_on_the_host():
    cfg = B.config(T=64, d=128, f=256, E=8, k=2)
    L = B.lib()
    st, n = _ws_size(cfg)
    assert st == 0
    fake = 1 << 40          # never dereferenced: the checks run before any launch
    # moe_forward(cfg, h, W_r, b_r, sel_bias, W1, b1, W3, W2, b2, y, aux, zloss, topk, counts,
    #             ws, ws_bytes, stream)
    def fwd(h=fake, sel=None, W1=fake, zl=None, ws_bytes=n):
        return L.moe_forward(ctypes.byref(cfg), h, fake, None, sel, W1, None, fake, fake, None,
                             fake, fake, zl, None, None, fake, ws_bytes, None)
    assert fwd(h=None) == B.MOE_ERR_INVALID_ARG             # missing h
    assert fwd(W1=fake + 2) == B.MOE_ERR_INVALID_ARG        # misaligned W1
    assert fwd(sel=fake + 2) == B.MOE_ERR_INVALID_ARG       # misaligned selection bias
    assert fwd(zl=fake + 2) == B.MOE_ERR_INVALID_ARG        # misaligned z-loss output
    assert fwd(ws_bytes=n - 1) == B.MOE_ERR_WORKSPACE       # workspace too small
    assert L.moe_expert_ffn(ctypes.byref(cfg), fake, fake, fake, None, fake, fake, None, fake,
                            fake, n - 1, None) == B.MOE_ERR_WORKSPACE
    assert L.moe_build_dispatch(ctypes.byref(cfg), fake, None, None, fake, fake, fake, None,
                                fake, n, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_combine(ctypes.byref(cfg), fake, fake, fake, fake + 8, None) == \
        B.MOE_ERR_INVALID_ARG
    assert L.moe_router_topk(ctypes.byref(cfg), fake, None, None, None, fake, fake, fake, fake, n,
                             None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_router_topk(ctypes.byref(cfg), fake, fake, None, fake + 1, fake, fake, fake, fake,
                             n, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_router_topk(ctypes.byref(cfg), fake, fake, None, None, fake, fake, fake, fake,
                             n - 1, None) == B.MOE_ERR_WORKSPACE
    assert L.moe_aux_loss(ctypes.byref(cfg), fake, fake, None, None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_aux_loss(ctypes.byref(cfg), fake, fake, fake, fake + 2, None) == \
        B.MOE_ERR_INVALID_ARG
    assert L.moe_update_sel_bias(ctypes.byref(cfg), fake, None, 0.1, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_update_sel_bias(ctypes.byref(cfg), fake, fake, float("inf"), None) == \
        B.MOE_ERR_INVALID_ARG
    assert L.moe_device_status(None, None) == B.MOE_ERR_INVALID_ARG


def test_router_partial_rows():
    for name, w in wl.WORKLOADS.items():
        rows = B.moe_router_partials(B.config_for(w))
        assert 1 <= rows <= w.T


@pytest.mark.parametrize("name,saved,expect", [("mixtral", 0, 16), ("mixtral", 1, 14),
                                               ("switch", 0, 14), ("switch", 1, 13),
                                               ("decode", 0, 17), ("many_small", 1, 14)])
def test_backward_launch_count(name, saved, expect):
    cfg = B.config_for(wl.WORKLOADS[name])
    assert B.moe_backward_launch_count(cfg, bool(saved)) == expect


def test_backward_arguments_are_checked_before_any_cuda_call():
    L = B.lib()
    fake = 1 << 40          # never dereferenced: the checks run before any launch
    f32 = B.config_for(wl.WORKLOADS["micro"])
    assert B.moe_backward_workspace_size(f32) > 0
    k = ctypes.c_int32()
    assert L.moe_backward_launch_count(ctypes.byref(f32), 0, ctypes.byref(k)) == B.MOE_OK
    assert k.value == 16  # f32: CUDA-core GEMMs, pre-activations recomputed
    assert L.moe_backward_launch_count(ctypes.byref(f32), 1, ctypes.byref(k)) == \
        B.MOE_ERR_UNSUPPORTED
    cfg = B.config(T=64, d=128, f=256, E=8, k=2)
    assert L.moe_backward_launch_count(ctypes.byref(cfg), 2, ctypes.byref(k)) == \
        B.MOE_ERR_INVALID_ARG
    nws, nbws = B.moe_workspace_size(cfg), B.moe_backward_workspace_size(cfg)

    # moe_backward(cfg, h, W_r, b_r, W1, b1, W3, W2, b2, topk, counts, dy, aux_w, z_w, dh, dW_r,
    #              db_r, dW1, db1, dW3, dW2, db2, ws, ws_bytes, bws, bws_bytes, saved, stream)
    def bwd(c=cfg, b_r=None, db_r=None, aux=0.0, ws=fake, bws=fake, bws_bytes=nbws, saved=0,
            dW1=fake):
        return L.moe_backward(ctypes.byref(c), fake, fake, b_r, dW1, None, fake, fake, None,
                              None, None, fake, aux, 0.0, fake, fake, db_r, fake, None, fake,
                              fake, None, ws, nws, bws, bws_bytes, saved, None)
    assert bwd(c=f32, saved=1) == B.MOE_ERR_UNSUPPORTED  # f32 layers recompute
    assert bwd(saved=2) == B.MOE_ERR_INVALID_ARG
    assert bwd(aux=float("nan")) == B.MOE_ERR_INVALID_ARG
    assert bwd(ws=None) == B.MOE_ERR_INVALID_ARG
    assert bwd(bws=fake + 8) == B.MOE_ERR_INVALID_ARG
    assert bwd(dW1=fake + 2) == B.MOE_ERR_INVALID_ARG
    assert bwd(b_r=fake) == B.MOE_ERR_INVALID_ARG          # b_r without db_r
    assert bwd(db_r=fake) == B.MOE_ERR_INVALID_ARG         # db_r without b_r
    assert bwd(bws_bytes=nbws - 1) == B.MOE_ERR_WORKSPACE

    # moe_forward_train(..., ws, ws_bytes, bws, bws_bytes, stream)
    def fwd_train(c=cfg, bws=fake, bws_bytes=nbws):
        return L.moe_forward_train(ctypes.byref(c), fake, fake, None, None, fake, None, fake,
                                   fake, None, fake, fake, None, None, None, fake, nws, bws,
                                   bws_bytes, None)
    assert fwd_train(bws=None) == B.MOE_ERR_INVALID_ARG
    assert fwd_train(bws_bytes=nbws - 1) == B.MOE_ERR_WORKSPACE
    nf = B.moe_workspace_size(f32)
    assert L.moe_forward_train(ctypes.byref(f32), fake, fake, None, None, fake, fake, None, fake,
                               fake, fake, fake, None, None, None, fake, nf, fake, 1 << 30,
                               None) == B.MOE_ERR_UNSUPPORTED

"""Pins for the oracle's backward pass, against central finite differences of the oracle's FORWARD
functions (router, gates, expert FFN + combine, auxiliary value, z-loss), which share no code with
the backward: a dropped term, a wrong sign, a transposed operand or a wrong index in any of the
backward's chain-rule steps moves at least one gradient entry by far more than the tolerance.

The loss is L = sum(dy * y) + aux_weight * aux + zloss_weight * zloss with the routing held fixed
(the pages: top-k selection is not differentiable; the gradient reaches the router through the
gates, and through P_i in the auxiliary term). Every input lies on a 2^-14 grid and is smaller
than 4 in magnitude, so x +- 2^-8 and x +- 2^-9 are exact in f32 and the differences see only
the smooth function; the two central differences are combined by Richardson extrapolation. Each perturbed point is checked to select the same experts, so the differentiated
function is the layer's own near that point. CPU only."""
import math

import numpy as np
import pytest

import oracle

GRID = 2.0 ** -14
EPS = 2.0 ** -9


def _q(a):
    """Round to the 2^-14 grid (exact in f32 for |a| < 4)."""
    return (np.clip(np.round(np.asarray(a) / GRID), -3.9 / GRID, 3.9 / GRID) * GRID).astype(
        np.float32)


def _layer(seed, T, d, f, E, k, act, gate, bias, router_bias, sel_bias=False):
    rng = np.random.default_rng(seed)
    p = dict(
        h=_q(rng.standard_normal((T, d))),
        W_r=_q(rng.standard_normal((d, E)) * 0.8),
        b_r=_q(rng.standard_normal(E) * 0.5) if router_bias else None,
        W1=_q(rng.standard_normal((E, f, d)) / math.sqrt(d)),
        W3=_q(rng.standard_normal((E, f, d)) / math.sqrt(d)) if act == oracle.SWIGLU else None,
        W2=_q(rng.standard_normal((E, d, f)) / math.sqrt(f)),
        b1=_q(rng.standard_normal((E, f)) * 0.3) if bias else None,
        b2=_q(rng.standard_normal((E, d)) * 0.3) if bias else None,
    )
    dy = rng.standard_normal((T, d)).astype(np.float32).astype(np.float64)  # as passed (f32)
    sb = rng.standard_normal(E) * 0.2 if sel_bias else None
    return p, dy, sb


def _route(p, k, sel_bias):
    z, pr = oracle.router(p["h"], p["W_r"], p["b_r"])
    keys = z if sel_bias is None else oracle.selection_keys(pr, sel_bias)
    idx, bnd, _ = oracle.topk(keys, k)
    return z, pr, idx, bnd


def _loss(p, dy, idx, counts, keep, act, gate, aux_w, z_w, sel_bias):
    z, pr, idx_now, _ = _route(p, idx.shape[1], sel_bias)
    assert np.array_equal(idx_now, idx), "a perturbation changed the routing"
    g = oracle.gates(z, pr, idx, gate)
    T = dy.shape[0]
    y = oracle.forward_rows(np.arange(T), p["h"], idx, g, p["W1"], p["W3"], p["W2"], p["b1"],
                            p["b2"], act, keep=keep)
    L = float((dy * y).sum())
    if aux_w:
        L += aux_w * oracle.aux_loss(counts, pr, idx.shape[1])
    if z_w:
        L += z_w * oracle.zloss(z)
    return L


def _check(seed, T, d, f, E, k, act, gate, bias=False, router_bias=False, capacity=0.0,
           aux_w=0.0, z_w=0.0, sel_bias=False):
    p, dy, sb = _layer(seed, T, d, f, E, k, act, gate, bias, router_bias, sel_bias)
    z, pr, idx, bnd = _route(p, k, sb)
    keep = None
    if capacity > 0:
        C = oracle.capacity(capacity, T, k, E)
        counts, _, _, slot_of = oracle.dispatch_capacity(idx, E, C)
        keep = (slot_of >= 0).reshape(T, k)
        assert not keep.all(), "the capacity case should drop a slot"
    else:
        counts, _, _, _ = oracle.dispatch(idx, E)
    g = oracle.backward(p["h"], p["W_r"], p["b_r"], p["W1"], p["W3"], p["W2"], p["b1"], p["b2"],
                        idx, dy, act, gate, keep=keep, aux_weight=aux_w, zloss_weight=z_w)
    names = [("h", "dh"), ("W_r", "dW_r"), ("b_r", "db_r"), ("W1", "dW1"), ("W3", "dW3"),
             ("W2", "dW2"), ("b1", "db1"), ("b2", "db2")]
    worst = 0.0
    for pname, gname in names:
        if p[pname] is None:
            assert g[gname] is None
            continue
        arr = p[pname]
        fd = np.empty(arr.shape)
        for i in np.ndindex(arr.shape):
            x0 = arr[i]
            cd = []
            for eps in (2 * EPS, EPS):
                arr[i] = x0 + np.float32(eps)
                lp = _loss(p, dy, idx, counts, keep, act, gate, aux_w, z_w, sb)
                arr[i] = x0 - np.float32(eps)
                lm = _loss(p, dy, idx, counts, keep, act, gate, aux_w, z_w, sb)
                arr[i] = x0
                cd.append((lp - lm) / (2 * eps))
            fd[i] = (4 * cd[1] - cd[0]) / 3  # Richardson: the eps^2 term cancels
        an = g[gname]
        assert an.shape == fd.shape, gname
        scale = max(1.0, float(np.abs(fd).max()))
        err = float(np.abs(an - fd).max()) / scale
        worst = max(worst, err)
        assert err < 1e-7, (gname, err)
        # the gradient is not trivially zero (a dropped contribution would show)
        assert np.abs(fd).max() > 1e-3, gname
    return worst


def test_swiglu_renorm_top2():
    _check(1, T=6, d=8, f=12, E=5, k=2, act=oracle.SWIGLU, gate=oracle.RENORM)


def test_gelu_bias_renorm_top2_router_bias():
    _check(2, T=6, d=8, f=12, E=5, k=2, act=oracle.GELU_TANH, gate=oracle.RENORM, bias=True,
           router_bias=True)


def test_gelu_raw_prob_top1_with_aux_and_zloss():
    _check(3, T=7, d=8, f=8, E=4, k=1, act=oracle.GELU_TANH, gate=oracle.RAW_PROB, bias=True,
           aux_w=0.37, z_w=0.11)


def test_swiglu_raw_prob_top3_aux_zloss_router_bias():
    _check(4, T=5, d=8, f=8, E=6, k=3, act=oracle.SWIGLU, gate=oracle.RAW_PROB,
           router_bias=True, aux_w=0.5, z_w=0.25)


def test_renorm_with_capacity_drops():
    _check(5, T=8, d=8, f=8, E=4, k=2, act=oracle.SWIGLU, gate=oracle.RENORM, capacity=0.75,
           aux_w=0.2)


def test_selection_bias_changes_choice_not_gradient_form():
    _check(6, T=6, d=8, f=8, E=5, k=2, act=oracle.GELU_TANH, gate=oracle.RENORM, bias=True,
           sel_bias=True, aux_w=0.3)


def test_dg_is_the_gate_derivative():
    """dg[t, j] equals the finite difference of sum(dy * y) in gate g[t, j] (the forward takes
    the gates as an input)."""
    T, d, f, E, k = 5, 8, 8, 4, 2
    p, dy, _ = _layer(7, T, d, f, E, k, oracle.SWIGLU, oracle.RENORM, False, False)
    z, pr, idx, _ = _route(p, k, None)
    g0 = oracle.gates(z, pr, idx, oracle.RENORM)
    b = oracle.backward(p["h"], p["W_r"], None, p["W1"], p["W3"], p["W2"], None, None, idx, dy,
                        oracle.SWIGLU, oracle.RENORM)
    for t in range(T):
        for j in range(k):
            gp, gm = g0.copy(), g0.copy()
            gp[t, j] += 1e-3
            gm[t, j] -= 1e-3
            yp = oracle.forward_rows(np.arange(T), p["h"], idx, gp, p["W1"], p["W3"], p["W2"],
                                     act=oracle.SWIGLU)
            ym = oracle.forward_rows(np.arange(T), p["h"], idx, gm, p["W1"], p["W3"], p["W2"],
                                     act=oracle.SWIGLU)
            fd = float((dy * (yp - ym)).sum()) / 2e-3
            assert abs(fd - b["dg"][t, j]) <= 1e-9 * max(1.0, abs(fd))  # linear in g


@pytest.mark.parametrize("fn,dfn", [("gelu_tanh", "gelu_tanh_grad"), ("silu", "silu_grad")])
def test_activation_derivatives(fn, dfn):
    """Closed-form derivatives against finite differences of the activations, plus special
    values: both slopes are 1/2 at 0, tend to 1 for large x and to 0 for large -x."""
    f, df = getattr(oracle, fn), getattr(oracle, dfn)
    for x in np.linspace(-6, 6, 97):
        e = 1e-5
        fd = (f(x + e) - f(x - e)) / (2 * e)
        assert abs(df(x) - fd) < 1e-8
    assert df(0.0) == pytest.approx(0.5, abs=1e-15)
    assert df(30.0) == pytest.approx(1.0, abs=1e-9)
    assert abs(df(-30.0)) < 1e-9


def test_backward_is_linear_in_dy_without_aux_terms():
    T, d, f, E, k = 6, 8, 8, 4, 2
    p, dy, _ = _layer(8, T, d, f, E, k, oracle.GELU_TANH, oracle.RENORM, True, True)
    _, _, idx, _ = _route(p, k, None)
    a = oracle.backward(p["h"], p["W_r"], p["b_r"], p["W1"], None, p["W2"], p["b1"], p["b2"],
                        idx, dy, oracle.GELU_TANH, oracle.RENORM)
    b = oracle.backward(p["h"], p["W_r"], p["b_r"], p["W1"], None, p["W2"], p["b1"], p["b2"],
                        idx, -2.0 * dy, oracle.GELU_TANH, oracle.RENORM)
    for key in ("dh", "dW_r", "db_r", "dW1", "dW2", "db1", "db2", "dg"):
        np.testing.assert_allclose(b[key], -2.0 * a[key], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("act,gate,k,capacity", [(oracle.SWIGLU, oracle.RENORM, 2, 0.0),
                                                (oracle.GELU_TANH, oracle.RAW_PROB, 1, 0.0),
                                                (oracle.SWIGLU, oracle.RENORM, 2, 0.75)])
def test_sampled_backward_equals_the_full_backward(act, gate, k, capacity):
    """The sampled form (used at sizes where the full backward is out of reach) gives the same
    entries as the full backward, which the finite differences above pin."""
    T, d, f, E = 9, 8, 12, 4
    p, dy, _ = _layer(9, T, d, f, E, k, act, gate, act == oracle.GELU_TANH, True)
    _, _, idx, _ = _route(p, k, None)
    keep = None
    if capacity > 0:
        _, _, _, slot_of = oracle.dispatch_capacity(idx, E, oracle.capacity(capacity, T, k, E))
        keep = (slot_of >= 0).reshape(T, k)
    args = (p["h"], p["W_r"], p["b_r"], p["W1"], p["W3"], p["W2"], p["b1"], p["b2"], idx, dy,
            act, gate)
    full = oracle.backward(*args, keep=keep, aux_weight=0.3, zloss_weight=0.2)
    toks = np.array([0, 4, T - 1])
    cols = [(e, n) for e in range(E) for n in (0, f - 1)]
    sm = oracle.backward_sampled(*args, toks, cols, keep=keep, aux_weight=0.3, zloss_weight=0.2)
    np.testing.assert_allclose(sm["dh"], full["dh"][toks], rtol=1e-12, atol=1e-13)
    for c, (e, n) in enumerate(cols):
        np.testing.assert_allclose(sm["dW1"][c], full["dW1"][e, n], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sm["dW2"][c], full["dW2"][e, :, n], rtol=1e-12, atol=1e-13)
        if act == oracle.SWIGLU:
            np.testing.assert_allclose(sm["dW3"][c], full["dW3"][e, n], rtol=1e-12, atol=1e-13)

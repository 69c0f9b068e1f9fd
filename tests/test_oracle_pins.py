"""Pins for the double-precision oracle, each against something other than the oracle itself:
values the pages print, closed forms, brute force, and independent library routines (numpy,
scipy). CPU only."""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from sparse_mixture_experts_70_b300 import workloads as wl


# ---------------------------------------------------------------------------------------------
# router: logits and softmax

def test_router_one_hot_weights_select_inputs():
    """W_r[i, e] = 1 iff i == pi(e) makes z[t, e] = h[t, pi(e)] exactly (d != E, so a transposed
    or mis-strided W_r cannot pass)."""
    rng = np.random.default_rng(0)
    T, d, E = 7, 16, 5
    h = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32))
    perm = rng.permutation(d)[:E]
    Wr = np.zeros((d, E), np.float32)
    Wr[perm, np.arange(E)] = 1.0
    z, p = oracle.router(h, torch.from_numpy(Wr))
    np.testing.assert_array_equal(z, h.numpy().astype(np.float64)[:, perm])


def test_router_reads_bf16_exactly_and_adds_bias():
    rng = np.random.default_rng(1)
    T, d, E = 5, 8, 3
    h = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32)).to(torch.bfloat16)
    Wr = np.zeros((d, E), np.float32)
    Wr[3, 0] = Wr[5, 1] = Wr[0, 2] = 1.0
    br = np.array([0.5, -2.0, 3.25], np.float32)
    z, _ = oracle.router(h, torch.from_numpy(Wr), torch.from_numpy(br))
    hw = h.to(torch.float32).numpy().astype(np.float64)
    np.testing.assert_array_equal(z, hw[:, [3, 5, 0]] + br.astype(np.float64))


def test_router_softmax_matches_scipy_and_two_expert_sigmoid():
    rng = np.random.default_rng(2)
    T, d, E = 33, 24, 9
    h = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32))
    Wr = torch.from_numpy((rng.standard_normal((d, E)) * 3).astype(np.float32))
    z, p = oracle.router(h, Wr)
    np.testing.assert_allclose(z, h.numpy().astype(np.float64) @ Wr.numpy().astype(np.float64),
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(p, scipy.special.softmax(z, axis=1), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-13)
    # E = 2: p_0 = sigmoid(z_0 - z_1)
    z2, p2 = oracle.router(h, Wr[:, :2].contiguous())
    np.testing.assert_allclose(p2[:, 0], scipy.special.expit(z2[:, 0] - z2[:, 1]), rtol=1e-12)


# ---------------------------------------------------------------------------------------------
# top-k

@pytest.mark.parametrize("E", [1, 2, 3, 4, 5, 6])
def test_topk_brute_force_all_subsets(E):
    """Enumerate every k-subset S; exactly one has min_S z > max_notS z; the oracle must return it,
    in descending order of z."""
    rng = np.random.default_rng(100 + E)
    z = rng.standard_normal((40, E))
    for k in range(1, E + 1):
        idx, bnd, ins = oracle.topk(z, k)
        for t in range(z.shape[0]):
            valid = [S for S in itertools.combinations(range(E), k)
                     if all(z[t, a] > z[t, b] for a in S for b in range(E) if b not in S)]
            assert len(valid) == 1
            assert set(idx[t].tolist()) == set(valid[0])
            assert all(z[t, idx[t, j]] > z[t, idx[t, j + 1]] for j in range(k - 1))
            rest = [b for b in range(E) if b not in valid[0]]
            if rest:
                assert bnd[t] == pytest.approx(min(z[t, list(valid[0])]) - max(z[t, rest]))
            else:
                assert bnd[t] == math.inf


def test_topk_matches_partial_sort_on_wide_rows():
    rng = np.random.default_rng(7)
    z = rng.standard_normal((200, 128))
    for k in (1, 2, 4, 8):
        idx, _, _ = oracle.topk(z, k)
        ref = np.argsort(-z, axis=1, kind="stable")[:, :k]
        np.testing.assert_array_equal(idx, ref)


def test_topk_ties_prefer_lower_index():
    z = np.array([[1.0, 3.0, 3.0, 2.0], [0.0, 0.0, 0.0, 0.0], [5.0, 1.0, 5.0, 5.0]])
    idx, bnd, ins = oracle.topk(z, 2)
    np.testing.assert_array_equal(idx, [[1, 2], [0, 1], [0, 2]])
    assert bnd[0] == 1.0 and bnd[1] == 0.0 and bnd[2] == 0.0
    assert ins[0] == 0.0


# ---------------------------------------------------------------------------------------------
# gates, with the worked example of the lensaml.com explainer, Step 3

def test_worked_example_top2_gates(golden):
    g = golden("lensa_step3_worked_combine.txt")
    p = np.zeros(8)
    un = [int(x) for x in g["unchosen_experts"]]
    p[un] = g["unchosen_p"]
    share = 1.0 - float(np.sum(g["unchosen_p"]))
    assert share == pytest.approx(g["chosen_share"], abs=1e-9)
    ch = [int(x) for x in g["chosen_experts"]]
    p[ch] = np.array(g["gates"]) * share
    z = np.log(p)[None, :] + 0.7            # logits are defined up to a constant
    idx, _, _ = oracle.topk(z, 2)
    assert idx[0].tolist() == ch
    g_ren = oracle.gates(z, p[None, :], idx, oracle.RENORM)
    assert g_ren[0].tolist() == pytest.approx(g["gates"], abs=1e-12)
    assert float(g_ren.sum()) == pytest.approx(1.0, abs=1e-15)
    assert len(ch) / 8 == pytest.approx(g["active_share"])


def test_gates_renorm_sum_to_one_and_equal_probability_ratio():
    rng = np.random.default_rng(3)
    h = torch.from_numpy(rng.standard_normal((64, 32)).astype(np.float32))
    Wr = torch.from_numpy(rng.standard_normal((32, 10)).astype(np.float32))
    z, p = oracle.router(h, Wr)
    for k in (1, 2, 3, 10):
        idx, _, _ = oracle.topk(z, k)
        g = oracle.gates(z, p, idx, oracle.RENORM)
        np.testing.assert_allclose(g.sum(1), 1.0, atol=1e-12)
        chosen_p = np.take_along_axis(p, idx.astype(np.int64), 1)
        np.testing.assert_allclose(g, chosen_p / chosen_p.sum(1, keepdims=True), rtol=1e-12)
        if k == 1:
            np.testing.assert_array_equal(g, 1.0)


def test_gates_raw_prob_is_router_probability():
    rng = np.random.default_rng(4)
    h = torch.from_numpy(rng.standard_normal((50, 16)).astype(np.float32))
    Wr = torch.from_numpy(rng.standard_normal((16, 6)).astype(np.float32))
    z, p = oracle.router(h, Wr)
    idx, _, _ = oracle.topk(z, 1)
    g = oracle.gates(z, p, idx, oracle.RAW_PROB)
    np.testing.assert_array_equal(g[:, 0], p.max(1))
    idx6, _, _ = oracle.topk(z, 6)
    g6 = oracle.gates(z, p, idx6, oracle.RAW_PROB)
    np.testing.assert_allclose(g6.sum(1), 1.0, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# dispatch

def _brute_force_groups(idx, E):
    T = idx.shape[0]
    return [[t for t in range(T) if e in idx[t].tolist()] for e in range(E)]


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (9, 4, 2), (100, 8, 2), (257, 16, 4), (64, 5, 5)])
def test_dispatch_is_stable_counting_sort(T, E, k):
    rng = np.random.default_rng(T * 1000 + E * 10 + k)
    z = rng.standard_normal((T, E)) + np.linspace(0, 2, E)   # skewed on purpose
    idx, _, _ = oracle.topk(z, k)
    counts, offsets, st, so = oracle.dispatch(idx, E)
    assert counts.sum() == T * k and offsets[-1] == T * k
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    np.testing.assert_array_equal(np.sort(so), np.arange(T * k))
    flat = idx.reshape(-1)
    for s in range(T * k):
        assert st[so[s]] == s // k
    groups = _brute_force_groups(idx, E)
    for e in range(E):
        assert counts[e] == len(groups[e])
        assert st[offsets[e]:offsets[e + 1]].tolist() == groups[e]
        assert all(flat[s] == e for s in range(T * k) if offsets[e] <= so[s] < offsets[e + 1])


def test_dispatch_reproduces_printed_slot_histogram(golden):
    g = golden("lensa_step4_histogram.txt")
    T, k, E = int(g["T"]), int(g["k"]), int(g["E"])
    counts_printed = [int(c) for c in g["counts"]]
    labels = np.repeat(np.arange(E), counts_printed)           # 512 slot labels, sorted
    idx = np.stack([labels[:T], labels[T:]], axis=1).astype(np.int32)
    assert all(idx[t, 0] != idx[t, 1] for t in range(T))       # a valid top-2 routing
    counts, offsets, _, _ = oracle.dispatch(idx, E)
    assert counts.tolist() == counts_printed
    assert int(counts.sum()) == T * k == 512
    assert round(counts.max() / counts.sum(), 3) == g["busiest_share"]
    assert round((counts[0] + counts[1]) / counts.sum(), 2) == g["top2_share"]
    assert int((counts == 0).sum()) == g["idle"]
    assert T * k // E == g["balanced"]


# ---------------------------------------------------------------------------------------------
# auxiliary load-balancing value (lensaml.com explainer, Step 4)

def test_aux_is_one_under_uniform_probability():
    rng = np.random.default_rng(5)
    for (T, E, k) in [(10, 4, 1), (64, 8, 2), (33, 16, 4)]:
        p = np.full((T, E), 1.0 / E)
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        counts, *_ = oracle.dispatch(idx, E)
        assert oracle.aux_loss(counts, p, k) == pytest.approx(1.0, abs=1e-12)


def test_aux_is_one_under_uniform_counts_and_E_when_collapsed():
    rng = np.random.default_rng(6)
    T, E, k = 64, 8, 2
    p = scipy.special.softmax(rng.standard_normal((T, E)) * 2, axis=1)
    counts = np.full(E, T * k // E, np.int32)
    assert oracle.aux_loss(counts, p, k) == pytest.approx(1.0, abs=1e-12)
    # every token to expert 0 with probability 1: E . 1 . 1
    p1 = np.zeros((T, E)); p1[:, 0] = 1.0
    c1 = np.zeros(E, np.int32); c1[0] = T
    assert oracle.aux_loss(c1, p1, 1) == pytest.approx(float(E), abs=1e-12)


def test_aux_with_zero_router_weights_is_one():
    rng = np.random.default_rng(8)
    h = torch.from_numpy(rng.standard_normal((40, 12)).astype(np.float32))
    z, p = oracle.router(h, torch.zeros(12, 6))
    np.testing.assert_array_equal(p, 1.0 / 6)
    idx, _, _ = oracle.topk(z, 3)
    counts, *_ = oracle.dispatch(idx, 6)
    assert oracle.aux_loss(counts, p, 3) == pytest.approx(1.0, abs=1e-14)


# ---------------------------------------------------------------------------------------------
# activations

def test_gelu_tanh_against_exact_gelu():
    xs = np.linspace(-8, 8, 4001)
    approx = np.array([oracle.gelu_tanh(x) for x in xs])
    exact = xs * scipy.special.ndtr(xs)
    err = np.abs(approx - exact)
    assert err.max() < 5e-4            # the tanh form's known approximation error
    assert err.max() > 1e-5            # ... and it is the tanh form, not the erf form
    assert oracle.gelu_tanh(0.0) == 0.0
    assert oracle.gelu_tanh(30.0) == 30.0 and oracle.gelu_tanh(-30.0) == 0.0


def test_silu_against_library_sigmoid_and_odd_identity():
    for x in np.linspace(-20, 20, 401):
        assert oracle.silu(x) == pytest.approx(x * scipy.special.expit(x), rel=1e-14, abs=1e-300)
        assert oracle.silu(x) - oracle.silu(-x) == pytest.approx(x, abs=1e-13)
    assert oracle.silu(0.0) == 0.0


# ---------------------------------------------------------------------------------------------
# expert FFN

def _mlp_inputs(rng, E, f, d, dtype=torch.float32):
    W1 = torch.from_numpy(rng.standard_normal((E, f, d)).astype(np.float32)).to(dtype)
    W3 = torch.from_numpy(rng.standard_normal((E, f, d)).astype(np.float32)).to(dtype)
    W2 = torch.from_numpy(rng.standard_normal((E, d, f)).astype(np.float32)).to(dtype)
    return W1, W3, W2


def test_expert_mlp_linear_regime_matches_numpy_matmul():
    """Pre-activations far above zero make GELU(a) = a and SiLU(a) = a to double precision, so the
    expert reduces to plain matrix products that numpy computes independently (d != f catches a
    transposed operand; several experts catch a wrong expert stride)."""
    rng = np.random.default_rng(9)
    E, f, d, n = 3, 12, 7, 6
    W1 = np.abs(rng.standard_normal((E, f, d))).astype(np.float32) + 4.0
    W3 = rng.standard_normal((E, f, d)).astype(np.float32)
    W2 = rng.standard_normal((E, d, f)).astype(np.float32)
    b1 = rng.standard_normal((E, f)).astype(np.float32)
    b2 = rng.standard_normal((E, d)).astype(np.float32)
    x = np.abs(rng.standard_normal((n, d))) + 1.0
    ex = np.array([0, 1, 2, 2, 1, 0], np.int32)
    T = lambda a: torch.from_numpy(a)
    yg = oracle.expert_ffn(x, ex, T(W1), None, T(W2), T(b1), T(b2), act=oracle.GELU_TANH)
    ys = oracle.expert_ffn(x, ex, T(W1), T(W3), T(W2), act=oracle.SWIGLU)
    W1d, W3d, W2d = W1.astype(np.float64), W3.astype(np.float64), W2.astype(np.float64)
    for r in range(n):
        e = ex[r]
        a = W1d[e] @ x[r]
        assert a.min() > 40
        ref_g = W2d[e] @ (a + b1[e]) + b2[e]
        ref_s = W2d[e] @ (a * (W3d[e] @ x[r]))
        np.testing.assert_allclose(yg[r], ref_g, rtol=1e-12, atol=1e-9)
        np.testing.assert_allclose(ys[r], ref_s, rtol=1e-12, atol=1e-9)


def test_expert_mlp_dead_regime_gives_output_bias():
    rng = np.random.default_rng(10)
    E, f, d = 2, 6, 5
    W1 = -np.abs(rng.standard_normal((E, f, d))).astype(np.float32) - 10.0
    W2 = rng.standard_normal((E, d, f)).astype(np.float32)
    b2 = rng.standard_normal((E, d)).astype(np.float32)
    x = np.abs(rng.standard_normal((3, d))) + 1.0
    ex = np.array([1, 0, 1], np.int32)
    y = oracle.expert_ffn(x, ex, torch.from_numpy(W1), None, torch.from_numpy(W2),
                          torch.zeros(E, f), torch.from_numpy(b2), act=oracle.GELU_TANH)
    np.testing.assert_allclose(y, b2[ex].astype(np.float64), atol=1e-12)


def test_expert_mlp_general_regime_within_activation_bound():
    """Moderate pre-activations: compare against numpy with the exact (erf) GELU; the difference is
    bounded by the tanh form's approximation error times the row sums of |W2|."""
    rng = np.random.default_rng(11)
    E, f, d, n = 4, 32, 16, 10
    W1, _, W2 = _mlp_inputs(rng, E, f, d)
    x = rng.standard_normal((n, d))
    ex = rng.integers(0, E, n).astype(np.int32)
    y = oracle.expert_ffn(x, ex, W1, None, W2, act=oracle.GELU_TANH)
    W1d, W2d = W1.double().numpy(), W2.double().numpy()
    for r in range(n):
        a = W1d[ex[r]] @ x[r]
        ref = W2d[ex[r]] @ (a * scipy.special.ndtr(a))
        bound = 5e-4 * np.abs(W2d[ex[r]]).sum(1)
        assert np.all(np.abs(y[r] - ref) <= bound)


def test_expert_mlp_reads_bf16_weights_exactly():
    rng = np.random.default_rng(12)
    E, f, d = 2, 8, 8
    W1, W3, W2 = _mlp_inputs(rng, E, f, d, torch.bfloat16)
    x = rng.standard_normal((4, d))
    ex = np.array([0, 1, 1, 0], np.int32)
    y16 = oracle.expert_ffn(x, ex, W1, W3, W2, act=oracle.SWIGLU)
    y32 = oracle.expert_ffn(x, ex, W1.float(), W3.float(), W2.float(), act=oracle.SWIGLU)
    np.testing.assert_array_equal(y16, y32)


# ---------------------------------------------------------------------------------------------
# combine and the whole layer

def test_combine_reproduces_printed_worked_example(golden):
    g = golden("lensa_step3_worked_combine.txt")
    gates = np.array([g["gates"]])
    yslot = np.array([[g["E3_h"], g["E4_h"]]])
    y = oracle.combine(gates, yslot)
    assert np.round(y[0], 2).tolist() == pytest.approx(g["y"], abs=1e-12)


def test_k_equals_E_renorm_equals_dense_mixture():
    """With k = E every expert runs, the renormalised gates are the full softmax, and the layer is
    the dense mixture sum_e p_e FFN_e(h), evaluated here expert by expert."""
    rng = np.random.default_rng(13)
    T, d, f, E = 6, 8, 16, 4
    h = torch.from_numpy(rng.standard_normal((T, d)).astype(np.float32))
    Wr = torch.from_numpy(rng.standard_normal((d, E)).astype(np.float32))
    W1, W3, W2 = _mlp_inputs(rng, E, f, d)
    z, p = oracle.router(h, Wr)
    idx, _, _ = oracle.topk(z, E)
    g = oracle.gates(z, p, idx, oracle.RENORM)
    y = oracle.forward_rows(np.arange(T), h, idx, g, W1, W3, W2, act=oracle.SWIGLU)
    dense = np.zeros((T, d))
    hx = h.numpy().astype(np.float64)
    for e in range(E):
        ye = oracle.expert_ffn(hx, np.full(T, e, np.int32), W1, W3, W2, act=oracle.SWIGLU)
        dense += p[:, e:e + 1] * ye
    np.testing.assert_allclose(y, dense, rtol=1e-12, atol=1e-12)


def test_forward_rows_subset_is_rowwise():
    w = wl.small(T=40, d=16, f=32, E=5, k=2, act=wl.ACT_GELU_TANH, dtype="f32", has_bias=True)
    inp = wl.random_biases(w, wl.generate(w), seed=3)
    full = oracle.reference(w, inp)
    sub = np.array([0, 7, 39, 21])
    part = oracle.reference(w, inp, tokens=sub)
    np.testing.assert_array_equal(part["y"], full["y"][sub])
    # and the row equals the explicit sum of gated expert outputs
    hx = inp["h"].numpy().astype(np.float64)
    for r, t in enumerate(sub):
        ys = oracle.expert_ffn(np.repeat(hx[t:t + 1], 2, 0), full["idx"][t], inp["W1"], None,
                               inp["W2"], inp["b1"], inp["b2"], act=oracle.GELU_TANH)
        np.testing.assert_allclose(part["y"][r], full["g"][t] @ ys, rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------------------------
# parameter counts printed by the pages

def test_micro_parameter_counts(golden):
    g = golden("param_counts.txt")
    d, L, f, E, k = int(g["micro_d"]), int(g["micro_layers"]), int(g["micro_f"]), int(g["micro_E"]), int(g["micro_k"])
    attn = 4 * d * d
    tot, act = oracle.param_count(L, d, f, E, k, 2, attn, 0)
    assert (tot, act) == (4_460_544, 1_314_816)
    assert round(tot / 1e6, 2) == g["micro_total_millions"]
    assert round(act / 1e6, 2) == g["micro_active_millions_alt"]
    assert round(tot / act, 2) == g["micro_ratio"]
    # with two LayerNorms per block and a final one (weight and bias each)
    tot_n, act_n = oracle.param_count(L, d, f, E, k, 2, attn + 2 * 2 * d, 2 * d)
    assert round(tot_n / 1e6, 2) == g["micro_total_millions"]
    assert round(act_n / 1e6, 2) == g["micro_active_millions"]
    assert round(tot_n / act_n, 2) == g["micro_ratio"]
    t64, a64 = oracle.param_count(L, d, f, 64, k, 2, attn, 0)
    assert round(t64 / a64, 1) == g["micro_E64_ratio"]


def test_7b_what_if_and_mixtral_counts(golden):
    g = golden("param_counts.txt")
    d, f = int(g["b7_d"]), int(g["b7_f"])
    assert round(3 * d * f / 1e6) == g["b7_expert_millions"]
    vocab = 32000
    per_layer = 4 * d * d + 2 * d                 # attention projections + two RMSNorm weights
    shared = 2 * vocab * d + d                    # input/output embeddings + final norm
    tot, act = oracle.param_count(int(g["b7_layers"]), d, f, int(g["b7_E"]), int(g["b7_k"]), 3,
                                  per_layer, shared)
    assert round(tot / 1e9, 1) == g["b7_total_billions"]
    assert round(act / 1e9, 1) == g["b7_active_billions"]
    assert round(tot / act, 1) == g["b7_ratio"]
    # E = 1 (the dense model) gives the familiar 6.74B
    t1, _ = oracle.param_count(32, d, f, 1, 1, 3, per_layer, shared)
    assert round(t1 / 1e9, 2) == 6.74
    md, mf = int(g["mixtral_d"]), int(g["mixtral_f"])
    assert round(3 * md * mf / 1e6) == g["mixtral_expert_millions"]
    assert round(int(g["mixtral_layers"]) * int(g["mixtral_E"]) * 3 * md * mf / 1e9, 1) == \
        g["mixtral_routed_billions"]


# ---------------------------------------------------------------------------------------------
# the synthetic workloads themselves

def test_decode_seed_routes_to_every_expert():
    w = wl.WORKLOADS["decode"]
    inp = wl.generate_router_inputs(w)
    r = oracle.route(w, inp)
    assert (r["counts"] > 0).all(), r["counts"]
    assert r["counts"].sum() == w.P


def test_many_small_routing_is_skewed_with_idle_experts():
    w = wl.WORKLOADS["many_small"]
    inp = wl.generate_router_inputs(w)
    r = oracle.route(w, inp)
    assert r["counts"].sum() == w.P
    assert (r["counts"] == 0).sum() >= 1
    assert r["counts"].max() > 4 * w.P / w.E


# ---------------------------------------------------------------------------------------------
# capacity and dropped slots (lensaml.com explainer, Step 5)

def _routing_with_demand(demand, T):
    labels = np.repeat(np.arange(len(demand)), demand)
    assert len(labels) == 2 * T and max(demand) <= T
    return np.stack([labels[:T], labels[T:]], axis=1).astype(np.int32)


def test_capacity_reproduces_printed_step5_example(golden):
    g = golden("lensa_step5_capacity.txt")
    T, k, E = int(g["T"]), int(g["k"]), int(g["E"])
    C = oracle.capacity(g["factor"], T, k, E)
    assert C == g["capacity"] == 64
    kept_printed = [int(x) for x in g["kept"]]
    demand = [kk + int(o) for kk, o in zip(kept_printed, g["overflow"])]
    assert demand == [104, 104, 78, 55, 50, 46, 50, 25] and sum(demand) == T * k
    idx = _routing_with_demand(demand, T)
    counts, offsets, st, so = oracle.dispatch_capacity(idx, E, C)
    assert counts.tolist() == demand
    assert np.diff(offsets).tolist() == kept_printed
    dropped = int((so < 0).sum())
    assert dropped == g["dropped"] == 94
    assert round(dropped / (T * k), 3) == g["dropped_share"]


@pytest.mark.parametrize("factor", [0.25, 0.5, 1.0, 1.25, 2.0])
def test_capacity_keeps_the_first_C_slots_in_token_order(factor):
    rng = np.random.default_rng(int(factor * 100))
    T, E, k = 300, 6, 2
    z = rng.standard_normal((T, E)) + np.array([2.0, 1.0, 0.5, 0, 0, -1.0])
    idx, _, _ = oracle.topk(z, k)
    C = oracle.capacity(factor, T, k, E)
    assert C == int(np.floor(factor * T * k / E))
    counts, offsets, st, so = oracle.dispatch_capacity(idx, E, C)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(np.minimum(counts, C))]))
    for e in range(E):
        slots = [s for s in range(T * k) if flat[s] == e]      # token order
        kept, dropped = slots[:C], slots[C:]
        assert [so[s] for s in kept] == list(range(offsets[e], offsets[e] + len(kept)))
        assert all(so[s] == -1 for s in dropped)
        assert st[offsets[e]:offsets[e + 1]].tolist() == [s // k for s in kept]


def test_capacity_unlimited_equals_dropless_and_zero_drops_all():
    rng = np.random.default_rng(21)
    idx, _, _ = oracle.topk(rng.standard_normal((77, 9)), 3)
    ref = oracle.dispatch(idx, 9)
    big = oracle.dispatch_capacity(idx, 9, 77 * 3)
    none = oracle.dispatch_capacity(idx, 9, -1)
    for a, b, c in zip(ref, big, none):
        np.testing.assert_array_equal(a, b)
        np.testing.assert_array_equal(a, c)
    counts, offsets, st, so = oracle.dispatch_capacity(idx, 9, 0)
    np.testing.assert_array_equal(counts, ref[0])
    assert offsets[-1] == 0 and (so == -1).all()


def test_dropped_slots_contribute_nothing():
    w = wl.small(T=50, d=16, f=32, E=4, k=2, act=wl.ACT_GELU_TANH, dtype="f32", has_bias=True,
                 router_bias_var=4.0, capacity_factor=0.75)
    inp = wl.random_biases(w, wl.generate(w), seed=9)
    ref = oracle.reference(w, inp)
    keep = (ref["slot_of"] >= 0).reshape(w.T, w.k)
    assert 0 < keep.sum() < w.P
    hx = inp["h"].numpy().astype(np.float64)
    for t in range(w.T):
        ys = oracle.expert_ffn(np.repeat(hx[t:t + 1], 2, 0), ref["idx"][t], inp["W1"], None,
                               inp["W2"], inp["b1"], inp["b2"], act=oracle.GELU_TANH)
        expect = (ref["g"][t] * keep[t]) @ ys
        np.testing.assert_allclose(ref["y"][t], expect, rtol=1e-13, atol=1e-14)
        if not keep[t].any():
            assert (ref["y"][t] == 0).all()
    # the auxiliary value uses the routed (pre-drop) counts
    assert ref["counts"].sum() == w.P


# ---------------------------------------------------------------------------------------------
# router z-loss (ST-MoE, named by arjunjaggi.com) and the selection-only routing bias
# (DeepSeek-V3, named by lensaml.com Step 4); the formulas are the cited papers'

def test_zloss_closed_forms():
    E = 8
    # all logits equal to c: log-sum-exp = c + ln E
    for c in (0.0, 1.5, -3.0):
        z = np.full((5, E), c)
        assert oracle.zloss(z) == pytest.approx((c + np.log(E)) ** 2, rel=1e-15)
    # one expert: log-sum-exp is the logit itself
    z1 = np.array([[0.5], [-2.0], [3.0]])
    assert oracle.zloss(z1) == pytest.approx(np.mean(z1[:, 0] ** 2), rel=1e-15)
    # one dominant logit: log-sum-exp -> that logit (the others add exp(-60) terms)
    z = np.zeros((1, 4))
    z[0, 2] = 60.0
    assert oracle.zloss(z) == pytest.approx(60.0 ** 2, rel=1e-15)
    assert oracle.zloss(np.zeros((0, 4))) == 0.0


def test_zloss_matches_scipy_logsumexp():
    from scipy.special import logsumexp
    rng = np.random.default_rng(31)
    z = rng.standard_normal((200, 13)) * 4.0
    assert oracle.zloss(z) == pytest.approx(np.mean(logsumexp(z, axis=1) ** 2), rel=1e-13)


def test_biased_selection_brute_force_and_unbiased_gates():
    """The chosen set is the unique S with min over S of p + b > max outside S (random keys have
    no ties); the gates are the unbiased ones: RENORM = p_j / sum_S p, RAW_PROB = p_j."""
    rng = np.random.default_rng(33)
    for E, k in [(4, 1), (5, 2), (6, 3), (6, 5)]:
        z = rng.standard_normal((40, E))
        p = np.exp(z - z.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        b = rng.standard_normal(E) * 0.3
        key = oracle.selection_keys(p, b)
        np.testing.assert_array_equal(key, p + b)
        idx, _, _ = oracle.topk(key, k)
        for t in range(40):
            best = [S for S in itertools.combinations(range(E), k)
                    if min(key[t, list(S)]) > max([key[t, e] for e in range(E) if e not in S],
                                                  default=-np.inf)]
            assert len(best) == 1 and set(idx[t]) == set(best[0])
            assert list(idx[t]) == sorted(idx[t], key=lambda e: -key[t, e])
        g = oracle.gates(z, p, idx, oracle.RENORM)
        ps = np.take_along_axis(p, idx, 1)
        np.testing.assert_allclose(g, ps / ps.sum(1, keepdims=True), rtol=1e-13)
        np.testing.assert_allclose(oracle.gates(z, p, idx, oracle.RAW_PROB), ps, rtol=0, atol=0)


def test_biased_selection_special_cases():
    rng = np.random.default_rng(34)
    z = rng.standard_normal((64, 6))
    p = np.exp(z) / np.exp(z).sum(1, keepdims=True)
    # no bias: the same choice as by the logits (softmax is monotone)
    np.testing.assert_array_equal(oracle.topk(oracle.selection_keys(p, np.zeros(6)), 2)[0],
                                  oracle.topk(z, 2)[0])
    # a bias above 1 puts its expert first for every token; one below -1 keeps it out
    b = np.zeros(6)
    b[4], b[1] = 2.0, -2.0
    idx = oracle.topk(oracle.selection_keys(p, b), 3)[0]
    assert (idx[:, 0] == 4).all() and not (idx == 1).any()


def test_sel_bias_update_rule():
    counts = np.array([5, 2, 3, 6], np.int32)          # T k = 16, mean load 4
    out = oracle.update_sel_bias(counts, T=8, k=2, gamma=0.125, b=[0.0, 1.0, -1.0, 0.5])
    np.testing.assert_array_equal(out, [-0.125, 1.125, -0.875, 0.375])
    even = oracle.update_sel_bias(np.array([4, 4, 4, 4], np.int32), T=8, k=2, gamma=0.3, b=[0.1] * 4)
    np.testing.assert_array_equal(even, [0.1] * 4)


def test_route_with_sel_bias_keeps_unbiased_p_and_aux():
    w = wl.small(T=120, d=32, f=32, E=6, k=2, act=wl.ACT_GELU_TANH, dtype="f32")
    inp = wl.generate(w)
    plain = oracle.route(w, inp)
    b = np.array([0.3, 0, 0, 0, -0.3, 0.1])
    biased = oracle.route(w, dict(inp, sel_bias=torch.tensor(b, dtype=torch.float32)))
    np.testing.assert_array_equal(plain["p"], biased["p"])
    assert plain["zloss"] == biased["zloss"]
    assert (biased["counts"][0] > plain["counts"][0]) and (biased["counts"][4] < plain["counts"][4])
    assert biased["aux"] == pytest.approx(oracle.aux_loss(biased["counts"], biased["p"], w.k))

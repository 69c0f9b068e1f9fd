"""GPU parity: libmoe (through its C ABI) against the double-precision oracle, on the same seeded
inputs. Indices, counts and the permutation are compared bit for bit (outside near ties); the
layer output within max-abs 1e-4 (f32) or relative L2 1e-2 (bf16)."""
import numpy as np
import pytest
import torch

import oracle
from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import workloads as wl

from parity import (AUX_REL, GATE_ABS, check_dispatch_valid, check_layer_output, rel_l2,
                    routing_agreement, run_forward, run_steps, to_dev)

pytestmark = pytest.mark.gpu

G, S = wl.ACT_GELU_TANH, wl.ACT_SWIGLU

SMALL = [
    wl.small("single_expert", T=1, d=64, f=64, E=1, k=1),
    wl.small("k_equals_E", T=37, d=64, f=128, E=4, k=4),
    wl.small("ragged_swiglu", T=300, d=192, f=320, E=6, k=2),
    wl.small("ragged_gelu_bias_f32", T=133, d=128, f=192, E=5, k=2, act=G, dtype="f32",
             has_bias=True),
    wl.small("f32_swiglu", T=200, d=128, f=256, E=8, k=2, dtype="f32"),
    # f32 FFN with its 64 x 64 tiles (at least two blocks per SM): GEMM1 only (GELU with biases,
    # SwiGLU), and both GEMMs with skewed loads
    wl.small("f32_big_tiles_gelu_bias", T=2048, d=128, f=512, E=4, k=2, act=G, dtype="f32",
             has_bias=True),
    wl.small("f32_big_tiles_swiglu", T=1100, d=256, f=512, E=6, k=2, dtype="f32"),
    wl.small("f32_big_tiles_both", T=4000, d=256, f=256, E=4, k=2, dtype="f32",
             router_bias_var=2.0),
    wl.small("gelu_bias_raw_prob", T=517, d=256, f=512, E=16, k=1, act=G,
             gate=wl.GATE_RAW_PROB, has_bias=True),
    wl.small("skewed_idle", T=1000, d=128, f=256, E=32, k=4, router_bias_var=8.0),
    wl.small("many_chunks", T=5000, d=64, f=64, E=64, k=4),
    wl.small("wide_E", T=700, d=128, f=128, E=256, k=8),
    wl.small("several_tiles", T=1100, d=512, f=768, E=3, k=2),
    # router paths: tensor-core router with E padded to 48 and 112, small router with E = 20
    wl.small("tc_router_E40", T=600, d=256, f=128, E=40, k=3, router_bias_var=1.0),
    wl.small("tc_router_E100_raw_prob", T=300, d=128, f=128, E=100, k=1, act=G,
             gate=wl.GATE_RAW_PROB),
    wl.small("small_router_E20_f32", T=77, d=320, f=64, E=20, k=5, dtype="f32"),
    # tensor-core logits: E = 32 (two accumulator chains), E = 8 with d split over two K chunks;
    # token counts not a multiple of the 128-token tile
    wl.small("tc_router_E32_chains", T=2000, d=256, f=128, E=32, k=2, router_bias_var=1.0),
    wl.small("tc_router_E8_ksplit", T=1500, d=512, f=128, E=8, k=2),
    wl.small("smem_router_f32_many_tokens", T=1500, d=320, f=64, E=8, k=2, dtype="f32"),
    # capacity factor (drops): single-chunk and multi-chunk dispatch, f32 and bf16, everything
    # dropped (C = 0)
    wl.small("capacity_skewed_k2", T=800, d=128, f=256, E=8, k=2, router_bias_var=4.0,
             capacity_factor=1.0),
    wl.small("capacity_switch_gelu", T=3000, d=128, f=128, E=16, k=1, act=G,
             gate=wl.GATE_RAW_PROB, has_bias=True, router_bias_var=2.0, capacity_factor=1.25),
    wl.small("capacity_f32", T=200, d=64, f=128, E=4, k=2, dtype="f32", router_bias_var=2.0,
             capacity_factor=0.5),
    wl.small("capacity_zero", T=100, d=64, f=64, E=8, k=2, capacity_factor=0.02),
    # paired-CTA GEMM (experts of >= 4 M tiles): odd tile counts, ragged N tail, skew
    wl.small("paired_gelu_bias", T=2500, d=256, f=320, E=3, k=2, act=G, has_bias=True),
    wl.small("paired_swiglu_skewed", T=3000, d=128, f=256, E=4, k=2, router_bias_var=3.0),
    # selection-only routing bias (experts chosen by p + b, gates from p) on every router path:
    # few-token split-d (bf16), shared-memory W_r (f32), tiled (f32, E > 32), tensor cores
    wl.small("sel_bias_splitd", T=300, d=256, f=128, E=16, k=2, sel_bias_std=0.05),
    wl.small("sel_bias_small_f32", T=1500, d=128, f=64, E=8, k=2, dtype="f32", sel_bias_std=0.1),
    wl.small("sel_bias_tile_f32", T=200, d=128, f=64, E=40, k=3, dtype="f32", sel_bias_std=0.02),
    wl.small("sel_bias_tc", T=2000, d=256, f=128, E=64, k=4, router_bias_var=1.0,
             sel_bias_std=0.01),
    wl.small("sel_bias_tc_top1_raw", T=1800, d=128, f=128, E=100, k=1, act=G,
             gate=wl.GATE_RAW_PROB, sel_bias_std=0.01),
    # the largest k (32) on the tensor-core and tiled router paths; E = 256 with a selection bias
    # on the bf16 tiled router
    wl.small("k32_tc", T=400, d=128, f=64, E=64, k=32, router_bias_var=1.0),
    wl.small("k32_tile_f32", T=150, d=64, f=64, E=48, k=32, dtype="f32"),
    wl.small("e256_sel_bias_tile", T=600, d=128, f=64, E=256, k=8, sel_bias_std=0.002),
    # paired kernel on an expert's odd last M tile (the second CTA's rows all masked): E = 1,
    # k = 1 and E = 2, k = 2 fix the rows per expert at T, so the last tile holds 40, 100 or 128
    # rows; SwiGLU with a ragged last N tile, GELU with biases, the top-1 scatter, and the
    # fused gather
    wl.small("pair_half_tail40_swiglu", T=552, d=256, f=320, E=1, k=1),
    wl.small("pair_half_tail100_gelu", T=868, d=192, f=256, E=1, k=1, act=G, has_bias=True,
             gate=wl.GATE_RAW_PROB),
    wl.small("pair_half_tail128_k2", T=640, d=128, f=384, E=2, k=2),
    wl.small("pair_half_gather", T=552, d=128, f=256, E=2, k=2, fuse_gather=True),
    # paired GEMM with more units than clusters and a partial last wave (308 / 88 units of
    # 256 x 256 for the SwiGLU layer, 200 / 80 for the top-1 GELU layer with biases and the fused
    # scatter) and long K loops (d = 1024, f = 1792 / 2560)
    wl.small("split_tail_swiglu_k2", T=2600, d=1024, f=1792, E=2, k=2),
    wl.small("split_tail_gelu_top1", T=5120, d=1024, f=2560, E=1, k=1, act=G, has_bias=True,
             gate=wl.GATE_RAW_PROB),
    # a paired GELU GEMM1 with biases whose 80 units leave a last wave of 6 on 74 clusters
    wl.small("pair_partial_wave_gelu", T=5120, d=256, f=1024, E=1, k=1, act=G, has_bias=True,
             gate=wl.GATE_RAW_PROB, seed=19),
    # moe_forward with GEMM1 gathering its rows of h (single-CTA and paired kernels, ragged row
    # counts that leave part of a 4-row gather past an expert's end), with and without top-1 scatter
    wl.small("gather_ragged_k3", T=301, d=192, f=320, E=5, k=3, fuse_gather=True),
    wl.small("gather_paired_gelu_bias", T=2500, d=256, f=320, E=3, k=2, act=G, has_bias=True,
             fuse_gather=True),
    wl.small("gather_top1_scatter", T=999, d=128, f=256, E=6, k=1, act=G, gate=wl.GATE_RAW_PROB,
             has_bias=True, router_bias_var=1.0, fuse_gather=True),
    # experts averaging two to three M tiles on the single-CTA kernel, with skewed routing (one
    # expert of 27 rows next to experts of three or four tiles): the top-1 GELU layer with
    # biases and the fused scatter over a ragged last N tile (f = 640), and SwiGLU with ragged
    # K and N (d = 320)
    wl.small("multi_tile_gelu_bias_top1", T=900, d=256, f=640, E=4, k=1, act=G,
             has_bias=True, gate=wl.GATE_RAW_PROB, router_bias_var=2.0, seed=41),
    wl.small("multi_tile_swiglu_k2", T=700, d=320, f=384, E=4, k=2, router_bias_var=2.0,
             seed=42),
]


def _inputs(w):
    inp = wl.generate(w)
    if w.has_bias:
        inp = wl.random_biases(w, inp, seed=w.seed + 100)
    return inp


def _fused_scatter(w) -> bool:
    return w.dtype == "bf16" and w.k == 1 and w.capacity_factor == 0


def _check_steps(w, inputs, ref, got):
    assert got["status"] == B.MOE_OK, B.status_string(got["status"])
    idx = got["idx"].numpy()
    diff = routing_agreement(ref, idx)
    keep = np.setdiff1d(np.arange(w.T), diff)
    np.testing.assert_allclose(got["gates"].numpy()[keep], ref["g"][keep], rtol=0, atol=GATE_ABS)
    counts, offsets = got["counts"].numpy(), got["offsets"].numpy()
    st, so = got["sorted_token"].numpy(), got["slot_of"].numpy()
    kept = int(offsets[-1])
    if len(diff) == 0:
        np.testing.assert_array_equal(counts, ref["counts"])
        np.testing.assert_array_equal(offsets, ref["offsets"])
        np.testing.assert_array_equal(st[:kept], ref["sorted_token"][:kept])
        np.testing.assert_array_equal(so, ref["slot_of"])
    else:
        check_dispatch_valid(idx, w.E, counts, offsets, st, so, ref["capacity"])
    # the permute is a copy: bit-exact
    assert torch.equal(got["x_perm"][:kept], inputs["h"][torch.from_numpy(st[:kept]).long()])
    assert got["aux"].item() == pytest.approx(ref["aux"], rel=AUX_REL)
    assert got["zloss"].item() == pytest.approx(ref["zloss"], rel=AUX_REL)
    return diff


def _check_expert_rows(w, inputs, got, rows):
    """y_perm rows against the oracle's expert MLP applied to the same (exact) x_perm rows."""
    offsets = got["offsets"].numpy()
    expert_of_row = np.searchsorted(offsets, rows, side="right") - 1
    x = got["x_perm"][torch.from_numpy(rows).long()].double().numpy()
    yr = oracle.expert_ffn(x, expert_of_row.astype(np.int32), inputs["W1"], inputs.get("W3"),
                           inputs["W2"], inputs.get("b1"), inputs.get("b2"), oracle.act_code(w))
    yg = got["y_perm"][torch.from_numpy(rows).long()].double().numpy()
    if w.dtype == "f32":
        assert np.abs(yg - yr).max() <= 1e-4
    else:
        assert rel_l2(yg, yr) <= 1e-2


def _random_case(seed: int):
    """A seeded random layer shape and variant within the library's limits, small enough for the
    oracle to check every output."""
    rng = np.random.default_rng(1000 + seed)
    dtype = "f32" if rng.random() < 0.3 else "bf16"
    act = G if rng.random() < 0.5 else S
    E = int(rng.integers(1, 41))
    k = int(rng.integers(1, min(E, 8) + 1))
    return wl.small(
        f"random_{seed}", T=int(rng.integers(1, 900)), d=64 * int(rng.integers(1, 6)),
        f=64 * int(rng.integers(1, 9)), E=E, k=k, act=act,
        gate=wl.GATE_RAW_PROB if rng.random() < 0.3 else wl.GATE_RENORM, dtype=dtype,
        has_bias=bool(act == G and rng.random() < 0.5),
        router_bias_var=float(rng.choice([1.0, 4.0])) if rng.random() < 0.4 else None,
        seed=int(rng.integers(1, 10_000)),
        capacity_factor=float(rng.choice([0.5, 1.0, 1.25])) if rng.random() < 0.3 else 0.0,
        sel_bias_std=0.01 if rng.random() < 0.2 else 0.0)


RANDOM = [_random_case(i) for i in range(32)]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_cases_step_by_step(w):
    _check_case(w)


@pytest.mark.parametrize("w", RANDOM, ids=lambda w: w.name)
def test_random_shapes_step_by_step(w):
    """32 seeded random shapes and variants (dtype, activation, gate mode, biases, router bias,
    capacity, selection bias; T < 900, E <= 40, k <= 8)."""
    _check_case(w)


def _check_case(w):
    inputs = _inputs(w)
    ref = oracle.reference(w, inputs)
    dev = to_dev(inputs)
    got = run_steps(w, inputs, dev)
    diff = _check_steps(w, inputs, ref, got)
    kept = int(got["offsets"][-1])
    rows = np.arange(kept) if kept <= 4096 else np.unique(np.linspace(0, kept - 1, 2048).astype(int))
    if kept:
        _check_expert_rows(w, inputs, got, rows)
    if w.capacity_factor > 0:
        print(f"{w.name}: capacity {ref['capacity']}, kept {kept} of {w.P} slots")
        if kept == 0:
            assert (got["y"].float() == 0).all()
    check_layer_output(w, ref, got["y"], skip_tokens=diff)
    # moe_forward gathers its GEMM1 rows from h directly (same bytes as x_perm): identical bits,
    # except where a dropless top-1 bf16 layer also fuses the combine into GEMM2 (one bf16
    # rounding fewer), which is checked against the oracle instead
    fw = run_forward(w, dev)
    assert fw["status"] == B.MOE_OK
    if _fused_scatter(w):
        check_layer_output(w, ref, fw["y"], skip_tokens=diff)
    else:
        assert torch.equal(fw["y"], got["y"])
    assert torch.equal(fw["idx"], got["idx"]) and torch.equal(fw["counts"], got["counts"])
    assert fw["aux"].item() == got["aux"].item()
    assert fw["zloss"].item() == got["zloss"].item()


def _token_sample(w):
    if w.T <= 256:
        return np.arange(w.T)
    n = {"mixtral": 256, "many_small": 256, "switch": 512}.get(w.name, 128)
    edge = max(n // 4, 4)
    mid = np.linspace(edge, w.T - edge - 1, n - 2 * edge).astype(np.int64)
    return np.unique(np.concatenate([np.arange(edge), mid, np.arange(w.T - edge, w.T)]))


def _tile_rows(offsets: np.ndarray, bm: int = 128) -> np.ndarray:
    """Rows of y_perm that touch every 128-row M tile of every expert: its first and last valid
    row and one row in each 32-row quarter (the four TMEM lane quarters of a tile's
    accumulator), so every tile's masked store and every epilogue warp's rows are compared."""
    rows = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for r0 in range(lo, hi, bm):
            last = min(r0 + bm, hi) - 1
            rows += [r0, last] + [r0 + 32 * q + 17 for q in range(4) if r0 + 32 * q + 17 <= last]
    return np.unique(np.array(rows, dtype=np.int64))


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_full_size_workloads(name):
    """The five workloads at full size, through moe_forward (the call the benchmark times) and
    through the five step calls: routing, counts and permutation over all tokens; the expert MLP
    output on rows of every M tile of every expert; the layer output on a deterministic token
    sample (every token for micro and decode)."""
    w = wl.WORKLOADS[name]
    inputs = _inputs(w)
    tokens = _token_sample(w)
    ref = oracle.reference(w, inputs, tokens=tokens)
    dev = to_dev(inputs)
    fw = run_forward(w, dev)
    assert fw["status"] == B.MOE_OK
    idx_fw = fw["idx"].numpy()
    diff = routing_agreement(ref, idx_fw)
    # the fused call's counts are those of its own routing, whether or not there are near ties
    np.testing.assert_array_equal(fw["counts"].numpy(), np.bincount(idx_fw.ravel(), minlength=w.E))
    if len(diff) == 0:
        np.testing.assert_array_equal(fw["counts"].numpy(), ref["counts"])
    assert fw["aux"].item() == pytest.approx(ref["aux"], rel=AUX_REL)
    assert fw["zloss"].item() == pytest.approx(ref["zloss"], rel=AUX_REL)
    stats = check_layer_output(w, ref, fw["y"], skip_tokens=diff)
    got = run_steps(w, inputs, dev)
    _check_steps(w, inputs, ref, got)
    assert torch.equal(got["idx"], fw["idx"]) and torch.equal(got["counts"], fw["counts"])
    rows = _tile_rows(got["offsets"].numpy())
    _check_expert_rows(w, inputs, got, rows)
    if _fused_scatter(w):
        check_layer_output(w, ref, got["y"], skip_tokens=diff)
    else:
        assert torch.equal(got["y"], fw["y"])
    if name == "decode":
        assert (got["counts"] > 0).all()
    print(f"{name}: near-tie tokens {len(diff)}, layer output {stats} on {len(tokens)} tokens, "
          f"expert rows checked {len(rows)} of {int(got['offsets'][-1])}")


LARGE = [
    # 2M slots: 1954 dispatch chunks, so the look-back runs over many rounds of co-resident blocks
    wl.small("many_slots", T=1_000_000, d=64, f=64, E=8, k=2, router_bias_var=1.0),
    # the largest E and k together over 640K slots (tiled router, k = 32 combine)
    wl.small("e256_k32_many", T=20_000, d=128, f=64, E=256, k=32),
    # long K: d = 8192 (GEMM1 with 128 K stages, few-token split-d router)
    wl.small("wide_d", T=300, d=8192, f=256, E=4, k=2),
]


@pytest.mark.parametrize("w", LARGE, ids=lambda w: w.name)
def test_large_cases(w):
    """Shapes at the edges of what the library takes, through moe_forward: routing, counts and
    aux over every token, the layer output on a deterministic token sample."""
    inputs = _inputs(w)
    tokens = oracle.sample_tokens(w.T, stride=max(1, w.T // 4096))
    ref = oracle.reference(w, inputs, tokens=tokens)
    dev = to_dev(inputs)
    fw = run_forward(w, dev)
    assert fw["status"] == B.MOE_OK
    diff = routing_agreement(ref, fw["idx"].numpy())
    if len(diff) == 0:
        np.testing.assert_array_equal(fw["counts"].numpy(), ref["counts"])
    assert fw["aux"].item() == pytest.approx(ref["aux"], rel=AUX_REL)
    stats = check_layer_output(w, ref, fw["y"], skip_tokens=diff)
    print(f"{w.name}: near-tie tokens {len(diff)}, {stats}")


@pytest.mark.parametrize("k,dtype", [(1, "bf16"), (2, "bf16"), (2, "f32")])
def test_every_token_to_one_expert(k, dtype):
    """A router bias of 50 on expert 5 sends every token's first choice there: one expert holds
    T rows (many GEMM tiles, every dispatch chunk a single expert), the others share the rest."""
    w = wl.small(f"one_hot_k{k}_{dtype}", T=3000, d=128, f=192, E=8, k=k, dtype=dtype,
                 act=G if k == 1 else S, gate=wl.GATE_RAW_PROB if k == 1 else wl.GATE_RENORM,
                 seed=77)
    inputs = _inputs(w)
    b = torch.zeros(w.E)
    b[5] = 50.0
    inputs["b_r"] = b
    ref = oracle.reference(w, inputs)
    assert ref["counts"][5] == w.T
    dev = to_dev(inputs)
    got = run_steps(w, inputs, dev)
    _check_steps(w, inputs, ref, got)
    assert int(got["counts"][5]) == w.T
    check_layer_output(w, ref, got["y"])
    fw = run_forward(w, dev)
    assert fw["status"] == B.MOE_OK
    check_layer_output(w, ref, fw["y"])
    assert fw["aux"].item() == pytest.approx(ref["aux"], rel=AUX_REL)


def test_empty_batch():
    w = wl.small("empty", T=0, d=64, f=64, E=4, k=2)
    cfg = B.config_for(w)
    ws = B.workspace(cfg)
    counts = torch.full((4,), 9, dtype=torch.int32, device="cuda")
    aux = torch.full((1,), 9.0, device="cuda")
    z = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    B.moe_forward(cfg, z, torch.zeros(64, 4, device="cuda"), None, z, None, z, z, None, z, aux,
                  None, counts, ws)
    assert B.moe_device_status(ws) == B.MOE_OK
    assert counts.cpu().tolist() == [0, 0, 0, 0] and aux.item() == 0.0


def test_outputs_stay_inside_their_buffers_and_runs_are_deterministic():
    w = wl.small("canary", T=333, d=128, f=192, E=12, k=3, router_bias_var=1.0)
    inputs = _inputs(w)
    dev = to_dev(inputs)
    cfg = B.config_for(w)
    ws = B.workspace(cfg)
    guard = 64
    ybuf = torch.full((w.T + 2 * guard, w.d), 7.0, dtype=torch.bfloat16, device="cuda")
    ibuf = torch.full((w.T * w.k + 2 * guard,), -5, dtype=torch.int32, device="cuda")
    cbuf = torch.full((w.E + 2 * guard,), -5, dtype=torch.int32, device="cuda")
    y = ybuf[guard:guard + w.T]
    idx = ibuf[guard:guard + w.T * w.k]
    cnt = cbuf[guard:guard + w.E]
    aux = torch.zeros(1, device="cuda")
    outs = []
    for _ in range(3):
        B.moe_forward(cfg, dev["h"], dev["W_r"], dev["b_r"], dev["W1"], None, dev["W3"],
                      dev["W2"], None, y, aux, idx, cnt, ws)
        assert B.moe_device_status(ws) == B.MOE_OK
        outs.append((y.clone(), idx.clone(), cnt.clone(), aux.clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    for a, b in zip(outs[0], outs[2]):
        assert torch.equal(a, b)
    assert (ybuf[:guard] == 7.0).all() and (ybuf[guard + w.T:] == 7.0).all()
    assert (ibuf[:guard] == -5).all() and (ibuf[guard + w.T * w.k:] == -5).all()
    assert (cbuf[:guard] == -5).all() and (cbuf[guard + w.E:] == -5).all()


def test_sel_bias_update_step():
    """moe_update_sel_bias moves each bias by +gamma below the mean load and -gamma above it
    (the oracle's rule, in f32), on the counts of a routed batch."""
    w = wl.small("update", T=700, d=128, f=64, E=10, k=3, router_bias_var=2.0, sel_bias_std=0.05)
    inputs = _inputs(w)
    dev = to_dev(inputs)
    got = run_steps(w, inputs, dev)
    counts = got["counts"].numpy()
    b = dev["sel_bias"].clone()
    B.moe_update_sel_bias(B.config_for(w), got["counts"].cuda(), b, 0.0078125)
    expect = oracle.update_sel_bias(counts, w.T, w.k, 0.0078125, inputs["sel_bias"].numpy())
    np.testing.assert_array_equal(b.cpu().numpy(), expect.astype(np.float32))
    assert (counts * w.E != w.P).any()

"""The seeded input generators (shared by the CUDA path and the oracle): deterministic, the
router inputs are the first draws of the full stream, and the value distributions are the stated
ones. CPU only, small shapes."""
import math

import torch

from sparse_mixture_experts_70_b300 import workloads as wl


def test_generate_is_deterministic_and_router_inputs_are_its_first_draws():
    w = wl.small(T=64, d=128, f=192, E=6, k=2, router_bias_var=2.0, seed=9)
    a, b = wl.generate(w), wl.generate(w)
    for key in a:
        if a[key] is None:
            assert b[key] is None
        else:
            assert torch.equal(a[key], b[key]), key
    r = wl.generate_router_inputs(w)
    for key in ("h", "W_r", "b_r"):
        assert torch.equal(r[key], a[key]), key
    other = wl.generate(w.with_(seed=10))
    assert not torch.equal(other["h"], a["h"])


def test_shapes_dtypes_and_scales():
    w = wl.small(T=4096, d=256, f=128, E=4, k=2, act=wl.ACT_SWIGLU, dtype="bf16", seed=3)
    x = wl.generate(w)
    assert x["h"].shape == (4096, 256) and x["h"].dtype == torch.bfloat16
    assert x["W_r"].dtype == torch.float32 and x["W_r"].shape == (256, 4)
    assert x["W1"].shape == (4, 128, 256) and x["W3"].shape == (4, 128, 256)
    assert x["W2"].shape == (4, 256, 128)
    assert x["b_r"] is None and x["b1"] is None and x["b2"] is None
    # h ~ N(0, 1); weights ~ N(0, 1/fan_in): W1 fan_in d, W2 fan_in f
    assert abs(x["h"].float().std().item() - 1.0) < 0.02
    assert abs(x["W1"].float().std().item() - 1 / math.sqrt(256)) < 0.002
    assert abs(x["W2"].float().std().item() - 1 / math.sqrt(128)) < 0.003
    g = wl.generate(wl.small(T=8, d=64, f=64, E=3, k=1, act=wl.ACT_GELU_TANH, dtype="f32",
                             has_bias=True))
    assert g["W3"] is None and g["h"].dtype == torch.float32
    assert torch.count_nonzero(g["b1"]) == 0 and torch.count_nonzero(g["b2"]) == 0


def test_the_five_workloads_have_their_stated_shapes():
    W = wl.WORKLOADS
    assert (W["micro"].T, W["micro"].d, W["micro"].f, W["micro"].E, W["micro"].k) == (256, 128, 512, 8, 2)
    assert (W["mixtral"].T, W["mixtral"].d, W["mixtral"].f, W["mixtral"].E, W["mixtral"].k) == (4096, 4096, 14336, 8, 2)
    assert (W["many_small"].T, W["many_small"].d, W["many_small"].f, W["many_small"].E,
            W["many_small"].k) == (16384, 2048, 1408, 64, 4)
    assert (W["switch"].T, W["switch"].d, W["switch"].f, W["switch"].E, W["switch"].k) == (32768, 1024, 4096, 128, 1)
    assert (W["decode"].T, W["decode"].d, W["decode"].f, W["decode"].E, W["decode"].k) == (32, 4096, 14336, 8, 2)
    assert W["micro"].dtype == "f32" and W["micro"].has_bias
    assert W["switch"].gate == wl.GATE_RAW_PROB and W["switch"].act == wl.ACT_GELU_TANH
    assert W["many_small"].router_bias_var == 2.0

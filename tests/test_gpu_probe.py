"""The FP32 FFMA probe that bench.py uses as the f32 layer's compute roof: its flop count is the
one stated in include/moe_probe.h, and the rate it gives lies within a plausible band of the
CUDA-core FFMA rate derived from the SM count and the SM clock (128 FP32 lanes per SM, 2 flops
per FMA)."""
import pytest
import torch

from sparse_mixture_experts_70_b300 import binding as B

pytestmark = pytest.mark.gpu


def test_ffma_probe_rate_is_plausible():
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    blocks, threads, iters = sms * 4, 512, 2048
    flops = B.moe_fp32_ffma_probe(blocks, threads, iters, out)
    assert flops == 2 * 8 * 16 * iters * blocks * threads
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(3):
        e0.record()
        B.moe_fp32_ffma_probe(blocks, threads, iters, out)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    rate = flops / (best * 1e-3)
    derived_max = sms * 128 * 2 * 2.2e9     # above the 2032 MHz maximum SM clock
    assert 0.25 * derived_max < rate < derived_max, (rate / 1e12, derived_max / 1e12)
    assert out.item() == 0.0                 # the guarded store never happens


def test_ffma_probe_rejects_bad_shapes():
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    for args in [(0, 256, 10), (148, 100, 10), (148, 2048, 10), (148, 256, 0)]:
        with pytest.raises(B.MoEError) as err:
            B.moe_fp32_ffma_probe(*args, out)
        assert err.value.status == B.MOE_ERR_INVALID_ARG

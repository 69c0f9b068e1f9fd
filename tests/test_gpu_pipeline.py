"""moe_pipeline_*: batches in host memory through the layer with overlapped copies. Every batch's
output must equal moe_forward on the same h, bit for bit (the layer computation is moe_forward;
only the copies differ)."""
import pytest
import torch

from sparse_mixture_experts_70_b300 import binding as B
from sparse_mixture_experts_70_b300 import workloads as wl

from parity import to_dev

pytestmark = pytest.mark.gpu

CASES = [
    wl.small("pipe_swiglu_k2", T=700, d=256, f=320, E=6, k=2),
    wl.small("pipe_top1_scatter", T=900, d=128, f=256, E=16, k=1, act=wl.ACT_GELU_TANH,
             gate=wl.GATE_RAW_PROB),
    wl.small("pipe_f32", T=130, d=128, f=192, E=5, k=2, act=wl.ACT_GELU_TANH, dtype="f32",
             has_bias=True),
]


def _batches(w, dev, n):
    g = torch.Generator().manual_seed(w.seed + 7)
    return [torch.randn(w.T, w.d, generator=g).to(w.torch_dtype).pin_memory() for _ in range(n)]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("side_stream", [False, True])
def test_pipeline_matches_forward(w, side_stream):
    inputs = wl.generate(w)
    if w.has_bias:
        inputs = wl.random_biases(w, inputs, seed=w.seed + 100)
    dev = to_dev(inputs)
    cfg = B.config_for(w)
    layer = B.Layer(cfg, dev)
    hs = _batches(w, dev, 7)
    expect = []
    for h in hs:
        layer.forward(h.cuda())
        expect.append((layer.y.cpu().clone(), layer.aux.cpu().clone()))
    assert B.moe_device_status(layer.ws) == B.MOE_OK

    stream = torch.cuda.Stream() if side_stream else torch.cuda.current_stream()
    ys = [torch.full((w.T, w.d), 3.0, dtype=w.torch_dtype).pin_memory() for _ in hs]
    auxs = [torch.full((1,), -1.0).pin_memory() for _ in hs]
    with B.Pipeline(cfg, dev, stream=stream) as pipe:
        for i in range(4):                      # first run of batches, then a join
            pipe.submit(hs[i], ys[i], auxs[i])
        pipe.join()
        stream.synchronize()
        for i in range(4):
            assert torch.equal(ys[i], expect[i][0]), i
            assert auxs[i].item() == expect[i][1].item()
        for i in range(4, 7):                   # the pipeline keeps working after a join
            pipe.submit(hs[i], ys[i], auxs[i])
        assert pipe.device_status() == B.MOE_OK
    for i in range(4, 7):
        assert torch.equal(ys[i], expect[i][0]), i
        assert auxs[i].item() == expect[i][1].item()


def test_pipeline_orders_after_the_callers_stream():
    """Work enqueued on the pipeline's stream before the first submit (here: writing h on the
    device and copying it to the host buffer the batch reads) completes before the copy-in."""
    w = wl.small("pipe_order", T=256, d=128, f=128, E=4, k=2)
    dev = to_dev(wl.generate(w))
    cfg = B.config_for(w)
    layer = B.Layer(cfg, dev)
    h_dev = torch.randn(w.T, w.d, device="cuda").to(torch.bfloat16)
    layer.forward(h_dev)
    expect = layer.y.cpu()
    stream = torch.cuda.Stream()
    h_host = torch.zeros(w.T, w.d, dtype=torch.bfloat16).pin_memory()
    y_host = torch.zeros(w.T, w.d, dtype=torch.bfloat16).pin_memory()
    aux = torch.zeros(1).pin_memory()
    torch.cuda.synchronize()
    with B.Pipeline(cfg, dev, stream=stream) as pipe:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(20_000_000)  # keep the stream busy so a missing fence would show
            h_host.copy_(h_dev, non_blocking=True)
        pipe.submit(h_host, y_host, aux)
        assert pipe.device_status() == B.MOE_OK
    assert torch.equal(y_host, expect)

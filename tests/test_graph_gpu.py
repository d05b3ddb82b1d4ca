"""Forward(graph=True): the layer replayed from a CUDA graph (GPU only).

The first call on a pair of x / y buffers runs eagerly and records the
library's launches into a graph; later calls replay it.  A replay must give
exactly the eager call's output and statistics (bit for bit) for new
contents of the same input buffer, a new buffer pair must get its own graph,
and the device status must stay clean.  Covers the decode path (one block per
token router with the grouping in its last block, split-K up GEMM finishing
its SwiGLU in the last slice's CTA), FP8 weights, expert choice, a capacity
cut with statistics, and the host pipeline on top of a graph Forward.
"""
import pytest
import torch

from moe_inputs import Workload

pytestmark = pytest.mark.gpu

CASES = [
    Workload("graph_decode_t1", T=1, d=512, E=8, F=512, k=2),
    Workload("graph_decode_t5_shared", T=5, d=256, E=16, F=320, k=2, n_shared=1, F_s=192, select_bias=True),
    Workload("graph_prefill_capacity", T=600, d=256, E=16, F=256, k=2, capacity=70, zipf_s=1.2),
    Workload("graph_fp8_decode", T=3, d=256, E=8, F=384, k=2, weights="fp8"),
    Workload("graph_expert_choice", T=64, d=256, E=8, F=256, k=2, routing="expert"),
]


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_layer_95_b300 as moe
    moe.lib()
    return torch.device("cuda")


def _forwards(w):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    layer = layer_of(w)
    L = moe_inputs.make_layer(w, "cuda")
    q8 = None
    if w.weights == "fp8":
        q8 = moe.quantize_experts_fp8(layer, L["w1"], L["w3"], L["w2"])
    args = (layer, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"], L["ws1"], L["ws3"],
            L["ws2"])
    eager = moe.Forward(*args, stats=True, fp8=q8)
    graph = moe.Forward(*args, stats=True, fp8=q8, graph=True)
    return layer, L, eager, graph


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_graph_replay_equals_eager(cuda, w):
    layer, L, eager, graph = _forwards(w)
    x = L["x"].clone()
    y = torch.empty((w.T, w.d), dtype=layer.y_dtype, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    for it in range(4):  # capture, then replays on new contents of the same buffers
        if it:
            x.copy_(torch.randn(x.shape, generator=g, device="cuda").to(x.dtype))
        graph(x, y)
        ref = eager(x)
        torch.cuda.synchronize()
        assert torch.equal(y, ref), it
        for n in graph.stats:
            assert torch.equal(graph.stats[n], eager.stats[n]), (it, n)
    assert len(graph._graphs) == 1
    y2 = graph(L["x"])  # another buffer pair: a graph of its own
    torch.cuda.synchronize()
    assert len(graph._graphs) == 2
    assert torch.equal(y2, eager(L["x"]))
    assert graph.device_status() == 0 and eager.device_status() == 0


def test_host_pipeline_on_a_graph_forward(cuda):
    import mixture_experts_layer_95_b300 as moe
    w = CASES[1]
    layer, L, eager, graph = _forwards(w)
    xs = [torch.randn((w.T, w.d), generator=torch.Generator().manual_seed(i)).to(layer.torch_dtype).pin_memory()
          for i in range(5)]
    ys = [torch.empty((w.T, w.d), dtype=layer.y_dtype).pin_memory() for _ in range(5)]
    pipe = moe.HostPipeline(graph)
    pipe.run(xs, ys)
    torch.cuda.synchronize()
    for xh, yh in zip(xs, ys):
        assert torch.equal(yh, eager(xh.cuda()).cpu())
    assert len(graph._graphs) == 2  # one per device slot

"""HostPipeline (batches in pinned host memory, copies overlapped with the
neighbouring layer calls) gives, for every batch, bit for bit the result of a
plain layer call on the same batch (GPU only)."""
import pytest
import torch

from moe_inputs import Workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [
    Workload("pipe_prefill", T=512, d=256, E=8, F=384, k=2, n_shared=1, F_s=128),
    Workload("pipe_decode", T=3, d=256, E=8, F=256, k=2),
], ids=lambda w: w.name)
def test_host_pipeline_matches_direct_calls(w):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    L = moe_inputs.make_layer(w, "cuda")
    layer = layer_of(w)
    fw = moe.Forward(layer, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"], L["ws1"],
                     L["ws3"], L["ws2"])
    g = torch.Generator(device="cuda").manual_seed(11)
    xs = [torch.randn((w.T, w.d), generator=g, device="cuda").to(L["x"].dtype) for _ in range(5)]
    want = [fw(x).clone() for x in xs]
    x_h = [x.cpu().pin_memory() for x in xs]
    y_h = [torch.full((w.T, w.d), float("nan"), dtype=want[0].dtype).pin_memory() for _ in xs]
    pipe = moe.HostPipeline(fw)
    stream = torch.cuda.current_stream()
    pipe.run(x_h, y_h, stream)
    stream.synchronize()
    for i in range(5):
        assert torch.equal(y_h[i], want[i].cpu()), i
    # a second run reuses both device slots, in the other order, into fresh buffers
    out = [torch.empty_like(y_h[0]).pin_memory() for _ in range(5)]
    pipe.run(x_h[::-1], out, stream)
    stream.synchronize()
    assert fw.device_status() == 0
    for j in range(5):
        assert torch.equal(out[j], want[4 - j].cpu()), j
    with pytest.raises(ValueError):
        pipe.run([xs[0]], [y_h[0]])  # a device tensor where a pinned host one belongs

"""Failure detection on the GPU without a fault (GPU only).

Every mbarrier wait of the tensor-core GEMMs is bounded.  The library's test
switch moe_test_stall_gemm(1) makes their producers issue no loads, so the
consumer warps' waits run out (20 ms in that mode): each kernel must record
MOE_ERR_TIMEOUT in the workspace status word, free its TMEM and return, and the
context must stay usable for the next, normal call.  One case per GEMM kernel:
the 1-CTA kernel (75 rows per expert), the CTA-pair kernel (550 rows per
expert: both CTAs of a pair give up and meet at the final cluster barrier) and
the decode kernel with the weights on the MMA's M side, with bf16 and with FP8
weights (2 rows per expert), and the two fused small-batch kernels (one
token; every warp's own ring), with bf16 and with FP8 weights.  The backward
on CTA pairs (recomputed G and U, the SwiGLU backward whose epilogue has G and
U loads and dG / dU / H stores of its own in flight, dX and the K-grouped
weight gradients) gets the same treatment.
"""
import pytest
import torch

from moe_inputs import Workload

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = -7

CASES = [
    (Workload("stall_tc_bf16", T=300, d=256, E=8, F=256, k=2), "tc"),
    (Workload("stall_pair_bf16", T=1100, d=256, E=4, F=256, k=2), "tc_pair"),
    (Workload("stall_decode_bf16", T=8, d=256, E=8, F=256, k=2), "tc_decode32"),
    (Workload("stall_decode_fp8", T=8, d=256, E=8, F=256, k=2, weights="fp8"), "tc_decode32"),
    (Workload("stall_fused_bf16", T=1, d=256, E=8, F=256, k=2, n_shared=1, F_s=128), "fused"),
    (Workload("stall_fused_fp8", T=1, d=256, E=8, F=256, k=2, weights="fp8"), "fused"),
]


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


@pytest.mark.parametrize("w,up_kernel", CASES, ids=[w.name for w, _ in CASES])
def test_bounded_wait_times_out_and_the_context_survives(cuda, w, up_kernel):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import check_layer, check_layer_fp8, layer_of
    layer = layer_of(w)
    assert moe.plan_describe(layer.cfg())["up"] == up_kernel
    L = moe_inputs.make_layer(w, "cuda")
    q8 = None
    shared = (L["ws1"], L["ws3"], L["ws2"]) if w.n_shared else (None, None, None)
    if w.weights == "fp8":
        q8 = moe.quantize_experts_fp8(layer, L["w1"], L["w3"], L["w2"], *shared)
    fw = moe.Forward(layer, L["w_gate"], L["w1"], L["w3"], L["w2"], None, None, *shared, fp8=q8)
    torch.cuda.synchronize()
    assert moe.test_stall_gemm(True) is False
    try:
        fw(L["x"])
        torch.cuda.synchronize()
    finally:
        moe.test_stall_gemm(False)
    assert fw.device_status() == MOE_ERR_TIMEOUT
    assert fw.device_status() == 0  # read-and-clear
    fw(L["x"])
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    rep = check_layer_fp8(w, L=L) if q8 is not None else check_layer(w, L=L)
    assert rep["ok"], rep


def test_backward_bounded_wait_times_out_and_the_context_survives(cuda):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    from tests.test_backward_gpu import check_backward
    w = Workload("stall_backward_pair", T=1100, d=256, E=4, F=256, k=2, n_shared=1, F_s=128)
    layer = layer_of(w)
    assert moe.plan_describe(layer.cfg())["up"] == "tc_pair"
    L = moe_inputs.make_layer(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(1234)
    dy = torch.randn((w.T, w.d), generator=g, device="cuda").to(layer.torch_dtype)
    bw = moe.Backward(layer, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"],
                      L["ws1"], L["ws3"], L["ws2"])
    torch.cuda.synchronize()
    assert moe.test_stall_gemm(True) is False
    try:
        bw(L["x"], dy, dL=2.0)
        torch.cuda.synchronize()
    finally:
        moe.test_stall_gemm(False)
    assert bw.device_status() == MOE_ERR_TIMEOUT
    assert bw.device_status() == 0  # read-and-clear
    got = {n: t.clone() for n, t in bw(L["x"], dy, dL=2.0).items()}
    torch.cuda.synchronize()
    assert bw.device_status() == 0
    fresh = moe.backward(layer, L["x"], L["w_gate"], L["w1"], L["w3"], L["w2"], dy, L["logit_bias"],
                         L["select_bias"], L["ws1"], L["ws3"], L["ws2"], dL=2.0)
    for n in fresh:
        assert torch.equal(got[n], fresh[n]), n
    rep = check_backward(w)
    assert rep["ok"], rep

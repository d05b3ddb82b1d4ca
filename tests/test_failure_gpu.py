"""Failure detection on the GPU without a fault (GPU only).

The tensor-core GEMM bounds every mbarrier wait.  The host-side test switch
MOE_TEST_STALL_GEMM=1 makes its producer issue no loads, so the consumer
warps' waits run out (20 ms in that mode): the kernel must record
MOE_ERR_TIMEOUT in the workspace status word, free its TMEM and return, and
the context must stay usable for the next, normal call.
"""
import pytest
import torch

from moe_inputs import Workload

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = -7


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


def test_bounded_wait_times_out_and_the_context_survives(cuda, monkeypatch):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import check_layer, layer_of
    w = Workload("stall_bf16", T=300, d=256, E=8, F=256, k=2)
    L = moe_inputs.make_layer(w, "cuda")
    fw = moe.Forward(layer_of(w), L["w_gate"], L["w1"], L["w3"], L["w2"])
    monkeypatch.setenv("MOE_TEST_STALL_GEMM", "1")
    fw(L["x"])
    assert fw.device_status() == MOE_ERR_TIMEOUT
    assert fw.device_status() == 0  # read-and-clear
    monkeypatch.delenv("MOE_TEST_STALL_GEMM")
    fw(L["x"])
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    rep = check_layer(w, L=L)
    assert rep["ok"], rep

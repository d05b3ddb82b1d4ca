"""moe_bias_update against the oracle, bit for bit (GPU only).

The update is b_e -/+ gamma, one fp32 rounding of an exact difference on both
sides, and the sign comes from integer counts, so the results must be equal.
"""
import numpy as np
import pytest
import torch

from moe_inputs import Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


@pytest.mark.parametrize("w", [Workload("bias_zipf", T=700, d=128, E=64, F=64, k=2, zipf_s=1.2, select_bias=True),
                               Workload("bias_small", T=33, d=64, E=4, F=64, k=2, select_bias=True)],
                         ids=lambda w: w.name)
def test_bias_update_matches_oracle(cuda, w):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    import oracle
    from tests._parity import layer_of
    layer = layer_of(w)
    L = moe_inputs.make_layer(w, "cuda")
    gamma = float(np.float32(1e-3))
    bias = L["select_bias"].clone()
    for _ in range(3):  # route -> count -> update, three rounds
        ids, gates, _ = moe.route(layer, L["x"], L["w_gate"], L["logit_bias"], bias)
        counts = moe.permute(layer, ids, gates, L["x"])["counts"]
        before = bias.cpu().numpy().copy()
        moe.bias_update(layer, counts, bias, gamma)
        torch.cuda.synchronize()
        ref = oracle.bias_update(counts.cpu().numpy(), before, w.T, w.k, gamma).astype(np.float32)
        np.testing.assert_array_equal(bias.cpu().numpy(), ref)

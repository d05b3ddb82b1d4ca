"""Tokens with NaN or Inf inputs on the GPU (GPU only).

A non-finite token row makes that token's router scores NaN or infinite.  The
top-k must still give k distinct valid ids (a NaN score ranks as -inf, ties to
the lower index), so the grouping scan's histogram matches the ids and no
position leaves its expert's segment; the other tokens' outputs must be
exactly those of a run in which the bad rows are zero (every output row of
the expert GEMMs and the combine depends on its own token only, and the
kernel choice on the configuration only).  Covers the warp router on a
decode-sized batch, a prefill-sized batch and the logits-GEMM router (E > 32).
"""
import pytest
import torch

from moe_inputs import Workload

pytestmark = pytest.mark.gpu

CASES = [
    Workload("nonfinite_decode", T=8, d=256, E=8, F=256, k=2),
    Workload("nonfinite_prefill", T=300, d=256, E=8, F=384, k=2),
    Workload("nonfinite_gemm_router", T=300, d=128, E=40, F=128, k=4),
]
BAD = (3, 5)


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_nonfinite_tokens_leave_the_others_exact(cuda, w):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    layer = layer_of(w)
    L = moe_inputs.make_layer(w, "cuda")
    x_bad = L["x"].clone()
    x_bad[BAD[0]] = float("nan")
    x_bad[BAD[1], 7] = float("inf")
    x_zero = L["x"].clone()
    x_zero[list(BAD)] = 0
    fw = moe.Forward(layer, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"], L["ws1"],
                     L["ws3"], L["ws2"])
    y_bad = fw(x_bad).clone()
    assert fw.device_status() == 0
    y_zero = fw(x_zero).clone()
    assert fw.device_status() == 0
    keep = [t for t in range(w.T) if t not in BAD]
    assert torch.equal(y_bad[keep], y_zero[keep])
    assert torch.isnan(y_bad[BAD[0]].float()).all()
    ids, gates, _ = moe.route(layer, x_bad, L["w_gate"], L["logit_bias"], L["select_bias"])
    ids = ids.cpu()
    assert ids[BAD[0]].tolist() == list(range(w.k))  # all scores NaN: the lowest indices
    for t in range(w.T):
        row = ids[t].tolist()
        assert len(set(row)) == w.k and all(0 <= e < w.E for e in row), (t, row)


def test_nonfinite_tokens_fp8_decode(cuda):
    """The same with FP8 experts on a decode-sized batch: the E4M3 hi/lo split
    of x and of H is per row, so a NaN row stays in its own row."""
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    w = Workload("nonfinite_fp8_decode", T=8, d=256, E=8, F=256, k=2)
    layer = layer_of(w)
    L = moe_inputs.make_layer(w, "cuda")
    q8 = moe.quantize_experts_fp8(layer, L["w1"], L["w3"], L["w2"])
    fw = moe.Forward(layer, L["w_gate"], None, None, None, fp8=q8)
    x_bad = L["x"].clone()
    x_bad[BAD[0]] = float("nan")
    x_bad[BAD[1], 7] = float("inf")
    x_zero = L["x"].clone()
    x_zero[list(BAD)] = 0
    y_bad = fw(x_bad).clone()
    assert fw.device_status() == 0
    y_zero = fw(x_zero).clone()
    assert fw.device_status() == 0
    keep = [t for t in range(w.T) if t not in BAD]
    assert torch.equal(y_bad[keep], y_zero[keep])

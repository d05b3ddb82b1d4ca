"""FP8 (E4M3, per-channel scale) expert weights on the GPU vs the oracle (GPU only).

The quantisation kernel must reproduce the oracle's codes and scales bit for
bit (both take the fp32 quotient and round to nearest even); the layer with
FP8 experts must match the oracle evaluated with the exactly dequantised
weights, within the bf16 layer's tolerance.  Covers the tensor-core kernel's
FP8 path in both modes: ragged N and K tails, the shared expert, split-K
decode batches with gathered rows, expert-choice routing, and the Mixtral
decode batches the benchmark times.  Comparison rules: tests/_parity.py.
"""
import json

import numpy as np
import pytest
import torch

from moe_inputs import WORKLOADS, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_layer_95_b300 as moe
    moe.lib()
    return torch.device("cuda")


def _assert_ok(rep):
    assert rep["ok"], json.dumps(rep, indent=1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_matches_oracle_bit_for_bit(cuda, dtype):
    from tests._parity import check_quantize
    g = torch.Generator(device="cuda").manual_seed(3)
    w = torch.randn((300, 272), generator=g, device="cuda") * torch.rand((300, 1), generator=g, device="cuda") * 3
    w[7] = 0.0                              # all-zero row
    w[9, :] = torch.tensor(1.0)             # constant row: every code 448
    w[11, ::2] = 2.0 ** -10                 # row maximum 448 below: scale 1, so these are exact
    w[11, 1::2] = 3 * 2.0 ** -11            # ties and near-ties on the subnormal grid
    w[11, 0] = 448.0
    rep = check_quantize(w.to(dtype).contiguous())
    assert rep["codes_equal"] and rep["scales_equal"], rep


SMALL_FP8 = [
    Workload("fp8_shared_ragged", T=300, d=272, E=8, F=400, k=2, n_shared=1, F_s=208, weights="fp8"),
    Workload("fp8_many_tiles", T=1000, d=256, E=4, F=640, k=2, weights="fp8"),
    Workload("fp8_decode_t1", T=1, d=512, E=8, F=512, k=2, weights="fp8"),
    Workload("fp8_decode_t5_shared", T=5, d=256, E=16, F=320, k=2, n_shared=1, F_s=192, select_bias=True,
             weights="fp8"),
    Workload("fp8_gemm_router_capacity", T=520, d=384, E=64, F=256, k=4, capacity=40, weights="fp8"),
    Workload("fp8_expert_choice", T=300, d=256, E=8, F=384, k=2, routing="expert", weights="fp8"),
    # one token, 160 up-GEMM tiles: balanced split-K with FP8 stages (two k-blocks
    # each); 40 experts keep it off the fused small-batch kernels
    Workload("fp8_decode_balanced_splitk_t1_e40", T=1, d=384, E=40, F=10240, k=2, weights="fp8"),
    # the fused small-batch kernels with FP8 codes (one token): ragged slices,
    # shared expert, selection bias; 8 decisions over 32 experts
    Workload("fp8_fused_t1_shared_ragged", T=1, d=272, E=8, F=400, k=2, n_shared=1, F_s=208, select_bias=True,
             weights="fp8"),
    Workload("fp8_fused_t1_k8_e32", T=1, d=512, E=32, F=512, k=8, zipf_s=1.2, weights="fp8"),
    # two tokens, the general FP8 decode path: shared expert, capacity cut
    Workload("fp8_small_t2_shared_ragged", T=2, d=272, E=8, F=400, k=2, n_shared=1, F_s=208, select_bias=True,
             weights="fp8"),
    Workload("fp8_small_t2_capacity", T=2, d=512, E=16, F=512, k=4, capacity=1, zipf_s=1.2, weights="fp8"),
    # 17..32 rows per touched expert: the FP8 decode GEMM's 48-row token tiles (shared expert: 48, 48, 4)
    Workload("fp8_decode_48rows_shared", T=100, d=256, E=8, F=320, k=2, n_shared=1, F_s=192, weights="fp8"),
]


@pytest.mark.parametrize("w", SMALL_FP8, ids=[w.name for w in SMALL_FP8])
def test_fp8_layer_matches_oracle(cuda, w):
    from tests._parity import check_layer_fp8
    _assert_ok(check_layer_fp8(w))


def test_fp8_subnormal_codes_are_widened_exactly(cuda):
    """Rows whose maximum sits in a column where x is 0: the up GEMM then sees
    only the row's small weights, which quantise to subnormal E4M3 codes
    (|w / scale| < 2^-6), so y depends on widening those codes exactly."""
    import moe_inputs
    from tests._parity import check_layer_fp8
    w = Workload("fp8_subnormal_codes", T=200, d=256, E=4, F=256, k=2, weights="fp8")
    L = moe_inputs.make_layer(w, "cuda")
    L["x"][:, 0] = 0
    for n in ("w1", "w3"):
        L[n][:, :, 1:] *= 1e-4
        L[n][:, :, 0] = 1.0  # scale = 1/448: the rest maps below 2^-6
    q1 = __import__("mixture_experts_layer_95_b300").quantize_fp8(L["w1"])[0]
    exp_zero = ((q1[:, :, 1:] & 0x78) == 0).float().mean().item()
    assert exp_zero > 0.9  # almost every code the GEMM uses is subnormal (or zero)
    _assert_ok(check_layer_fp8(w, L=L))


@pytest.mark.parametrize("how", ["tiny", "huge", "zero", "outlier"])
def test_fp8_fused_one_token_of_extreme_scale(cuda, how):
    """The fused one-token kernels meet E4M3 codes with f16 activations scaled
    by a power of two per warp slice (x, then H): a token scaled by 2^-40 or
    2^+30, a zero token (y exactly 0) and one entry 2^12 above the rest must
    each stay within tolerance."""
    import moe_inputs
    from tests._parity import check_layer_fp8
    w = Workload(f"fp8_fused_scale_{how}", T=1, d=256, E=8, F=384, k=2, n_shared=1, F_s=128, weights="fp8")
    L = moe_inputs.make_layer(w, "cuda")
    x = L["x"].float()
    if how == "tiny":
        x *= 2.0 ** -40
    elif how == "huge":
        x *= 2.0 ** 30
    elif how == "zero":
        x[:] = 0.0
    else:
        x[0, 5] = 4096.0
    L["x"] = x.to(L["x"].dtype).contiguous()
    rep = check_layer_fp8(w, L=L, per_token=True)
    print(json.dumps(rep))
    _assert_ok(rep)


def test_fp8_fused_one_token_of_subnormal_scale(cuda):
    """A token of bf16 subnormals (x scaled by 2^-130): the slice scale 2^-e
    would overflow fp32 there, so it is held at 2^125.  H (about x^2)
    underflows fp32 on every path, so y must come out finite and negligible
    -- not NaN from 0 x inf."""
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    w = Workload("fp8_fused_scale_subnormal", T=1, d=256, E=8, F=384, k=2, n_shared=1, F_s=128, weights="fp8")
    layer = layer_of(w)
    assert moe.plan_describe(layer.cfg())["up"] == "fused"
    L = moe_inputs.make_layer(w, "cuda")
    x = (L["x"].float() * 2.0 ** -130).to(L["x"].dtype).contiguous()
    assert int((x != 0).sum()) > 200  # subnormal, not flushed
    q8 = moe.quantize_experts_fp8(layer, L["w1"], L["w3"], L["w2"], L["ws1"], L["ws3"], L["ws2"])
    fw = moe.Forward(layer, L["w_gate"], None, None, None, L["logit_bias"], L["select_bias"], fp8=q8)
    y = fw(x)
    torch.cuda.synchronize()
    assert fw.device_status() == 0
    assert bool(torch.isfinite(y.float()).all())
    assert float(y.float().abs().max()) < 1e-30


@pytest.mark.parametrize("T", [3, 40])
def test_fp8_decode_tokens_of_very_different_scales(cuda, T):
    """Decode-sized batches carry the bf16 token rows (and H) to the FP8 MMA
    as E4M3 hi + lo codes with a power-of-two scale per row.  Rows scaled by
    2^-40 and 2^+30, a zero row and a row with one entry 2^12 above the rest
    (whose small entries fall below the lo codes' range) must each stay
    within tolerance against their own RMS; the zero row gives exactly 0."""
    import moe_inputs
    from tests._parity import check_layer_fp8
    w = Workload(f"fp8_decode_scales_t{T}", T=T, d=256, E=8, F=384, k=2, n_shared=1, F_s=128, weights="fp8")
    L = moe_inputs.make_layer(w, "cuda")
    x = L["x"].float()
    x[0] *= 2.0 ** -40
    x[1] *= 2.0 ** 30
    x[2] = 0.0
    if T > 3:
        x[3, 5] = 4096.0
    L["x"] = x.to(L["x"].dtype).contiguous()
    rep = check_layer_fp8(w, L=L, per_token=True)
    print(json.dumps(rep))
    _assert_ok(rep)


# 1, 8 and 32 tokens (at most 16 rows per touched expert on average): 32-row
# token tiles; 128 tokens: 48-row tiles over the token codes split in expert
# order; each at the size the benchmark times
@pytest.mark.parametrize("name", ["mixtral_decode_t1_fp8", "mixtral_decode_t8_fp8", "mixtral_decode_t32_fp8",
                                  "mixtral_decode_t128_fp8"])
def test_fp8_mixtral_decode(cuda, name):
    from tests._parity import check_layer_fp8
    rep = check_layer_fp8(WORKLOADS[name])
    print(json.dumps(rep))
    _assert_ok(rep)


def test_forward_fp8_rejects_bad_configs(cuda):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    w = Workload("fp8_bad", T=4, d=264, E=4, F=64, k=2)  # d not a multiple of 16
    L = moe_inputs.make_layer(w, "cuda")
    layer = moe.Layer(T=4, d=264, E=4, k=2, d_ff=64)
    with pytest.raises(moe.MoeError):
        moe.quantize_fp8(L["w1"])  # 264 columns: not a multiple of 16
    q8 = {n: torch.zeros(s, dtype=t, device="cuda") for n, s, t in (
        ("w1", (4, 64, 264), torch.uint8), ("w3", (4, 64, 264), torch.uint8), ("w2", (4, 264, 64), torch.uint8),
        ("s1", (4, 64), torch.float32), ("s3", (4, 64), torch.float32), ("s2", (4, 264), torch.float32))}
    fw = moe.Forward(layer, L["w_gate"], None, None, None, fp8=q8)
    with pytest.raises(moe.MoeError):
        fw(L["x"])

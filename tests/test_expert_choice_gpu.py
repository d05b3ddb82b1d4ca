"""Expert-choice routing on the GPU vs the fp64 oracle, through the C ABI (GPU only).

Buckets of C tokens per expert ("One Deep Concept #04", section 11): small
layers covering every router variant (one block per token, warp router,
tensor-core / CUDA-core logits GEMM), ragged buckets, buckets larger than
T k / E, the C = T dense limit, a one-token batch that every expert takes, and
the Mixtral-prefill-sized layer the benchmark times, checked on every routing
output and a sample of output rows.  Comparison rules: tests/_parity.py.
"""
import json

import pytest
import torch

from moe_inputs import WORKLOADS, Workload

pytestmark = pytest.mark.gpu

SMALL_EC = [
    # warp router (E <= 16, T > 256), C = 75: ragged 128-row tiles, shared expert
    Workload("ec_warp_shared_bf16", T=300, d=256, E=8, F=384, k=2, n_shared=1, F_s=256, routing="expert"),
    # one block per token (T <= 256), fp32 layer
    Workload("ec_split_d_f32", T=200, d=128, E=8, F=128, k=2, dtype="f32", routing="expert"),
    # E = 64: logits GEMM + softmax pass; E*C = 2048 rows, the up GEMM gathers x itself
    Workload("ec_gemm_router_bf16", T=512, d=256, E=64, F=256, k=4, routing="expert"),
    # fp32 logits GEMM (E = 20), buckets of 3 tokens
    Workload("ec_gemm_router_f32", T=300, d=128, E=20, F=96, k=3, dtype="f32", capacity=3, routing="expert"),
    # C = 200 > T k / E: more rows than token choice would have, many tokens in several buckets
    Workload("ec_large_bucket_bf16", T=256, d=128, E=4, F=128, k=1, capacity=200, routing="expert"),
    # C = T: every expert takes every token (the dense mixture)
    Workload("ec_dense_bf16", T=64, d=128, E=4, F=128, k=2, capacity=64, routing="expert"),
    # one token: C = 1, so all eight experts take it (split-K GEMMs)
    Workload("ec_one_token_bf16", T=1, d=512, E=8, F=512, k=2, routing="expert"),
    # Zipf logit offset: the popular experts' scores dominate, so many tokens get no expert at
    # all (y = 0) and RMS(y) shrinks; a single bf16 H then costs ~3% of RMS(y) at the busiest
    # tokens, so the layer keeps H as a hi + lo pair (as the skewed token-choice layer does)
    Workload("ec_zipf_empty_tokens_bf16", T=400, d=256, E=16, F=128, k=1, zipf_s=1.2, h_split=True,
             routing="expert"),
    # decode-sized buckets (C = 2 of 16 tokens): the down GEMM runs the combine, and
    # counts the tokens no expert took, in its last CTA per column block
    Workload("ec_decode_empty_tokens_bf16", T=16, d=256, E=8, F=256, k=1, zipf_s=1.2, routing="expert"),
]


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_layer_95_b300 as moe
    moe.lib()
    return torch.device("cuda")


def _assert_ok(rep):
    assert rep["ok"], json.dumps(rep, indent=1)


@pytest.mark.parametrize("w", SMALL_EC, ids=[w.name for w in SMALL_EC])
def test_expert_choice_small(cuda, w):
    from tests._parity import check_layer_ec
    _assert_ok(check_layer_ec(w))


def test_expert_choice_tied_scores_keep_lower_tokens(cuda):
    """All tokens identical: every score ties, so each expert must take tokens 0..C-1."""
    import moe_inputs
    from tests._parity import check_layer_ec
    w = Workload("ec_all_ties_bf16", T=300, d=128, E=4, F=64, k=1, routing="expert")
    L = moe_inputs.make_layer(w, "cuda")
    L["x"] = L["x"][:1].expand(w.T, w.d).contiguous()
    rep = check_layer_ec(w, L=L)
    _assert_ok(rep)
    assert rep["experts_inside_margin"] == w.E  # every boundary is a tie
    assert rep["buckets_equal_oracle"]  # ... resolved to the lowest token indices, as the oracle does


def test_expert_choice_rejects_token_choice_steps(cuda):
    import mixture_experts_layer_95_b300 as moe
    layer = moe.Layer(T=16, d=64, E=4, k=2, d_ff=64, routing="expert")
    x = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError):
        moe.route(layer, x, wg)


def test_expert_choice_mixtral_prefill_sampled(cuda):
    from tests._parity import check_layer_ec
    rep = check_layer_ec(WORKLOADS["mixtral_prefill_ec"], n_sample=48)
    _assert_ok(rep)

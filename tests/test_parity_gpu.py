"""CUDA path vs the fp64 oracle, element by element, through the C ABI (GPU only).

Small workloads span several 128-row tiles, ragged segment ends, K and N
tails, empty experts, dropped entries and every routing variant; the
full-size benchmark workloads (Mixtral, DeepSeek-V3, skewed) are checked on every
routing and grouping output and
on a seeded sample of output rows, in the same launch configuration the
benchmark times.  See tests/_parity.py for the comparison rules.
"""
import json

import pytest
import torch

from moe_inputs import WORKLOADS, Workload

pytestmark = pytest.mark.gpu

# Router kernels by shape: T <= 256 and E <= 32 -> one block per token;
# E <= 16 -> warp router (32-token chunks); otherwise tensor-core (bf16) or
# CUDA-core (fp32) logits GEMM + softmax/top-k pass (64-token chunks).
SMALL = [
    WORKLOADS["tiny_f32"],
    Workload("small_bf16", T=300, d=512, E=8, F=384, k=2),
    Workload("ragged_bf16", T=77, d=264, E=6, F=200, k=3),
    Workload("ragged_f32", T=77, d=264, E=6, F=200, k=3, dtype="f32"),
    Workload("gemm_router_capacity_zipf_bf16", T=520, d=384, E=64, F=256, k=4, capacity=40, zipf_s=1.2,
             h_split=True),
    Workload("split_h_shared_ragged_bf16", T=150, d=264, E=6, F=200, k=2, n_shared=1, F_s=136, capacity=30,
             h_split=True),
    Workload("gemm_router_f32", T=300, d=128, E=20, F=96, k=3, dtype="f32"),
    Workload("warp_router_f32", T=300, d=264, E=8, F=96, k=2, dtype="f32"),
    # enough rows that both CUDA-core GEMMs take 64-row tiles (the small cases
    # above take 32-row tiles), with a shared expert and a ragged F
    Workload("many_tiles_shared_f32", T=1024, d=256, E=8, F=520, k=2, n_shared=1, F_s=264, dtype="f32"),
    Workload("shared_selectbias_bf16", T=200, d=256, E=32, F=128, k=8, n_shared=1, F_s=192, select_bias=True),
    Workload("dense_limit_bf16", T=64, d=128, E=8, F=128, k=8, renormalize=False),
    Workload("single_expert_bf16", T=130, d=128, E=1, F=256, k=1),
    Workload("capacity_zero_shared_bf16", T=40, d=128, E=4, F=64, k=2, capacity=0, n_shared=1, F_s=64),
    Workload("decode_like_t1_bf16", T=1, d=512, E=8, F=512, k=2),
    # a few tokens: the expert GEMMs split K into fp32 slices (shared expert,
    # ragged F and the hi + lo H included)
    Workload("split_k_shared_t3_bf16", T=3, d=256, E=16, F=320, k=2, n_shared=1, F_s=192, select_bias=True,
             h_split=True),
    Workload("decode_like_t5_bf16", T=5, d=512, E=8, F=512, k=2),
    # 17..32 rows per touched expert: 64-row token tiles of the decode GEMM
    Workload("decode_64rows_shared_bf16", T=100, d=256, E=8, F=320, k=2, n_shared=1, F_s=192),
    Workload("many_tiles_bf16", T=1000, d=256, E=4, F=640, k=2),
    # >= 512 rows per expert: both GEMMs run on CTA pairs (256-row tiles whose
    # upper half may be empty at a segment end; N tail of 64 in the down GEMM)
    Workload("pair_tiles_shared_bf16", T=1100, d=320, E=4, F=384, k=2, n_shared=1, F_s=256),
    # a few hundred rows per expert (DeepSeek-V3-like segments): CTA pairs whose
    # last tile of a segment is an M = 128 tile (64 rows per SM, the upper SM's
    # rows partly or wholly absent) when at most 128 rows remain; ragged N and
    # K; shared expert (600 rows: 256 + 256 + 88) in the same launches
    Workload("wide_chunks_shared_ragged_bf16", T=600, d=272, E=4, F=400, k=2, n_shared=1, F_s=208, select_bias=True),
    Workload("wide_chunks_e16_bf16", T=2000, d=256, E=16, F=256, k=2),
    # 128-191 rows per expert: the 1-SM kernel's 128-row tiles
    Workload("one_sm_160rows_bf16", T=640, d=256, E=8, F=264, k=2),
    # expert rows kept in bf16 for the combine: 1-SM tiles (k = 8 + shared), CTA
    # pairs, and decode-sized split-K (the combine rounds each entry's slice sum)
    Workload("yperm_bf16_k8_shared", T=300, d=256, E=32, F=128, k=8, n_shared=1, F_s=192, select_bias=True,
             yperm_bf16=True),
    Workload("yperm_bf16_pairs", T=1100, d=256, E=4, F=384, k=2, yperm_bf16=True),
    Workload("yperm_bf16_split_k_t3", T=3, d=256, E=16, F=320, k=2, n_shared=1, F_s=192, yperm_bf16=True),
    Workload("yperm_bf16_decode_64rows", T=100, d=256, E=8, F=320, k=2, n_shared=1, F_s=192, yperm_bf16=True),
    # the logits GEMM with rows of 18 fp32 logits (72 bytes, not whole 16-byte
    # chunks): its epilogue stores element by element
    Workload("gemm_router_e18_bf16", T=300, d=256, E=18, F=128, k=3),
    # one token on a router too wide for the fused small-batch kernels: the
    # decode GEMM with split-K
    Workload("decode_t1_e40_bf16", T=1, d=512, E=40, F=512, k=2),
    # one token, E <= 32: the two fused small-batch kernels.  Ragged hidden
    # slices (F / 16 not a multiple of 8; the last warps' slices shorter or
    # empty), a d that is not a multiple of 16, shared expert, biases, both
    # gate normalisations, capacity 0 (every routed entry dropped), 8 routing
    # decisions over 32 experts
    Workload("fused_t1_ragged", T=1, d=520, E=8, F=1000, k=2),
    Workload("fused_t1_k8_shared_long_d", T=1, d=4104, E=32, F=520, k=8, n_shared=1, F_s=264),
    Workload("fused_t1_shared_selectbias_plain", T=1, d=1024, E=16, F=2056, k=4, n_shared=1, F_s=776,
             select_bias=True, renormalize=False),
    Workload("fused_t1_capacity_zero_shared", T=1, d=256, E=4, F=128, k=2, capacity=0, n_shared=1, F_s=64),
    Workload("fused_t1_capacity_zero", T=1, d=256, E=4, F=128, k=2, capacity=0),
    Workload("fused_t1_tiny_f_empty_warps", T=1, d=128, E=6, F=40, k=3, zipf_s=1.2),
    # two tokens: the general decode path (the fused kernels take one), with
    # the same features
    Workload("small_t2_shared_selectbias", T=2, d=1024, E=16, F=2056, k=4, n_shared=1, F_s=776, select_bias=True),
    Workload("small_t2_capacity_shared", T=2, d=256, E=4, F=256, k=3, capacity=1, n_shared=1, F_s=128),
    Workload("small_t2_k8_plain_gates_e32", T=2, d=384, E=32, F=384, k=8, renormalize=False),
    # three tokens: the general decode path
    Workload("decode_t3_shared_capacity", T=3, d=256, E=4, F=256, k=2, capacity=1, n_shared=1, F_s=128),
]


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_layer_95_b300 as moe
    moe.lib()  # fail loudly if the library is missing
    return torch.device("cuda")


def _assert_ok(rep):
    assert rep["ok"], json.dumps(rep, indent=1)


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_workloads_match_oracle(cuda, w):
    from tests._parity import check_layer
    _assert_ok(check_layer(w))


def test_all_tokens_to_one_expert(cuda):
    """Empty groups and one long segment (six 128-row tiles)."""
    import moe_inputs
    from tests._parity import check_layer
    w = Workload("all_to_one_bf16", T=700, d=128, E=8, F=192, k=1)
    L = moe_inputs.make_layer(w, "cuda")
    L["logit_bias"] = torch.tensor([30.0] + [0.0] * 7, device="cuda")
    rep = check_layer(w, L=L)
    _assert_ok(rep)


def test_zero_tokens_is_a_no_op(cuda):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    w = Workload("empty", T=0, d=128, E=4, F=64, k=2)
    L = moe_inputs.make_layer(w, "cuda")
    layer = moe.Layer(T=0, d=128, E=4, k=2, d_ff=64)
    y = moe.forward(layer, L["x"], L["w_gate"], L["w1"], L["w3"], L["w2"])
    assert y.shape == (0, 128)


FULL = [("mixtral_decode_t1", None), ("mixtral_decode_t8", None), ("mixtral_decode_t32", None),
        ("mixtral_decode_t128", 48), ("mixtral_prefill", 48), ("skewed_capacity", 96), ("deepseek_v3", 24)]


@pytest.mark.parametrize("name,n_sample", FULL, ids=[n for n, _ in FULL])
def test_full_size_workloads_match_oracle(cuda, name, n_sample):
    from tests._parity import check_layer
    rep = check_layer(WORKLOADS[name], n_sample=n_sample)
    print(json.dumps(rep))
    _assert_ok(rep)

"""Seeded synthetic inputs for the MoE layer, shared by the CUDA path and the oracle.

This module holds none of the layer's arithmetic: it only draws tensors and
names the workloads.  Both sides of a parity check receive the very same
tensors from here (drawn once, on the device under test, then copied to the
host for the oracle), so no generator has to be re-implemented bit-exactly.

Recipe (every workload):
  * one torch.Generator per tensor, on the target device, seeded with
    ``(seed << 8) | tensor_index`` so that a tensor's values depend only on the
    seed, its index and its own shape (decode sizes with different T share the
    expert weights);
  * x ~ N(0, 1); router and expert weights ~ N(0, 1/fan_in) with fan_in = d for
    W_gate, W1, W3 (and their shared-expert copies) and fan_in = F for W2;
  * values are drawn in fp32 and, for bf16 workloads, rounded to bf16 (round to
    nearest even);
  * the selection-only bias (DeepSeek-V3-shaped layer) ~ U(-0.1, 0.1), fp32;
  * the skewed layer adds to every token's logits the log-probability of a
    Zipf(s) rank distribution over the experts (expert 0 the most popular).

Weights are stored as the layer consumes them: W_gate [E, d], W1 and W3
[E, F, d], W2 [E, d, F], shared W1/W3 [F_s, d], shared W2 [d, F_s].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

TENSOR_INDEX = {"x": 0, "w_gate": 1, "w1": 2, "w3": 3, "w2": 4, "ws1": 5, "ws3": 6, "ws2": 7,
                "select_bias": 8}


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    F: int
    k: int
    dtype: str = "bf16"          # "bf16" or "f32" (x, weights and y)
    n_shared: int = 0
    F_s: int = 0
    renormalize: bool = True
    capacity: int = -1           # < 0: unlimited
    alpha: float = 0.01
    select_bias: bool = False    # draw a selection-only bias ~ U(-0.1, 0.1)
    zipf_s: float = 0.0          # > 0: add Zipf(s) log-probabilities to the logits
    h_split: bool = False        # layer option: keep H as a hi + lo bf16 pair
    routing: str = "token"       # "token": tokens pick top-k experts; "expert": experts pick C tokens
    weights: str = "same"        # "same": experts stored in `dtype`; "fp8": E4M3 codes + per-row fp32 scales
    yperm_bf16: bool = False     # layer option: expert rows of the down GEMM kept in bf16 for the combine
    seed: int = 0
    notes: str = field(default="", compare=False)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _cap(T, k, E, factor=1.25):
    return int(math.floor(factor * T * k / E))


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", T=256, d=256, E=8, F=512, k=2, dtype="f32"),
    "mixtral_prefill": Workload("mixtral_prefill", T=4096, d=4096, E=8, F=14336, k=2),
    "mixtral_decode_t1": Workload("mixtral_decode_t1", T=1, d=4096, E=8, F=14336, k=2),
    "mixtral_decode_t8": Workload("mixtral_decode_t8", T=8, d=4096, E=8, F=14336, k=2),
    "mixtral_decode_t32": Workload("mixtral_decode_t32", T=32, d=4096, E=8, F=14336, k=2),
    "mixtral_decode_t128": Workload("mixtral_decode_t128", T=128, d=4096, E=8, F=14336, k=2),
    # same expert shapes and tokens per expert as mixtral_prefill at half the
    # memory (4 experts, 2048 tokens): the case profiled with ncu --set full
    "mixtral_prefill_e4": Workload("mixtral_prefill_e4", T=2048, d=4096, E=4, F=14336, k=2),
    # expert-choice routing on the Mixtral prefill shape: every expert takes
    # C = T k / E = 1024 tokens (the same GEMM work as token choice)
    "mixtral_prefill_ec": Workload("mixtral_prefill_ec", T=4096, d=4096, E=8, F=14336, k=2, routing="expert"),
    # FP8 (E4M3, per-channel scales) expert weights for decode: half the bytes to stream
    "mixtral_decode_t1_fp8": Workload("mixtral_decode_t1_fp8", T=1, d=4096, E=8, F=14336, k=2, weights="fp8"),
    "mixtral_decode_t8_fp8": Workload("mixtral_decode_t8_fp8", T=8, d=4096, E=8, F=14336, k=2, weights="fp8"),
    "mixtral_decode_t32_fp8": Workload("mixtral_decode_t32_fp8", T=32, d=4096, E=8, F=14336, k=2, weights="fp8"),
    "mixtral_decode_t128_fp8": Workload("mixtral_decode_t128_fp8", T=128, d=4096, E=8, F=14336, k=2,
                                        weights="fp8"),
    # nine expert rows per token (eight routed, one shared), each a small part of
    # y: the layer keeps them in bf16 for the combine (half of its 2.1 GB of reads)
    "deepseek_v3": Workload("deepseek_v3", T=8192, d=7168, E=256, F=2048, k=8, n_shared=1, F_s=2048,
                            select_bias=True, yperm_bf16=True),
    # the DeepSeek-V3 expert shape and rows per expert (~256) at an eighth of
    # the weights (32 experts, 1024 tokens): the case profiled with ncu --set full
    "deepseek_v3_e32": Workload("deepseek_v3_e32", T=1024, d=7168, E=32, F=2048, k=8, n_shared=1, F_s=2048,
                                select_bias=True, yperm_bf16=True),
    # the capacity cut leaves most tokens with small outputs and a few with
    # outputs ~12x RMS(y); a bf16 H then costs ~2% of RMS(y) at those tokens,
    # so this layer keeps H as a hi + lo pair
    "skewed_capacity": Workload("skewed_capacity", T=16384, d=2048, E=64, F=1408, k=2,
                                capacity=_cap(16384, 2, 64), zipf_s=1.2, h_split=True),
}


def zipf_log_probs(E: int, s: float) -> torch.Tensor:
    """log of the Zipf(s) probability of rank r = e + 1 among E ranks (fp64 -> fp32)."""
    r = torch.arange(1, E + 1, dtype=torch.float64)
    w = r.pow(-s)
    return (w / w.sum()).log().to(torch.float32)


def _gen(device, seed, name):
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) << 8) | TENSOR_INDEX[name])
    return g


def _normal(shape, std, device, dtype, seed, name, chunk_dim0=False):
    g = _gen(device, seed, name)
    if chunk_dim0 and len(shape) == 3:
        out = torch.empty(shape, dtype=dtype, device=device)
        for e in range(shape[0]):
            out[e] = (torch.randn(shape[1:], generator=g, device=device) * std).to(dtype)
        return out
    return (torch.randn(shape, generator=g, device=device) * std).to(dtype)


def make_layer(w: Workload, device="cpu") -> dict:
    """Draw every input tensor of workload ``w`` on ``device``."""
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dev = torch.device(device)
    s = w.seed
    L = {
        "x": _normal((w.T, w.d), 1.0, dev, dt, s, "x"),
        "w_gate": _normal((w.E, w.d), 1.0 / math.sqrt(w.d), dev, dt, s, "w_gate"),
        "w1": _normal((w.E, w.F, w.d), 1.0 / math.sqrt(w.d), dev, dt, s, "w1", True),
        "w3": _normal((w.E, w.F, w.d), 1.0 / math.sqrt(w.d), dev, dt, s, "w3", True),
        "w2": _normal((w.E, w.d, w.F), 1.0 / math.sqrt(w.F), dev, dt, s, "w2", True),
        "ws1": None, "ws3": None, "ws2": None, "logit_bias": None, "select_bias": None,
    }
    if w.n_shared:
        L["ws1"] = _normal((w.F_s, w.d), 1.0 / math.sqrt(w.d), dev, dt, s, "ws1")
        L["ws3"] = _normal((w.F_s, w.d), 1.0 / math.sqrt(w.d), dev, dt, s, "ws3")
        L["ws2"] = _normal((w.d, w.F_s), 1.0 / math.sqrt(w.F_s), dev, dt, s, "ws2")
    if w.select_bias:
        g = _gen(dev, s, "select_bias")
        L["select_bias"] = (torch.rand((w.E,), generator=g, device=dev) * 0.2 - 0.1).float()
    if w.zipf_s > 0:
        L["logit_bias"] = zipf_log_probs(w.E, w.zipf_s).to(dev)
    return L


def to_numpy(t):
    """Host numpy view for the oracle: float32 stays float32, bf16 becomes uint16 bits."""
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def layer_numpy(L: dict) -> dict:
    return {k: to_numpy(v) for k, v in L.items()}


# ---- work accounting (what counts as the layer's algorithmic work) ----------

def expert_params(d: int, F: int) -> int:
    """Parameters of one SwiGLU expert: W1, W3 (F x d) and W2 (d x F)."""
    return 3 * d * F


def algorithmic_flops(w: Workload, kept_total: int) -> float:
    """FLOPs of one layer call: routed (kept) expert work, shared expert, router.

    Counts 2 FLOPs per multiply-add; no padded tile rows, no dropped entries.
    """
    routed = 2.0 * expert_params(w.d, w.F) * kept_total
    shared = 2.0 * expert_params(w.d, w.F_s) * w.T * w.n_shared
    router = 2.0 * w.T * w.d * w.E
    return routed + shared + router


def expert_weight_bytes(w: Workload, n_touched: int) -> float:
    """Bytes of expert weights a call must read: touched routed experts + shared
    (FP8: one byte per weight plus a 4-byte scale per weight row)."""
    if w.weights == "fp8":
        rows = lambda d, F: 2 * F + d  # rows of W1, W3 and W2
        return float(expert_params(w.d, w.F) * n_touched + expert_params(w.d, w.F_s) * w.n_shared
                     + 4 * (rows(w.d, w.F) * n_touched + rows(w.d, w.F_s) * w.n_shared))
    eb = 2 if w.dtype == "bf16" else 4
    return float(eb * (expert_params(w.d, w.F) * n_touched + expert_params(w.d, w.F_s) * w.n_shared))


def up_gemm_bytes(w: Workload, n_touched: int, kept_total: int) -> float:
    """Algorithmic HBM bytes of one up-GEMM launch: W1 and W3 of the touched
    experts and the shared expert (up_weight_bytes), every kept token row read
    once and every row of H written once (activations in the layer's dtype)."""
    ab = 4 if w.dtype == "f32" else 2
    return up_weight_bytes(w, n_touched) + float(ab * (kept_total * (w.d + w.F) + w.T * w.n_shared * (w.d + w.F_s)))


def up_weight_bytes(w: Workload, n_touched: int) -> float:
    """Bytes of W1 and W3 (touched experts + shared) the up GEMM must read."""
    if w.weights == "fp8":
        per = lambda F: 2 * F * w.d + 4 * 2 * F
    else:
        eb = 2 if w.dtype == "bf16" else 4
        per = lambda F: 2 * F * w.d * eb
    return float(per(w.F) * n_touched + per(w.F_s) * w.n_shared)

"""Backward pass on the GPU vs the fp64 oracle's backward, through the C ABI (GPU only).

moe_backward recomputes the routing and grouping with the forward kernels; the
oracle takes those same ids (and dropped slots) and differentiates the layer in
fp64 (pinned to autograd and finite differences in test_oracle_backward.py).
dx and dW_g must satisfy max |g_gpu - g_oracle| <= 2e-2 * RMS(g_oracle), the
forward pass's bf16 rule.  The expert weight gradients are sums over an
expert's token rows of products of two operands the GPU rounds to bf16 (dG or
dU with x; g*dy with h): rounding perturbs each term by at most 2^-8 of its
own magnitude, so an entry made of few large terms can miss by several percent
of the tensor's RMS while the tensor as a whole is accurate to ~u/2.  They are
checked two ways: entry by entry, |g_gpu - g_oracle| <= 2^-7 * S (twice the
rounding bound) where S is the oracle's sum over the same terms of the products
of absolute values (|da| |x|, |db| |x|, |g dy| |h|), so a wrong entry, column
or row fails wherever it lands; and norm-wise, expert by expert,
||g_gpu - g_oracle||_F <= 2e-2 ||g_oracle||_F for every expert's block (an
expert with no tokens must give exactly 0).  Covers ragged
tiles and K windows, the shared expert, a capacity cut, selection and logit
biases, both gate normalisations, the logits-GEMM router and a one-token batch.
"""
import json

import numpy as np
import pytest
import torch

from moe_inputs import Workload

pytestmark = pytest.mark.gpu

TOL = 2e-2
ENTRY_TOL = 2.0 ** -7  # times the entry's magnitude sum

CASES = [
    Workload("bwd_basic", T=300, d=256, E=8, F=384, k=2),
    Workload("bwd_shared_capacity_biases", T=200, d=256, E=16, F=256, k=2, n_shared=1, F_s=192, capacity=20,
             select_bias=True, zipf_s=1.2),
    Workload("bwd_plain_gates", T=130, d=128, E=4, F=128, k=2, renormalize=False),
    Workload("bwd_gemm_router", T=300, d=128, E=40, F=128, k=4),
    Workload("bwd_one_token_shared", T=1, d=256, E=8, F=256, k=2, n_shared=1, F_s=128),
    # >= 512 rows per expert: the row-indexed products run on CTA pairs (ragged N and K)
    Workload("bwd_pair_shared", T=1100, d=272, E=4, F=400, k=2, n_shared=1, F_s=208),
    # ~300 rows per expert: CTA pairs with M = 128 tail tiles (the SwiGLU
    # backward's D product keeps 256-row tiles)
    Workload("bwd_pair_half_shared", T=600, d=272, E=4, F=400, k=2, n_shared=1, F_s=208, select_bias=True),
]


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_layer_95_b300 as moe
    moe.lib()
    return torch.device("cuda")


def check_backward(w, dL=2.0):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    import oracle
    from tests._parity import layer_of
    layer = layer_of(w)
    L = moe_inputs.make_layer(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(1234)
    dy = torch.randn((w.T, w.d), generator=g, device="cuda").to(layer.torch_dtype)
    G = moe.backward(layer, L["x"], L["w_gate"], L["w1"], L["w3"], L["w2"], dy, L["logit_bias"], L["select_bias"],
                     L["ws1"], L["ws3"], L["ws2"], dL=dL)
    ids, gates, _ = moe.route(layer, L["x"], L["w_gate"], L["logit_bias"], L["select_bias"])
    grp = moe.permute(layer, ids, gates, L["x"])
    torch.cuda.synchronize()
    Ln = moe_inputs.layer_numpy(L)
    ref = oracle.backward(Ln, w.k, ids.cpu().numpy(), grp["slot_pos"].cpu().numpy(),
                          oracle.widen(moe_inputs.to_numpy(dy)), w.renormalize, w.alpha, dL, magnitudes=True)
    rep = dict(workload=w.name, dropped=int(grp["n_dropped"].item()))
    ok = True
    for name in G:
        a = G[name].double().cpu().numpy()
        b = ref[name]
        finite = bool(np.isfinite(a).all())
        if name in ("dx", "dw_gate"):
            rms = float(np.sqrt(np.mean(b ** 2)))
            rel = float(np.abs(a - b).max()) / rms if rms > 0 else float(np.abs(a).max())
            rep[name] = dict(max_rel=rel, finite=finite)
        else:  # per expert block (the shared expert's matrices are one block)
            blocks_a = a if name in ("dw1", "dw3", "dw2") else a[None]
            blocks_b = b if name in ("dw1", "dw3", "dw2") else b[None]
            rel = 0.0
            for ea, eb in zip(blocks_a, blocks_b):
                nb = float(np.linalg.norm(eb))
                r = float(np.linalg.norm(ea - eb)) / nb if nb > 0 else (0.0 if not ea.any() else float("inf"))
                rel = max(rel, r)
            S = ref["sum_abs_" + name]
            # worst entry against its own bound; an entry whose magnitude sum is
            # 0 (no term reaches it) must come out exactly 0
            bound = ENTRY_TOL * S
            excess = np.where(bound > 0, np.abs(a - b) / np.where(bound > 0, bound, 1.0),
                              np.where(a != 0, np.inf, 0.0))
            worst = float(excess.max()) if excess.size else 0.0
            rep[name] = dict(block_fro_rel=rel, entry_err_over_bound=worst, finite=finite)
            ok = ok and worst <= 1.0
        ok = ok and rel <= TOL and finite
    rep["ok"] = bool(ok)
    return rep


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_backward_matches_oracle(cuda, w):
    rep = check_backward(w)
    assert rep["ok"], json.dumps(rep, indent=1)


def test_backward_is_deterministic(cuda):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    w = CASES[1]
    layer = layer_of(w)
    L = moe_inputs.make_layer(w, "cuda")
    dy = torch.ones((w.T, w.d), device="cuda", dtype=layer.torch_dtype)
    args = (layer, L["x"], L["w_gate"], L["w1"], L["w3"], L["w2"], dy, L["logit_bias"], L["select_bias"], L["ws1"],
            L["ws3"], L["ws2"])
    a = moe.backward(*args, dL=1.0)
    b = moe.backward(*args, dL=1.0)
    for n in a:
        assert torch.equal(a[n], b[n]), n


def test_backward_rejects_fp32_and_expert_choice(cuda):
    import mixture_experts_layer_95_b300 as moe
    for layer in (moe.Layer(T=4, d=64, E=4, k=2, d_ff=64, dtype="f32"),
                  moe.Layer(T=4, d=64, E=4, k=2, d_ff=64, routing="expert")):
        assert moe.lib().moe_backward_workspace_size(__import__("ctypes").byref(layer.cfg())) == 0


SAVED_CASES = [CASES[0], CASES[1], CASES[4], CASES[5], CASES[6]]


@pytest.mark.parametrize("w", SAVED_CASES, ids=[w.name for w in SAVED_CASES])
def test_backward_saved_equals_recompute(cuda, w):
    """moe_forward_train + moe_backward_saved give moe_backward's gradients
    bit for bit (G and U come from the same accumulators either way), and
    the training forward's y passes the forward's bf16 rule against
    moe_forward's y."""
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    layer = layer_of(w)
    L = moe_inputs.make_layer(w, "cuda")
    g = torch.Generator(device="cuda").manual_seed(99)
    dy = torch.randn((w.T, w.d), generator=g, device="cuda").to(layer.torch_dtype)
    bw = moe.Backward(layer, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"], L["ws1"],
                      L["ws3"], L["ws2"])
    y_train = bw.forward_train(L["x"]).clone()
    saved = {n: t.clone() for n, t in bw(L["x"], dy, dL=1.5, saved=True).items()}
    assert bw.device_status() == 0
    recomputed = bw(L["x"], dy, dL=1.5)
    assert bw.device_status() == 0
    for n in saved:
        assert torch.equal(saved[n], recomputed[n]), n
    y = moe.forward(layer, L["x"], L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"],
                    L["ws1"], L["ws3"], L["ws2"])
    a, b = y_train.double(), y.double()
    rms = float(b.pow(2).mean().sqrt())
    assert float((a - b).abs().max()) <= TOL * rms


def test_forward_train_rejects_expert_choice(cuda):
    import ctypes
    import mixture_experts_layer_95_b300 as moe
    layer = moe.Layer(T=4, d=64, E=4, k=2, d_ff=64, routing="expert")
    c = layer.cfg()
    rc = moe.lib().moe_forward_train(ctypes.byref(c), *([None] * 11), None, None, 0, None)
    assert rc == -2


def test_forward_train_statistics_equal_the_forward(cuda):
    """moe_forward_train's load statistics are moe_forward's, bit for bit (the
    same router and grouping scan; the counts are copied out of the
    workspace, where the backward reads them)."""
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    w = CASES[1]  # shared expert, capacity cut, selection bias
    layer = layer_of(w)
    L = moe_inputs.make_layer(w, "cuda")
    bw = moe.Backward(layer, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"], L["ws1"],
                      L["ws3"], L["ws2"])
    _, st_train = bw.forward_train(L["x"], stats=True)
    fw = moe.Forward(layer, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"], L["ws1"],
                     L["ws3"], L["ws2"], stats=True)
    fw(L["x"])
    torch.cuda.synchronize()
    assert int(st_train["n_dropped"].item()) > 0
    for n in ("counts", "kept", "f", "p", "L", "n_dropped"):
        assert torch.equal(st_train[n], fw.stats[n]), n

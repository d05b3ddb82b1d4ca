"""Pins of the oracle's backward pass (CPU only).

The gradients of <dy, y> + dL * L_balance (routing decisions held fixed, f held
constant, p differentiable: "MoE Deep Dive", Load Balancing Loss Derivation) are
pinned to two things other than the oracle's own backward: PyTorch autograd in
float64 on the same function written with library ops, and central finite
differences of the oracle's forward pass.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _layer(rng, T, d, E, F, shared=False, logit_bias=False):
    L = dict(
        x=_f32(rng.standard_normal((T, d))),
        w_gate=_f32(rng.standard_normal((E, d)) / math.sqrt(d)),
        w1=_f32(rng.standard_normal((E, F, d)) / math.sqrt(d)),
        w3=_f32(rng.standard_normal((E, F, d)) / math.sqrt(d)),
        w2=_f32(rng.standard_normal((E, d, F)) / math.sqrt(F)),
    )
    if shared:
        L["ws1"] = _f32(rng.standard_normal((F + 4, d)) / math.sqrt(d))
        L["ws3"] = _f32(rng.standard_normal((F + 4, d)) / math.sqrt(d))
        L["ws2"] = _f32(rng.standard_normal((d, F + 4)) / math.sqrt(F + 4))
    if logit_bias:
        L["logit_bias"] = _f32(rng.uniform(-0.5, 0.5, E))
    return L


def _torch_loss(L, ids, slot_pos, dy, renorm, alpha, dL, k):
    """The layer and its scalar loss written with PyTorch ops in float64."""
    t = {n: torch.tensor(np.asarray(v, np.float64), requires_grad=True)
         for n, v in L.items() if n != "logit_bias" and v is not None}
    T, E = ids.shape[0], t["w_gate"].shape[0]
    logits = t["x"] @ t["w_gate"].T
    if L.get("logit_bias") is not None:
        logits = logits + torch.tensor(np.asarray(L["logit_bias"], np.float64))
    p = torch.softmax(logits, dim=1)
    idx = torch.tensor(ids, dtype=torch.long)
    g = torch.gather(p, 1, idx)
    if renorm:
        g = g / g.sum(dim=1, keepdim=True)
    y = torch.zeros_like(t["x"])
    for j in range(k):
        for e in range(E):
            rows = [r for r in range(T) if ids[r, j] == e and (slot_pos is None or slot_pos[r, j] >= 0)]
            if not rows:
                continue
            xr = t["x"][rows]
            h = Fn.silu(xr @ t["w1"][e].T) * (xr @ t["w3"][e].T)
            y = y.index_add(0, torch.tensor(rows), g[rows, j:j + 1] * (h @ t["w2"][e].T))
    if "ws1" in t:
        y = y + (Fn.silu(t["x"] @ t["ws1"].T) * (t["x"] @ t["ws3"].T)) @ t["ws2"].T
    f = torch.tensor(np.bincount(ids.ravel(), minlength=E) / (T * k), dtype=torch.float64)  # constant
    Lb = alpha * E * (f * p.mean(dim=0)).sum()
    loss = (torch.tensor(dy) * y).sum() + dL * Lb
    loss.backward()
    return {n: (v.grad.numpy() if v.grad is not None else np.zeros(v.shape)) for n, v in t.items()}


@pytest.mark.parametrize("renorm,shared,capacity,lb", [(True, False, -1, False), (False, False, -1, True),
                                                       (True, True, 2, True), (False, True, 1, False)])
def test_backward_matches_torch_autograd(renorm, shared, capacity, lb):
    rng = np.random.default_rng(40 + int(renorm) + 2 * int(shared))
    T, d, E, F, k = 7, 12, 5, 10, 2
    L = _layer(rng, T, d, E, F, shared, lb)
    fw = oracle.forward(L, k, renormalize=renorm, capacity=capacity)
    dy = rng.standard_normal((T, d))
    alpha, dL = 0.01, 3.0
    got = oracle.backward(L, k, fw["ids"], fw["slot_pos"], dy, renorm, alpha, dL)
    ref = _torch_loss(L, fw["ids"], fw["slot_pos"], dy, renorm, alpha, dL, k)
    pairs = [("dx", "x"), ("dw_gate", "w_gate"), ("dw1", "w1"), ("dw3", "w3"), ("dw2", "w2")]
    if shared:
        pairs += [("dws1", "ws1"), ("dws3", "ws3"), ("dws2", "ws2")]
    for a, b in pairs:
        np.testing.assert_allclose(got[a], ref[b], rtol=1e-9, atol=1e-12, err_msg=a)
    if capacity >= 0:
        assert (fw["slot_pos"] < 0).any()  # some slot was dropped and contributes no gradient


def test_backward_matches_finite_differences_of_the_forward():
    rng = np.random.default_rng(50)
    T, d, E, F, k = 4, 6, 3, 5, 2
    L = {n: v.astype(np.float64) for n, v in _layer(rng, T, d, E, F).items()}
    # the oracle takes float32 storage; keep the probe points exactly representable
    L = {n: _f32(v) for n, v in L.items()}
    fw = oracle.forward(L, k)
    ids = fw["ids"]
    dy = rng.standard_normal((T, d))
    alpha, dL = 0.02, 1.5
    g = oracle.backward(L, k, ids, None, dy, True, alpha, dL)

    def loss(Lp):
        out = oracle.forward(Lp, k, ids=ids)
        f = np.bincount(ids.ravel(), minlength=E) / (T * k)
        return float((dy * out["y"]).sum() + dL * alpha * E * (f * out["probs"].mean(axis=0)).sum())

    h = 2.0 ** -12
    for name, grad in (("x", "dx"), ("w1", "dw1"), ("w2", "dw2"), ("w_gate", "dw_gate")):
        flat = L[name].reshape(-1)
        for idx in rng.choice(flat.size, 4, replace=False):
            up, dn = dict(L), dict(L)
            a = flat.copy(); a[idx] += h
            b = flat.copy(); b[idx] -= h
            up[name] = _f32(a.reshape(L[name].shape))
            dn[name] = _f32(b.reshape(L[name].shape))
            num = (loss(up) - loss(dn)) / (2 * h)
            assert abs(num - g[grad].reshape(-1)[idx]) <= 1e-5 * max(1.0, abs(num)), (name, idx, num)


def test_balance_loss_gradient_pushes_overloaded_experts_down():
    """Deep Dive: 'when f_i is biased high, gradients push p_i lower'."""
    rng = np.random.default_rng(60)
    T, d, E, F, k = 16, 8, 4, 6, 1
    L = _layer(rng, T, d, E, F)
    ids = np.zeros((T, k), np.int32)  # every token on expert 0: f = (1, 0, 0, 0)
    g = oracle.backward(L, k, ids, None, np.zeros((T, d)), True, 1.0, 1.0)
    # descent direction -dl raises logits of idle experts relative to expert 0
    assert np.all(g["dlogits"][:, 0] > 0) and np.all(g["dlogits"][:, 1:] < 0)


def test_magnitude_sums_are_per_token_absolute_gradients_summed():
    """The weight gradients' magnitude sums (the per-entry scale of the GPU
    comparison) equal, for every entry, the sum over tokens of |that token's
    own gradient of the entry| taken from autograd on the one-token layer:
    each token adds one term per expert block, so its absolute gradient is the
    product of absolute values.  They also bound |gradient| entry by entry."""
    rng = np.random.default_rng(70)
    T, d, E, F, k = 6, 8, 3, 7, 2
    L = _layer(rng, T, d, E, F, shared=True)
    fw = oracle.forward(L, k, capacity=3)
    dy = rng.standard_normal((T, d))
    got = oracle.backward(L, k, fw["ids"], fw["slot_pos"], dy, True, 0.01, 0.0, magnitudes=True)
    acc = {n: 0.0 for n in ("w1", "w3", "w2", "ws1", "ws3", "ws2")}
    for t in range(T):
        Lt = dict(L, x=L["x"][t:t + 1])
        ref = _torch_loss(Lt, fw["ids"][t:t + 1], fw["slot_pos"][t:t + 1], dy[t:t + 1], True, 0.01, 0.0, k)
        for n in acc:
            acc[n] = acc[n] + np.abs(ref[n])
    for n in acc:
        np.testing.assert_allclose(got["sum_abs_d" + n], acc[n], rtol=1e-9, atol=1e-13, err_msg=n)
        assert np.all(got["sum_abs_d" + n] >= np.abs(got["d" + n]) * (1 - 1e-12)), n
    assert (fw["slot_pos"] < 0).any()

"""Pins of the oracle's expert-choice routing ("One Deep Concept #04", section 11
"Expert Choice -- Reverse Who Selects Whom": every expert picks a fixed-size
bucket of tokens; a token may get any number of experts).  CPU only.

Each test ties the oracle to something other than itself: brute force over all
C-subsets, a hand-worked example, the C = T dense limit written with library
calls, a closed form of the balance loss, permutation equivariance.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _layer_f32(rng, T, d, E, F, shared=False):
    L = dict(
        x=_f32(rng.standard_normal((T, d))),
        w_gate=_f32(rng.standard_normal((E, d)) / math.sqrt(d)),
        w1=_f32(rng.standard_normal((E, F, d)) / math.sqrt(d)),
        w3=_f32(rng.standard_normal((E, F, d)) / math.sqrt(d)),
        w2=_f32(rng.standard_normal((E, d, F)) / math.sqrt(F)),
    )
    if shared:
        L["ws1"] = _f32(rng.standard_normal((F, d)) / math.sqrt(d))
        L["ws3"] = _f32(rng.standard_normal((F, d)) / math.sqrt(d))
        L["ws2"] = _f32(rng.standard_normal((d, F)) / math.sqrt(F))
    return L


def _swiglu_torch(x, w1, w3, w2):
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    return (Fn.linear(Fn.silu(Fn.linear(t(x), t(w1))) * Fn.linear(t(x), t(w3)), t(w2))).numpy()


def _brute_bucket(col, C):
    """The C-subset with the largest score sum; among equal sums the first in
    lexicographic order (itertools yields subsets in that order), which is the
    one that keeps the lower token indices on ties."""
    best, best_sum = None, -math.inf
    for sub in itertools.combinations(range(len(col)), C):
        s = sum(col[i] for i in sub)
        if s > best_sum:
            best, best_sum = sub, s
    return list(best)


@pytest.mark.parametrize("seed", range(6))
def test_selection_matches_brute_force_on_tie_heavy_scores(seed):
    rng = np.random.default_rng(100 + seed)
    T, E = 7, 3
    probs = rng.integers(0, 4, size=(T, E)).astype(np.float64)  # small integers: many exact ties
    for C in range(0, T + 1):
        sel, margin = oracle.ec_select(probs, C)
        for e in range(E):
            assert list(sel[e]) == _brute_bucket(probs[:, e], C), (seed, C, e)
            if 0 < C < T:
                order = sorted(range(T), key=lambda t: (-probs[t, e], t))
                assert margin[e] == probs[order[C - 1], e] - probs[order[C], e]
            else:
                assert math.isinf(margin[e])


def test_hand_example_two_experts_four_tokens():
    # d = 1, W_g = [[1], [0]]: logits (a_t, 0), so p[t,0] = sigmoid(a_t) and
    # p[t,1] = 1 - sigmoid(a_t).  With C = 2, expert 0 takes the two largest
    # a_t (tokens 0 and 2), expert 1 the two smallest (tokens 1 and 3).
    a = [2.0, -1.0, 0.5, -3.0]
    x = _f32([[v] for v in a])
    wg = _f32([[1.0], [0.0]])
    r = oracle.route(x, wg, 1)
    sel, margin = oracle.ec_select(r["probs"], 2)
    assert sel.tolist() == [[0, 2], [1, 3]]
    sig = [1.0 / (1.0 + math.exp(-v)) for v in a]
    # expert 0: 2nd largest sigmoid(0.5), 3rd largest sigmoid(-1)
    assert margin[0] == pytest.approx(sig[2] - sig[1], rel=1e-6)
    sl = oracle.ec_slots(sel, r["probs"])
    assert sl["slot_pos"].tolist() == [[0, -1], [-1, 2], [1, -1], [-1, 3]]
    np.testing.assert_allclose(sl["gates"][:, 0], [sig[0], 0, sig[2], 0], rtol=1e-6)
    np.testing.assert_allclose(sl["gates"][:, 1], [0, 1 - sig[1], 0, 1 - sig[3]], rtol=1e-6)
    assert sl["n_empty"] == 0


def test_dense_limit_every_expert_takes_every_token():
    # C = T: y = sum_e p_e Expert_e(x), the un-renormalised dense mixture
    rng = np.random.default_rng(11)
    T, d, E, F = 6, 16, 4, 12
    L = _layer_f32(rng, T, d, E, F)
    out = oracle.forward_expert_choice(L, T)
    logits = torch.from_numpy(L["x"]).double() @ torch.from_numpy(L["w_gate"]).double().T
    p = torch.softmax(logits, dim=1).numpy()
    ref = sum(p[:, [e]] * _swiglu_torch(L["x"], L["w1"][e], L["w3"][e], L["w2"][e]) for e in range(E))
    np.testing.assert_allclose(out["y"], ref, rtol=1e-10, atol=1e-13)
    assert out["n_empty"] == 0


def test_one_expert_per_token_when_buckets_partition_the_tokens():
    # E = 2, C = T/2 with complementary scores: every token is chosen exactly once
    rng = np.random.default_rng(12)
    T, d, F = 10, 1, 8
    x = _f32(rng.standard_normal((T, 1)))
    L = dict(x=x, w_gate=_f32([[1.0], [-1.0]]),
             w1=_f32(rng.standard_normal((2, F, d))), w3=_f32(rng.standard_normal((2, F, d))),
             w2=_f32(rng.standard_normal((2, d, F)) / math.sqrt(F)))
    out = oracle.forward_expert_choice(L, T // 2)
    live = (out["slot_pos"] >= 0).sum(axis=1)
    np.testing.assert_array_equal(live, 1)
    order = np.argsort(-x[:, 0], kind="stable")
    assert sorted(out["sel"][0].tolist()) == sorted(order[: T // 2].tolist())


def test_balance_loss_is_alpha_for_any_input():
    # f_e = C / (E C) = 1/E, so L = alpha * E * sum_e p_e / E = alpha * sum_e p_e = alpha
    rng = np.random.default_rng(13)
    for T, E, C in ((20, 4, 5), (33, 8, 3), (9, 3, 9)):
        L = _layer_f32(rng, T, 8, E, 8)
        out = oracle.forward_expert_choice(L, C, alpha=0.01, tokens=np.arange(1, dtype=np.int32))
        np.testing.assert_allclose(out["f"], 1.0 / E, rtol=0, atol=1e-15)
        assert out["L"] == pytest.approx(0.01, abs=1e-14)
        np.testing.assert_array_equal(out["counts"], C)


def test_slot_form_invariants():
    rng = np.random.default_rng(14)
    T, d, E, F, C = 40, 8, 6, 8, 9
    L = _layer_f32(rng, T, d, E, F)
    out = oracle.forward_expert_choice(L, C, tokens=np.arange(1, dtype=np.int32))
    sel, sp, probs = out["sel"], out["slot_pos"], out["probs"]
    for e in range(E):
        assert np.all(np.diff(sel[e]) > 0) and sel[e].min() >= 0 and sel[e].max() < T
        for i, t in enumerate(sel[e]):
            assert sp[t, e] == e * C + i
            assert out["gates"][t, e] == probs[t, e]
        assert (sp[:, e] >= 0).sum() == C
    assert out["n_empty"] == int(((sp >= 0).sum(axis=1) == 0).sum())
    assert np.all(out["margin"] >= 0)


def test_permutation_equivariance():
    rng = np.random.default_rng(15)
    T, d, E, F, C = 24, 16, 4, 12, 7
    L = _layer_f32(rng, T, d, E, F, shared=True)
    perm = rng.permutation(T)
    a = oracle.forward_expert_choice(L, C)
    b = oracle.forward_expert_choice(dict(L, x=np.ascontiguousarray(L["x"][perm])), C)
    inv = np.argsort(perm)
    for e in range(E):  # the same tokens, renamed
        assert sorted(inv[a["sel"][e]].tolist()) == b["sel"][e].tolist()
    np.testing.assert_allclose(b["y"], a["y"][perm], rtol=1e-12, atol=1e-14)


def test_bucket_rule():
    assert oracle.ec_bucket(4096, 8, 2) == 1024
    assert oracle.ec_bucket(3, 8, 2) == 1          # at least one token per expert
    assert oracle.ec_bucket(100, 4, 2, capacity=500) == 100  # at most T
    assert oracle.ec_bucket(100, 4, 2, capacity=30) == 30
    assert oracle.ec_bucket(0, 4, 2) == 0

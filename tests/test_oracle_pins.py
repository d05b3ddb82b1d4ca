"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test ties one oracle function to something other than the oracle itself:
a worked example printed on a page, a closed form, a special case that reduces
to a library routine (torch / scipy in float64), or brute force on tiny inputs.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as Fn

import oracle
from tests import _golden


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
    """Library form of one SwiGLU expert: down(silu(gate(x)) * up(x)), float64."""
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    return (Fn.linear(Fn.silu(Fn.linear(t(x), t(w1))) * Fn.linear(t(x), t(w3)), t(w2))).numpy()


def _route_from_probs(probs, k):
    """A d = 1 router whose softmax is exactly the given row: logits = log(probs)."""
    logits = np.log(np.asarray(probs, np.float64))
    return _f32([[1.0]]), _f32(logits[:, None])


# ---------------------------------------------------------------- routing pins

@pytest.mark.parametrize("fixture", ["deepdive_weighted_sum.txt", "notes_top2_flowchart.txt"])
def test_worked_example_gates(fixture):
    g = _golden.load(fixture)
    x, wg = _route_from_probs(g["probs"], g["k"][0])
    r = oracle.route(x, wg, g["k"][0], renormalize=True)
    assert list(r["ids"][0]) == g["selected"]
    np.testing.assert_allclose(r["gates"][0], g["gates"], rtol=1e-6)
    np.testing.assert_allclose(r["probs"][0], g["probs"], rtol=1e-6)


def test_notes_flowchart_output_is_weighted_sum_of_experts_3_and_7():
    """y = 0.7*E3(x) + 0.3*E7(x), each expert in its library form."""
    g = _golden.load("notes_top2_flowchart.txt")
    rng = np.random.default_rng(1)
    d, F, E = 16, 24, 8
    L = _layer_f32(rng, 1, d, E, F)
    xr, wg = _route_from_probs(g["probs"], 2)
    r = oracle.route(xr, wg, 2)
    y = oracle.layer_tokens(L["x"], L["w1"], L["w3"], L["w2"], r["ids"], r["gates"])
    e3 = _swiglu_torch(L["x"], L["w1"][3], L["w3"][3], L["w2"][3])
    e7 = _swiglu_torch(L["x"], L["w1"][7], L["w3"][7], L["w2"][7])
    np.testing.assert_allclose(y, 0.7 * e3 + 0.3 * e7, rtol=1e-6, atol=1e-12)


def _brute_topk(s, k):
    return sorted(range(len(s)), key=lambda e: (-s[e], e))[:k]


@pytest.mark.parametrize("E,vals", [(4, (0, 1, 2)), (5, (0, 1, 2)), (3, (0, 1, 2, 3))])
def test_topk_matches_brute_force_sort(E, vals):
    rows = list(itertools.product(vals, repeat=E))
    x = _f32(np.ones((len(rows), 1)))
    for k in range(1, E + 1):
        # scores enter through a d = 1 router: logits_t = W_g[:, 0] * x_t with W_g one column;
        # tokens differ, so fold each row into its own call
        for row in rows:
            r = oracle.route(x[:1], _f32(np.asarray(row)[:, None]), k)
            assert list(r["ids"][0]) == _brute_topk(row, k)
            srt = sorted(row, reverse=True)
            gap = math.inf if k == E else srt[k - 1] - srt[k]
            assert r["margin"][0] == gap


def test_topk_with_selection_bias_closed_form():
    """Bias steers the choice only; gates come from the unbiased softmax."""
    x = _f32([[1.0]])
    wg = _f32([[1.0], [0.9], [0.0]])
    r = oracle.route(x, wg, 2, select_bias=_f32([0.0, 0.0, 2.0]))
    assert list(r["ids"][0]) == [2, 0]
    e = math.e
    np.testing.assert_allclose(r["gates"][0], [1 / (1 + e), e / (1 + e)], rtol=1e-7)
    # no renormalisation: raw unbiased probabilities
    r = oracle.route(x, wg, 2, select_bias=_f32([0.0, 0.0, 2.0]), renormalize=False)
    z = e + math.exp(0.9) + 1.0
    np.testing.assert_allclose(r["gates"][0], [1 / z, e / z], rtol=1e-6)


def test_softmax_matches_scipy_and_topk_then_softmax_form():
    rng = np.random.default_rng(2)
    T, d, E, k = 40, 32, 12, 3
    x = _f32(rng.standard_normal((T, d)))
    wg = _f32(rng.standard_normal((E, d)) / math.sqrt(d))
    lb = _f32(rng.standard_normal(E))
    r = oracle.route(x, wg, k, logit_bias=lb)
    logits = x.astype(np.float64) @ wg.astype(np.float64).T + lb.astype(np.float64)
    np.testing.assert_allclose(r["probs"], scipy.special.softmax(logits, axis=1), rtol=1e-12)
    # "MoE Architecture" route(): top-k of the scores, then softmax over the k chosen
    sel = np.take_along_axis(logits, r["ids"].astype(np.int64), axis=1)
    np.testing.assert_allclose(r["gates"], scipy.special.softmax(sel, axis=1), rtol=1e-12)
    np.testing.assert_allclose(r["gates"].sum(1), 1.0, rtol=0, atol=1e-14)


# gates_for_ids evaluates the gates of ids chosen elsewhere (the GPU's, for a
# token inside the top-k margin); every parity comparison of y uses it.

@pytest.mark.parametrize("renorm", [True, False])
def test_gates_for_ids_reproduces_route_gates(renorm):
    """On the router's own ids the gates are the router's, bit for bit
    (logit and selection biases on, so the ids are not just the top-k of p)."""
    rng = np.random.default_rng(21)
    T, d, E, k = 64, 24, 16, 4
    x = _f32(rng.standard_normal((T, d)))
    wg = _f32(rng.standard_normal((E, d)) / math.sqrt(d))
    r = oracle.route(x, wg, k, logit_bias=_f32(rng.standard_normal(E)),
                     select_bias=_f32(rng.uniform(-0.5, 0.5, E)), renormalize=renorm)
    np.testing.assert_array_equal(oracle.gates_for_ids(r["probs"], r["ids"], renorm), r["gates"])


@pytest.mark.parametrize("renorm", [True, False])
def test_gates_for_ids_follow_the_ids_not_the_slots(renorm):
    """Permuting a token's ids permutes its gates the same way (up to the
    rounding of the renormalising sum, whose order follows the slots)."""
    rng = np.random.default_rng(22)
    T, E, k = 50, 10, 3
    probs = scipy.special.softmax(rng.standard_normal((T, E)), axis=1)
    ids = np.array([rng.choice(E, k, replace=False) for _ in range(T)], np.int32)
    g = oracle.gates_for_ids(probs, ids, renorm)
    perm = np.array([rng.permutation(k) for _ in range(T)])
    gp = oracle.gates_for_ids(probs, np.take_along_axis(ids, perm, axis=1), renorm)
    np.testing.assert_allclose(gp, np.take_along_axis(g, perm, axis=1), rtol=1e-15, atol=0)


@pytest.mark.parametrize("renorm", [True, False])
def test_gates_for_ids_equal_softmax_of_the_chosen_logits(renorm):
    """For any k distinct ids (not only the top k): renormalised gates are the
    softmax over the chosen logits alone ("MoE Architecture" route()), plain
    gates are the full softmax at those ids; both written with scipy from the
    logits, not from p.  Renormalising over all E, or taking p by slot, fails."""
    rng = np.random.default_rng(23)
    T, E, k = 40, 12, 5
    logits = rng.standard_normal((T, E)) * 2.0
    probs = scipy.special.softmax(logits, axis=1)
    ids = np.array([rng.choice(E, k, replace=False) for _ in range(T)], np.int32)
    g = oracle.gates_for_ids(probs, ids, renorm)
    sel = np.take_along_axis(logits, ids.astype(np.int64), axis=1)
    ref = scipy.special.softmax(sel, axis=1) if renorm else \
        np.take_along_axis(scipy.special.softmax(logits, axis=1), ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(g, ref, rtol=1e-12, atol=0)


def test_gates_for_ids_worked_example():
    """Deep Dive, Weighted Sum Output: 0.55 and 0.3 become 0.55/0.85 and 0.3/0.85,
    in either slot order; without renormalisation they stay 0.55 and 0.3."""
    gd = _golden.load("deepdive_weighted_sum.txt")
    probs = np.asarray([gd["probs"]], np.float64)
    a, b = gd["selected"]
    g = oracle.gates_for_ids(probs, np.array([[a, b]], np.int32), True)
    np.testing.assert_allclose(g[0], gd["gates"], rtol=1e-15)
    g = oracle.gates_for_ids(probs, np.array([[b, a]], np.int32), True)
    np.testing.assert_allclose(g[0], gd["gates"][::-1], rtol=1e-15)
    g = oracle.gates_for_ids(probs, np.array([[a, b]], np.int32), False)
    np.testing.assert_array_equal(g[0], [gd["probs"][a], gd["probs"][b]])
    with pytest.raises(RuntimeError):
        oracle.gates_for_ids(probs, np.array([[a, len(gd["probs"])]], np.int32), True)


def test_bf16_inputs_are_widened_exactly():
    rng = np.random.default_rng(3)
    T, d, E, F, k = 6, 16, 4, 8, 2
    L = _layer_f32(rng, T, d, E, F)
    Lb = {n: (torch.from_numpy(a).to(torch.bfloat16)) for n, a in L.items()}
    Lbits = {n: t.view(torch.int16).numpy().view(np.uint16) for n, t in Lb.items()}
    Lf = {n: t.float().numpy() for n, t in Lb.items()}
    a = oracle.forward(Lbits, k)
    b = oracle.forward(Lf, k)
    assert np.array_equal(a["ids"], b["ids"])
    assert np.array_equal(a["y"], b["y"])


# ------------------------------------------------------------ expert / layer pins

@pytest.mark.parametrize("renorm", [True, False])
def test_single_expert_is_plain_swiglu(renorm):
    rng = np.random.default_rng(4)
    L = _layer_f32(rng, 9, 24, 1, 40)
    out = oracle.forward(L, 1, renormalize=renorm)
    np.testing.assert_array_equal(out["gates"], 1.0)
    ref = _swiglu_torch(L["x"], L["w1"][0], L["w3"][0], L["w2"][0])
    np.testing.assert_allclose(out["y"], ref, rtol=1e-10, atol=1e-13)


def test_dense_limit_k_equals_E_without_renorm():
    rng = np.random.default_rng(5)
    T, d, E, F = 7, 16, 5, 12
    L = _layer_f32(rng, T, d, E, F)
    out = oracle.forward(L, E, renormalize=False)
    logits = torch.from_numpy(L["x"]).double() @ torch.from_numpy(L["w_gate"]).double().T
    p = torch.softmax(logits, dim=1).numpy()
    ref = sum(p[:, [e]] * _swiglu_torch(L["x"], L["w1"][e], L["w3"][e], L["w2"][e]) for e in range(E))
    np.testing.assert_allclose(out["y"], ref, rtol=1e-10, atol=1e-13)


def test_shared_expert_adds_unweighted():
    rng = np.random.default_rng(6)
    T, d, E, F, k = 5, 16, 4, 8, 2
    L = _layer_f32(rng, T, d, E, F, shared=True)
    with_s = oracle.forward(L, k)["y"]
    no_s = oracle.forward({n: v for n, v in L.items() if not n.startswith("ws")}, k)["y"]
    np.testing.assert_allclose(with_s - no_s, _swiglu_torch(L["x"], L["ws1"], L["ws3"], L["ws2"]),
                               rtol=1e-9, atol=1e-12)


def test_naive_equals_grouped_on_the_handbooks_shape():
    """The handbook checks forward_naive against forward_grouped on T=50, d=64,
    F=128, E=16, k=4 with one shared expert; here the oracle's naive rows are
    compared with a grouped evaluation built from the oracle's own grouping
    (segments of sorted_token_ids, library matmuls per expert)."""
    rng = np.random.default_rng(0)
    T, d, F, E, k = 50, 64, 128, 16, 4
    L = _layer_f32(rng, T, d, E, F, shared=True)
    out = oracle.forward(L, k)
    flat_at = np.full(T * k, -1, np.int64)
    sp = out["slot_pos"].reshape(-1)
    flat_at[sp[sp >= 0]] = np.nonzero(sp >= 0)[0]
    grouped = _swiglu_torch(L["x"], L["ws1"], L["ws3"], L["ws2"])
    for e in range(E):
        lo, hi = out["offsets"][e], out["offsets"][e + 1]
        if lo == hi:
            continue
        tok = out["sorted_token_ids"][lo:hi]
        ye = _swiglu_torch(L["x"][tok], L["w1"][e], L["w3"][e], L["w2"][e])
        w = out["gates"].reshape(-1)[flat_at[lo:hi]]
        np.add.at(grouped, tok, ye * w[:, None])
    np.testing.assert_allclose(out["y"], grouped, rtol=1e-10, atol=1e-12)


def test_permutation_equivariance():
    rng = np.random.default_rng(7)
    T, d, E, F, k = 33, 16, 6, 20, 2
    L = _layer_f32(rng, T, d, E, F, shared=True)
    perm = rng.permutation(T)
    a = oracle.forward(L, k)
    Lp = dict(L, x=np.ascontiguousarray(L["x"][perm]))
    b = oracle.forward(Lp, k)
    np.testing.assert_array_equal(b["ids"], a["ids"][perm])
    np.testing.assert_array_equal(b["counts"], a["counts"])
    np.testing.assert_allclose(b["y"], a["y"][perm], rtol=1e-12, atol=1e-14)


def test_capacity_on_a_single_expert_keeps_the_first_tokens():
    rng = np.random.default_rng(8)
    T, d, F, C = 10, 8, 12, 4
    L = _layer_f32(rng, T, d, 1, F)
    out = oracle.forward(L, 1, capacity=C)
    ref = _swiglu_torch(L["x"], L["w1"][0], L["w3"][0], L["w2"][0])
    ref[C:] = 0.0
    np.testing.assert_allclose(out["y"], ref, rtol=1e-10, atol=1e-13)
    assert out["n_dropped"] == T - C and list(out["kept"]) == [C]


# ------------------------------------------------------------------ grouping pins

def _brute_group(ids, E, C):
    T, k = ids.shape
    entries = {e: [(t, j) for t in range(T) for j in range(k) if ids[t, j] == e] for e in range(E)}
    counts = [len(entries[e]) for e in range(E)]
    kept = [len(entries[e]) if C < 0 else min(C, len(entries[e])) for e in range(E)]
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + kept[e])
    slot = np.full((T, k), -1)
    sorted_tok = []
    for e in range(E):
        for r, (t, j) in enumerate(entries[e][:kept[e]]):
            slot[t, j] = offsets[e] + r
            sorted_tok.append(t)
    return counts, kept, offsets, slot, sorted_tok


@pytest.mark.parametrize("C", [-1, 0, 1, 2, 3, 5])
def test_grouping_matches_brute_force(C):
    rng = np.random.default_rng(9 + C)
    T, E, k = 13, 4, 2
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    g = oracle.group(ids, E, C)
    counts, kept, offsets, slot, sorted_tok = _brute_group(ids, E, C)
    assert list(g["counts"]) == counts
    assert list(g["kept"]) == kept
    assert list(g["offsets"]) == offsets
    np.testing.assert_array_equal(g["slot_pos"], slot)
    assert list(g["sorted_token_ids"][:offsets[-1]]) == sorted_tok
    assert all(v == -1 for v in g["sorted_token_ids"][offsets[-1]:])
    assert g["n_dropped"] == T * k - offsets[-1]


def test_grouping_invariants_on_random_routing():
    rng = np.random.default_rng(10)
    T, d, E, k = 500, 32, 24, 3
    x = _f32(rng.standard_normal((T, d)))
    wg = _f32(rng.standard_normal((E, d)))
    r = oracle.route(x, wg, k)
    for C in (-1, 40, 70):
        g = oracle.group(r["ids"], E, C)
        assert g["counts"].sum() == T * k
        assert g["kept"].sum() + g["n_dropped"] == T * k
        if C >= 0:
            assert (g["kept"] <= C).all()
        assert g["offsets"][-1] == g["kept"].sum() and (np.diff(g["offsets"]) >= 0).all()
        for e in range(E):
            seg = g["sorted_token_ids"][g["offsets"][e]:g["offsets"][e + 1]]
            assert (np.diff(seg) > 0).all()
        sp = g["slot_pos"]
        tk = np.nonzero(sp >= 0)
        assert (g["sorted_token_ids"][sp[tk]] == tk[0]).all()


# --------------------------------------------------------------- load statistic pins

def test_lbalance_uniform_probabilities_give_alpha_for_any_f():
    rng = np.random.default_rng(11)
    T, d, E, k = 64, 8, 8, 2
    x = _f32(rng.standard_normal((T, d)))
    wg = _f32(np.zeros((E, d)))
    r = oracle.route(x, wg, k)
    np.testing.assert_array_equal(r["probs"], 1.0 / E)
    g = oracle.group(r["ids"], E)
    assert g["counts"][0] == T  # every tie goes to the lowest indices: f far from uniform
    st = oracle.load_stats(g["counts"], r["probs"], k, 0.01)
    assert abs(st["L"] - 0.01) < 1e-15


def test_lbalance_uniform_routing_gives_alpha_for_any_p():
    E, m = 8, 5
    T = E * m
    x = _f32(10.0 * np.eye(E)[np.arange(T) % E])
    wg = _f32(np.eye(E) + 0.1 * np.random.default_rng(12).standard_normal((E, E)))
    r = oracle.route(x, wg, 1)
    g = oracle.group(r["ids"], E)
    np.testing.assert_array_equal(g["counts"], m)
    st = oracle.load_stats(g["counts"], r["probs"], 1, 0.01)
    np.testing.assert_allclose(st["f"], 1.0 / E, rtol=0, atol=1e-16)
    assert abs(st["L"] - 0.01) < 1e-15


def test_lbalance_handbook_skewed_example():
    g = _golden.load("handbook_aux_skewed.txt")
    E, T, k = g["E"][0], g["T"][0], g["k"][0]
    probs = np.zeros((T, E))
    probs[:, g["hot_experts"]] = g["hot_prob"][0]
    counts = np.zeros(E, np.int32)
    counts[g["hot_experts"]] = T
    st = oracle.load_stats(counts, probs, k, 1.0)
    assert abs(st["L"] - g["expected_loss"][0]) < 1e-12


def test_lbalance_random_router_is_near_one():
    rng = np.random.default_rng(13)
    T, d, E, k = 4096, 64, 16, 4
    x = _f32(rng.standard_normal((T, d)))
    wg = _f32(rng.standard_normal((E, d)) / math.sqrt(d))
    r = oracle.route(x, wg, k)
    g = oracle.group(r["ids"], E)
    st = oracle.load_stats(g["counts"], r["probs"], k, 1.0)
    assert 0.98 < st["L"] < 1.15
    np.testing.assert_allclose(st["f"].sum(), 1.0, rtol=1e-14)
    np.testing.assert_allclose(st["p"].sum(), 1.0, rtol=1e-12)


# ------------------------------------------------------------ work accounting pin

def test_expert_parameter_arithmetic_matches_the_handbook_exercise():
    import moe_inputs
    g = _golden.load("handbook_exercise_params.txt")
    pe = moe_inputs.expert_params(g["d"][0], g["F"][0])
    assert pe == 8_650_752
    total = g["E"][0] * pe * g["layers"][0]
    active = g["k"][0] * pe * g["layers"][0]
    assert round(total / 1e9, 2) == g["total_billions"][0]
    assert round(active / 1e9, 2) == g["active_billions"][0]


# ------------------------------------------------------- selection-bias update pins

def test_bias_update_direction_matches_the_pages():
    g = _golden.load("bias_update_direction.txt")
    out = oracle.bias_update(np.array(g["counts"]), np.array(g["bias"], np.float32), g["T"][0], g["k"][0],
                             g["gamma"][0])
    expected = np.array(g["bias"]) + g["gamma"][0] * np.array(g["direction"], np.float64)
    np.testing.assert_array_equal(out, expected)


def test_bias_update_leaves_balanced_loads_alone_and_is_exact_in_integers():
    E, T, k = 8, 64, 2
    counts = np.full(E, T * k // E, np.int32)
    b = np.linspace(-1, 1, E).astype(np.float32)
    np.testing.assert_array_equal(oracle.bias_update(counts, b, T, k, 0.01), b.astype(np.float64))
    # the mean T*k/E = 16.5 is fractional: loads 16 and 17 sit on either side of it
    T, k, E = 33, 2, 4
    counts = np.array([17, 16, 17, 16], np.int32)
    out = oracle.bias_update(counts, np.zeros(E, np.float32), T, k, 0.5)
    np.testing.assert_array_equal(out, [-0.5, 0.5, -0.5, 0.5])


def test_bias_update_moves_routing_towards_balance():
    """Iterating route -> count -> update on a skewed router lowers the load of
    the most popular expert (the purpose the pages give for the bias)."""
    rng = np.random.default_rng(21)
    T, d, E, k = 512, 16, 8, 2
    x = _f32(rng.standard_normal((T, d)))
    wg = _f32(rng.standard_normal((E, d)) / math.sqrt(d))
    lb = _f32(np.log(np.arange(1, E + 1) ** -1.5))  # Zipf-like skew on the logits
    bias = np.zeros(E, np.float32)
    first = None
    for _ in range(40):
        r = oracle.route(x, wg, k, logit_bias=lb, select_bias=bias)
        counts = oracle.group(r["ids"], E)["counts"]
        first = counts.copy() if first is None else first
        bias = oracle.bias_update(counts, bias, T, k, 0.05).astype(np.float32)
    assert counts.max() < first.max()
    assert np.abs(counts - T * k / E).sum() < np.abs(first - T * k / E).sum()

"""GPU-vs-oracle parity harness (test infrastructure).

``check_layer`` draws a workload's inputs on the GPU, runs the CUDA library
through its C entry points (step by step and fused), runs the fp64 oracle on
the very same tensors and returns a report of every comparison:

* routing: for every token whose oracle margin between the k-th and (k+1)-th
  selection score exceeds 1e-3, the GPU's set of ids equals the oracle's;
  tokens inside the margin must still be a valid top-k (every chosen score
  >= every unchosen score - 1e-3).  Gates are compared by id (abs 1e-5).
* grouping: counts, kept, offsets, sorted_token_ids, slot_pos, n_dropped are
  compared BIT-EXACTLY with the oracle's grouping of the GPU's ids, and with
  the oracle's own grouping when no token is inside the margin.
* x_perm: bit-exact row gather.
* y: max |y_gpu - y_oracle| <= tol * RMS(y_oracle) over the checked tokens
  (all tokens, or for the large workloads a seeded sample plus the tokens at
  the first and last row of every 64-row block of every expert segment, so
  every output tile of the launch has checked rows), with tol = 2e-2
  for bf16 and 1e-4 for fp32; the oracle evaluates y with the GPU's ids.
  For bf16 layers the tolerance applies to the layer's fp32 result (the
  library's y_fp32 output): rounding the output itself to bf16 costs up to
  half an ulp, 2^-8 |y|, which alone exceeds 2e-2 RMS(y) wherever
  |y| > 5.1 RMS(y).  The stored bf16 output must then equal the
  round-to-nearest-even of that fp32 result bit for bit.
* statistics: f exact, p and L within fp32 summation error.
* determinism: two fused calls give bit-identical y; the fused call equals
  the chain of separate entry points bit for bit.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

import mixture_experts_layer_95_b300 as moe
import moe_inputs
import oracle

MARGIN = 1e-3
TOL = {"bf16": 2e-2, "f32": 1e-4}


def layer_of(w: moe_inputs.Workload) -> moe.Layer:
    return moe.Layer(T=w.T, d=w.d, E=w.E, k=w.k, d_ff=w.F, n_shared=w.n_shared, d_ff_shared=w.F_s, dtype=w.dtype,
                     renormalize=w.renormalize, capacity=w.capacity, alpha=w.alpha, h_split=w.h_split,
                     routing=w.routing, yperm_bf16=w.yperm_bf16)


def sample_tokens(T: int, n: int, seed: int = 1234, must=()) -> np.ndarray:
    if n >= T:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, n, replace=False).tolist()) | {0, T - 1} | set(int(t) for t in must if 0 <= t < T)
    return np.array(sorted(pick), dtype=np.int32)


def tile_cover_tokens(offsets, sorted_token_ids, step: int = 64) -> np.ndarray:
    """Tokens whose rows are the first and the last row of every `step`-row
    block of every expert segment.  The GEMMs cut each segment into 128-row
    (1-CTA), 256-row (CTA-pair) or 64-row tiles that all start on a multiple of
    64 rows from the segment start, so a 64-row cover puts a checked output row
    in every tile of every expert, whichever kernel ran."""
    rows = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for b in range(lo, hi, step):
            rows += [b, min(b + step, hi) - 1]
    return np.unique(np.asarray(sorted_token_ids, np.int64)[np.asarray(rows, np.int64)]) if rows else \
        np.zeros(0, np.int64)


def run_gpu(w: moe_inputs.Workload, L: dict, layer: moe.Layer):
    """Separate entry points, then the fused call twice."""
    ws = moe.workspace(layer)
    ids, gates, p_mean = moe.route(layer, L["x"], L["w_gate"], L["logit_bias"], L["select_bias"], ws=ws)
    g = moe.permute(layer, ids, gates, L["x"], ws=ws)
    y_perm, y_shared = moe.expert_ffn(layer, g["x_perm"], g["offsets"], g["gates_perm"], L["w1"], L["w3"], L["w2"],
                                      L["x"], L["ws1"], L["ws3"], L["ws2"], ws=ws)
    y_steps = moe.combine(layer, y_perm, g["slot_pos"], y_shared)
    f, Lb = moe.load_stats(layer, g["counts"], p_mean)
    status_steps = moe.last_device_status(layer, ws)
    fw = moe.Forward(layer, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"], L["ws1"],
                     L["ws3"], L["ws2"], stats=True)
    y1 = fw(L["x"])
    y2 = fw(L["x"])
    status_fused = fw.device_status()
    layer32 = dataclasses.replace(layer, y_fp32=True)
    fw32 = moe.Forward(layer32, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], L["select_bias"], L["ws1"],
                       L["ws3"], L["ws2"])
    y32 = fw32(L["x"])
    status_fused |= fw32.device_status()
    torch.cuda.synchronize()
    return dict(ids=ids, gates=gates, p_mean=p_mean, group=g, y_perm=y_perm, y_steps=y_steps, f=f, L=Lb,
                y1=y1, y2=y2, y32=y32, stats=fw.stats, status_steps=status_steps, status_fused=status_fused)


def check_layer(w: moe_inputs.Workload, n_sample: int | None = None, L: dict | None = None) -> dict:
    """Runs one workload on cuda:0 and the oracle; returns a report dict with
    'ok' and the individual measurements."""
    layer = layer_of(w)
    if L is None:
        L = moe_inputs.make_layer(w, "cuda")
    G = run_gpu(w, L, layer)
    rep = dict(workload=w.name, status_steps=G["status_steps"], status_fused=G["status_fused"])
    Ln = moe_inputs.layer_numpy(L)

    # ---- routing ----
    r = oracle.route(Ln["x"], Ln["w_gate"], w.k, Ln["logit_bias"], Ln["select_bias"], w.renormalize)
    gids = G["ids"].cpu().numpy()
    ggates = G["gates"].cpu().numpy()
    outside = r["margin"] > MARGIN
    same_set = np.array([set(a) == set(b) for a, b in zip(gids.tolist(), r["ids"].tolist())])
    rep["ids_mismatch_outside_margin"] = int((~same_set & outside).sum())
    rep["tokens_inside_margin"] = int((~outside).sum())
    # validity of every GPU choice against the oracle's scores
    scores = np.log(np.maximum(r["probs"], 1e-300))  # softmax is monotone: compare via log p + select_bias
    if Ln["select_bias"] is not None:
        scores = scores + Ln["select_bias"][None, :].astype(np.float64)
    chosen = np.zeros_like(scores, dtype=bool)
    np.put_along_axis(chosen, gids.astype(np.int64), True, axis=1)
    min_chosen = np.where(chosen, scores, np.inf).min(1)
    max_unchosen = np.where(chosen, -np.inf, scores).max(1)
    rep["invalid_topk_tokens"] = int((min_chosen < max_unchosen - MARGIN).sum())
    rep["duplicate_ids"] = int(sum(len(set(row)) != len(row) for row in gids.tolist()))
    ogates_for_gpu = oracle.gates_for_ids(r["probs"], gids, w.renormalize)
    rep["gates_max_abs_err"] = float(np.abs(ggates - ogates_for_gpu).max()) if gids.size else 0.0

    # ---- grouping (bit-exact, as a function of the GPU's ids) ----
    og = oracle.group(gids, w.E, w.capacity)
    gg = {k_: v.cpu().numpy() for k_, v in G["group"].items() if k_ != "x_perm"}
    grouping_equal = all(np.array_equal(gg[name].reshape(-1), og[name].reshape(-1))
                         for name in ("counts", "kept", "offsets", "sorted_token_ids", "slot_pos"))
    grouping_equal = grouping_equal and int(gg["n_dropped"][0]) == og["n_dropped"]
    rep["grouping_bit_exact"] = bool(grouping_equal)
    if rep["tokens_inside_margin"] == 0:
        og_own = oracle.group(r["ids"], w.E, w.capacity)
        rep["grouping_matches_oracle_routing"] = bool(
            all(np.array_equal(gg[name].reshape(-1), og_own[name].reshape(-1))
                for name in ("counts", "kept", "offsets", "sorted_token_ids", "slot_pos")))
    total = int(og["offsets"][-1])
    xp = G["group"]["x_perm"][:total]
    src = L["x"][torch.from_numpy(og["sorted_token_ids"][:total].astype(np.int64)).to(xp.device)]
    rep["x_perm_bit_exact"] = bool(torch.equal(xp, src))
    rep["n_dropped"] = og["n_dropped"]

    # ---- layer output ----
    # a sampled check also covers every (expert, row tile) of the launch
    must = np.nonzero((og["slot_pos"] < 0).any(1))[0][:8] if og["n_dropped"] else np.zeros(0, np.int64)
    if n_sample:
        must = np.concatenate([must, tile_cover_tokens(og["offsets"], og["sorted_token_ids"])])
        if w.n_shared:  # the shared expert's problem has one row per token
            must = np.concatenate([must, tile_cover_tokens([0, w.T], np.arange(w.T))])
    toks = sample_tokens(w.T, n_sample if n_sample else w.T, must=must)
    y_or = oracle.layer_tokens(Ln["x"], Ln["w1"], Ln["w3"], Ln["w2"], gids, ogates_for_gpu, og["slot_pos"], toks,
                               (Ln["ws1"], Ln["ws3"], Ln["ws2"]) if w.n_shared else None)
    y_gpu = G["y32"].cpu().numpy()[toks].astype(np.float64)
    y_stored = G["y1"].float().cpu().numpy()[toks].astype(np.float64)
    rms = float(np.sqrt(np.mean(y_or ** 2))) if y_or.size else 0.0
    err = float(np.abs(y_gpu - y_or).max()) if y_or.size else 0.0
    err_stored = float(np.abs(y_stored - y_or).max()) if y_or.size else 0.0
    rep.update(y_rms=rms, y_max_abs_err=err, y_rel=err / rms if rms > 0 else err, tol=TOL[w.dtype],
               y_rel_stored=err_stored / rms if rms > 0 else err_stored, y_tokens_checked=int(len(toks)),
               y_max_over_rms=float(np.abs(y_or).max() / rms) if rms > 0 else 0.0)
    rep["y_stored_is_rne_of_fp32"] = bool(torch.equal(G["y1"], G["y32"].to(G["y1"].dtype)))
    rep["y_deterministic"] = bool(torch.equal(G["y1"], G["y2"]))
    rep["fused_path"] = moe.plan_describe(layer.cfg())["up"] == "fused"
    if rep["fused_path"]:
        # the two fused small-batch kernels add in their own order: moe_forward
        # and the step-by-step entry points then agree to the bf16 rule, each
        # against the oracle
        y_st = G["y_steps"].float().cpu().numpy()[toks].astype(np.float64)
        err_st = float(np.abs(y_st - y_or).max()) if y_or.size else 0.0
        rep["y_rel_steps"] = err_st / rms if rms > 0 else err_st
        rep["fused_equals_steps"] = bool(rep["y_rel_steps"] <= TOL[w.dtype])
    else:
        rep["fused_equals_steps"] = bool(torch.equal(G["y1"], G["y_steps"]))

    # ---- statistics ----
    st = oracle.load_stats(og["counts"], r["probs"], w.k, w.alpha)
    s = {k_: v.cpu().numpy() for k_, v in G["stats"].items()}
    rep["stats_counts_exact"] = bool(np.array_equal(s["counts"], og["counts"]) and
                                     np.array_equal(s["kept"], og["kept"]) and
                                     int(s["n_dropped"][0]) == og["n_dropped"])
    rep["f_max_abs_err"] = float(np.abs(s["f"] - st["f"]).max())
    rep["p_max_abs_err"] = float(np.abs(s["p"] - st["p"]).max())
    rep["L_abs_err"] = float(abs(float(s["L"][0]) - st["L"]))
    rep["L"] = float(s["L"][0])
    rep["steps_stats_equal"] = bool(np.allclose(G["f"].cpu().numpy(), s["f"], rtol=0, atol=0) and
                                    abs(float(G["L"].cpu().numpy()[0]) - float(s["L"][0])) <= 1e-6 * max(1.0, abs(st["L"])))
    p_tol = 1e-5 + 1e-6 * math.sqrt(w.T)
    rep["ok"] = bool(
        rep["status_steps"] == 0 and rep["status_fused"] == 0 and rep["ids_mismatch_outside_margin"] == 0
        and rep["invalid_topk_tokens"] == 0 and rep["duplicate_ids"] == 0 and rep["gates_max_abs_err"] < 1e-5
        and rep["grouping_bit_exact"] and rep.get("grouping_matches_oracle_routing", True)
        and rep["x_perm_bit_exact"] and rep["y_rel"] <= rep["tol"] and rep["y_stored_is_rne_of_fp32"]
        and rep["y_deterministic"]
        and rep["fused_equals_steps"] and rep["stats_counts_exact"] and rep["f_max_abs_err"] <= 1e-7
        and rep["p_max_abs_err"] <= p_tol and rep["L_abs_err"] <= 1e-5 * max(1.0, abs(st["L"]))
        and rep["steps_stats_equal"])
    return rep


# ---------------------------------------------------------------- expert choice

EC_MARGIN = 1e-5  # score gap at a bucket boundary beyond fp32-vs-fp64 softmax error


def run_gpu_ec(L: dict, layer: moe.Layer):
    """Expert choice: the step entry points, then the fused call twice (+ fp32 y)."""
    ws = moe.workspace(layer)
    r = moe.route_expert_choice(layer, L["x"], L["w_gate"], L["logit_bias"], ws=ws)
    y_perm, y_shared = moe.expert_ffn(layer, r["x_perm"], r["offsets"], r["gates_perm"], L["w1"], L["w3"], L["w2"],
                                      L["x"], L["ws1"], L["ws3"], L["ws2"], ws=ws)
    y_steps = moe.combine(layer, y_perm, r["slot_pos"], y_shared)
    counts = torch.full((layer.E,), layer.bucket, dtype=torch.int32, device=L["x"].device)
    f, Lb = moe.load_stats(layer, counts, r["p_mean"])
    status_steps = moe.last_device_status(layer, ws)
    fw = moe.Forward(layer, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], None, L["ws1"], L["ws3"],
                     L["ws2"], stats=True)
    y1 = fw(L["x"])
    y2 = fw(L["x"])
    status_fused = fw.device_status()
    layer32 = dataclasses.replace(layer, y_fp32=True)
    fw32 = moe.Forward(layer32, L["w_gate"], L["w1"], L["w3"], L["w2"], L["logit_bias"], None, L["ws1"], L["ws3"],
                       L["ws2"])
    y32 = fw32(L["x"])
    status_fused |= fw32.device_status()
    torch.cuda.synchronize()
    return dict(route=r, y_steps=y_steps, f=f, L=Lb, y1=y1, y2=y2, y32=y32, stats=fw.stats,
                status_steps=status_steps, status_fused=status_fused)


def check_layer_ec(w: moe_inputs.Workload, n_sample: int | None = None, L: dict | None = None) -> dict:
    """Expert-choice parity.  Selection: for every expert whose oracle gap
    between its C-th and (C+1)-th score exceeds EC_MARGIN, the GPU's bucket
    equals the oracle's; every bucket must be valid (each chosen score >=
    each unchosen score - EC_MARGIN), distinct and ascending.  The slot map,
    offsets, x_perm and the empty-token count are compared bit-exactly with
    the oracle's slot form of the GPU's buckets; y against the oracle
    evaluated on those buckets; statistics against the closed forms."""
    layer = layer_of(w)
    C = layer.bucket
    assert C == oracle.ec_bucket(w.T, w.E, w.k, w.capacity)
    if L is None:
        L = moe_inputs.make_layer(w, "cuda")
    G = run_gpu_ec(L, layer)
    rep = dict(workload=w.name, C=C, status_steps=G["status_steps"], status_fused=G["status_fused"])
    Ln = moe_inputs.layer_numpy(L)
    r = oracle.route(Ln["x"], Ln["w_gate"], 1, Ln["logit_bias"], None, True)
    probs = r["probs"]
    own_sel, margin = oracle.ec_select(probs, C)
    R = {k_: v.cpu().numpy() for k_, v in G["route"].items() if k_ != "x_perm"}
    rep["probs_max_abs_err"] = float(np.abs(R["probs"] - probs).max())
    gsel = R["sorted_token_ids"].reshape(w.E, C)
    outside = margin > EC_MARGIN
    same = np.array([np.array_equal(gsel[e], own_sel[e]) for e in range(w.E)])
    rep["experts_inside_margin"] = int((~outside).sum())
    rep["bucket_mismatch_outside_margin"] = int((~same & outside).sum())
    rep["buckets_equal_oracle"] = bool(same.all())
    bad = 0
    for e in range(w.E):
        row = gsel[e]
        if not (np.all(np.diff(row) > 0) and row.min() >= 0 and row.max() < w.T):
            bad += 1
            continue
        chosen = np.zeros(w.T, bool)
        chosen[row] = True
        if chosen.all():
            continue
        if probs[chosen, e].min() < probs[~chosen, e].max() - EC_MARGIN:
            bad += 1
    rep["invalid_buckets"] = bad
    sl = oracle.ec_slots(gsel, probs)
    rep["slots_bit_exact"] = bool(np.array_equal(R["slot_pos"], sl["slot_pos"]))
    rep["offsets_exact"] = bool(np.array_equal(R["offsets"], np.arange(w.E + 1) * C))
    # gates: the GPU's own scores at the chosen pairs, and close to the oracle's
    gp = R["gates_perm"].reshape(w.E, C)
    own = np.array([R["probs"][gsel[e], e] for e in range(w.E)])
    rep["gates_are_gpu_scores"] = bool(np.array_equal(gp, own))
    xp = G["route"]["x_perm"]
    src = L["x"][torch.from_numpy(R["sorted_token_ids"].astype(np.int64)).to(xp.device)]
    rep["x_perm_bit_exact"] = bool(torch.equal(xp, src))

    must = tile_cover_tokens(R["offsets"], R["sorted_token_ids"]) if n_sample else ()
    toks = sample_tokens(w.T, n_sample if n_sample else w.T, must=must)
    y_or = oracle.layer_tokens(Ln["x"], Ln["w1"], Ln["w3"], Ln["w2"], sl["ids"], sl["gates"], sl["slot_pos"], toks,
                               (Ln["ws1"], Ln["ws3"], Ln["ws2"]) if w.n_shared else None)
    y_gpu = G["y32"].cpu().numpy()[toks].astype(np.float64)
    rms = float(np.sqrt(np.mean(y_or ** 2))) if y_or.size else 0.0
    err = float(np.abs(y_gpu - y_or).max()) if y_or.size else 0.0
    rep.update(y_rms=rms, y_max_abs_err=err, y_rel=err / rms if rms > 0 else err, tol=TOL[w.dtype],
               y_tokens_checked=int(len(toks)))
    rep["y_stored_is_rne_of_fp32"] = bool(torch.equal(G["y1"], G["y32"].to(G["y1"].dtype)))
    rep["y_deterministic"] = bool(torch.equal(G["y1"], G["y2"]))
    rep["fused_equals_steps"] = bool(torch.equal(G["y1"], G["y_steps"]))

    s = {k_: v.cpu().numpy() for k_, v in G["stats"].items()}
    rep["n_empty"] = sl["n_empty"]
    rep["stats_counts_exact"] = bool(np.all(s["counts"] == C) and np.all(s["kept"] == C)
                                     and int(s["n_dropped"][0]) == sl["n_empty"])
    st_p = probs.mean(axis=0)
    rep["f_max_abs_err"] = float(np.abs(s["f"] - 1.0 / w.E).max())
    rep["p_max_abs_err"] = float(np.abs(s["p"] - st_p).max())
    rep["L"] = float(s["L"][0])
    rep["L_abs_err"] = float(abs(rep["L"] - w.alpha))  # closed form: alpha * sum_e p_e = alpha
    rep["steps_stats_equal"] = bool(np.array_equal(G["f"].cpu().numpy(), s["f"]) and
                                    float(G["L"].cpu().numpy()[0]) == float(s["L"][0]))
    p_tol = 1e-5 + 1e-6 * math.sqrt(w.T)
    rep["ok"] = bool(
        rep["status_steps"] == 0 and rep["status_fused"] == 0 and rep["probs_max_abs_err"] < 1e-5
        and rep["bucket_mismatch_outside_margin"] == 0 and rep["invalid_buckets"] == 0
        and rep["slots_bit_exact"] and rep["offsets_exact"] and rep["gates_are_gpu_scores"]
        and rep["x_perm_bit_exact"] and rep["y_rel"] <= rep["tol"] and rep["y_stored_is_rne_of_fp32"]
        and rep["y_deterministic"] and rep["fused_equals_steps"] and rep["stats_counts_exact"]
        and rep["f_max_abs_err"] <= 1e-7 and rep["p_max_abs_err"] <= p_tol
        and rep["L_abs_err"] <= 1e-5 and rep["steps_stats_equal"])
    return rep


# ---------------------------------------------------------------- FP8 weights

def check_quantize(w_dev) -> dict:
    """GPU per-row E4M3 codes and scales vs the oracle's, bit for bit."""
    q, sc = moe.quantize_fp8(w_dev)
    oq, osc = oracle.quantize_fp8(moe_inputs.to_numpy(w_dev))
    gq, gsc = q.cpu().numpy(), sc.cpu().numpy()
    return dict(codes_equal=bool(np.array_equal(gq, oq)), scales_equal=bool(np.array_equal(gsc, osc)),
                n_code_mismatch=int((gq != oq).sum()))


def _oracle_y_fp8(Ln, q8, w, ids, gates, slot_pos, toks):
    """Oracle y for the listed tokens with the dequantised FP8 experts, one
    expert at a time (only experts some listed token uses are dequantised)."""
    x64 = oracle.widen(Ln["x"])
    y = np.zeros((len(toks), w.d))
    sel = np.zeros_like(ids, dtype=bool)
    sel[toks] = True
    for e in np.unique(ids[toks][slot_pos[toks] >= 0]):
        w1 = oracle.dequant_fp8(q8["w1"][e], q8["s1"][e])[None]
        w3 = oracle.dequant_fp8(q8["w3"][e], q8["s3"][e])[None]
        w2 = oracle.dequant_fp8(q8["w2"][e], q8["s2"][e])[None]
        mine = (ids == e) & sel
        sp = np.where(mine, slot_pos, -1).astype(np.int32)
        y += oracle.layer_tokens(x64, w1, w3, w2, np.zeros_like(ids), gates, sp, toks)
    if w.n_shared:
        sh = tuple(oracle.dequant_fp8(q8[n], q8[s]) for n, s in (("ws1", "ss1"), ("ws3", "ss3"), ("ws2", "ss2")))
        y += oracle.layer_tokens(x64, sh[0][None], sh[1][None], sh[2][None], np.zeros_like(ids), gates,
                                 np.full_like(ids, -1), toks, sh)
    return y


def check_layer_fp8(w: moe_inputs.Workload, n_sample: int | None = None, L: dict | None = None,
                    per_token: bool = False) -> dict:
    """FP8-weight layer: codes and scales bit-exact with the oracle's
    quantisation of the same bf16 weights; routing as the bf16 layer (the
    router is unchanged); y (fp32 result) within the bf16 tolerance of the
    oracle evaluated with the exactly dequantised weights on the GPU's ids;
    bf16 y = RNE(fp32 y); deterministic.  per_token=True holds every token
    to the tolerance against its own RMS instead, for inputs whose token rows
    differ in scale by many orders of magnitude: there the RMS over all
    tokens is one token's RMS / sqrt(T), which would hold that token to a
    sqrt(T) tighter bound than any other layer call gets."""
    layer = layer_of(w)
    if L is None:
        L = moe_inputs.make_layer(w, "cuda")
    names = ["w1", "w3", "w2"] + (["ws1", "ws3", "ws2"] if w.n_shared else [])
    q8 = moe.quantize_experts_fp8(layer, *(L[n] for n in names))
    rep = dict(workload=w.name)
    # quantisation, bit for bit (a row sample of each matrix when large)
    Ln = moe_inputs.layer_numpy(L)
    mism = 0
    for n in names:
        src = Ln[n].reshape(-1, Ln[n].shape[-1])
        rows = np.arange(src.shape[0]) if src.shape[0] <= 4096 else \
            np.random.default_rng(5).choice(src.shape[0], 4096, replace=False)
        oq, osc = oracle.quantize_fp8(np.ascontiguousarray(src[rows]))
        gq = q8[n].reshape(-1, src.shape[1]).cpu().numpy()[rows]
        gs = q8["s" + n[1:]].reshape(-1).cpu().numpy()[rows]
        mism += int((gq != oq).sum()) + int((gs != osc).sum())
    rep["quantisation_mismatches"] = mism
    q8n = {k_: v.cpu().numpy() for k_, v in q8.items()}
    del Ln["w1"], Ln["w3"], Ln["w2"]
    # routing from the GPU router (the same kernels the fused call runs)
    if w.routing == "expert":
        rt = moe.route_expert_choice(layer, L["x"], L["w_gate"], L["logit_bias"], gather=False)
        gsel = rt["sorted_token_ids"].cpu().numpy().reshape(w.E, layer.bucket)
        r = oracle.route(Ln["x"], Ln["w_gate"], 1, Ln["logit_bias"], None, True)
        own, margin = oracle.ec_select(r["probs"], layer.bucket)
        same = np.array([np.array_equal(gsel[e], own[e]) for e in range(w.E)])
        rep["ids_mismatch_outside_margin"] = int((~same & (margin > EC_MARGIN)).sum())
        sl = oracle.ec_slots(gsel, r["probs"])
        gids, ogates, og = sl["ids"], sl["gates"], dict(slot_pos=sl["slot_pos"])
    else:
        ids, gates, _ = moe.route(layer, L["x"], L["w_gate"], L["logit_bias"], L["select_bias"])
        gids = ids.cpu().numpy()
        r = oracle.route(Ln["x"], Ln["w_gate"], w.k, Ln["logit_bias"], Ln["select_bias"], w.renormalize)
        outside = r["margin"] > MARGIN
        same_set = np.array([set(a) == set(b) for a, b in zip(gids.tolist(), r["ids"].tolist())])
        rep["ids_mismatch_outside_margin"] = int((~same_set & outside).sum())
        og = oracle.group(gids, w.E, w.capacity)
        ogates = oracle.gates_for_ids(r["probs"], gids, w.renormalize)
    fw = moe.Forward(layer, L["w_gate"], None, None, None, L["logit_bias"], L["select_bias"], fp8=q8)
    y1 = fw(L["x"])
    y2 = fw(L["x"])
    fw32 = moe.Forward(dataclasses.replace(layer, y_fp32=True), L["w_gate"], None, None, None, L["logit_bias"],
                       L["select_bias"], fp8=q8)
    y32 = fw32(L["x"])
    rep["status"] = fw.device_status() | fw32.device_status()
    toks = sample_tokens(w.T, n_sample if n_sample else w.T)
    y_or = _oracle_y_fp8(Ln, q8n, w, gids, ogates, og["slot_pos"], toks)
    y_gpu = y32.cpu().numpy()[toks].astype(np.float64)
    rms = float(np.sqrt(np.mean(y_or ** 2))) if y_or.size else 0.0
    err = float(np.abs(y_gpu - y_or).max()) if y_or.size else 0.0
    rep.update(y_rms=rms, y_rel=err / rms if rms > 0 else err, tol=TOL["bf16"], y_tokens_checked=int(len(toks)))
    if y_or.size:  # worst token against its own RMS (a zero row must come out exactly zero)
        t_rms = np.sqrt(np.mean(y_or ** 2, axis=1))
        t_err = np.abs(y_gpu - y_or).max(axis=1)
        rel = np.where(t_rms > 0, t_err / np.where(t_rms > 0, t_rms, 1.0), np.where(t_err > 0, np.inf, 0.0))
        rep["y_rel_worst_token"] = float(rel.max())
    rep["y_stored_is_rne_of_fp32"] = bool(torch.equal(y1, y32.to(y1.dtype)))
    rep["y_deterministic"] = bool(torch.equal(y1, y2))
    rep["ok"] = bool(rep["quantisation_mismatches"] == 0 and rep["status"] == 0
                     and rep["ids_mismatch_outside_margin"] == 0
                     and (rep.get("y_rel_worst_token", 0.0) if per_token else rep["y_rel"]) <= rep["tol"]
                     and rep["y_stored_is_rne_of_fp32"] and rep["y_deterministic"])
    return rep

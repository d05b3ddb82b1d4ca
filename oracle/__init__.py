"""Plain fp64 CPU oracle for the MoE SwiGLU layer forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it: the arithmetic lives in ``moe_oracle.c`` (plain C,
double precision, OpenMP over independent tokens) and this module only moves
numpy arrays in and out of it.

Inputs are numpy arrays: ``float32`` for fp32 data, ``uint16`` holding bf16
bit patterns for bf16 data (the oracle widens them exactly).  Every float
result is ``float64``.

Parity status: routing, grouping, the SwiGLU experts, the combine and the load
statistics are each pinned by ``tests/test_oracle_pins.py`` (worked examples
printed on the pages, closed forms, special cases that reduce to library
routines, brute force on tiny inputs).  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_moe.so")

F32, BF16, F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle_moe.so (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-Wall", "-o", tmp, _SRC, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        vp, ip = ctypes.c_void_p, ctypes.c_int
        _lib.oracle_route.argtypes = [ip, ip, ip, ip, ip, vp, vp, vp, vp, ip, vp, vp, vp, vp]
        _lib.oracle_gates_for_ids.argtypes = [ip, ip, ip, vp, vp, ip, vp]
        _lib.oracle_group.argtypes = [ip, ip, ip, ip, vp, vp, vp, vp, vp, vp, vp, vp]
        _lib.oracle_layer_tokens.argtypes = [ip] * 8 + [vp] * 11 + [ip, vp]
        _lib.oracle_load_stats.argtypes = [ip, ip, ip, vp, vp, ctypes.c_double, vp, vp, vp]
        _lib.oracle_bias_update.argtypes = [ip, ip, ip, vp, ctypes.c_double, vp, vp]
        _lib.oracle_load_stats_n.argtypes = [ip, ip, ctypes.c_longlong, vp, vp, ctypes.c_double, vp, vp, vp]
        _lib.oracle_ec_select.argtypes = [ip, ip, ip, vp, vp, vp]
        ll = ctypes.c_longlong
        _lib.oracle_e4m3_encode.argtypes = [ip, vp, vp]
        _lib.oracle_e4m3_decode.argtypes = [ip, vp, vp]
        _lib.oracle_quantize_fp8.argtypes = [ll, ip, ip, vp, vp, vp]
        _lib.oracle_dequant_fp8.argtypes = [ll, ip, vp, vp, vp]
        _lib.oracle_layer_backward.argtypes = [ip] * 8 + [vp] * 11 + [ip, ctypes.c_double, vp, ctypes.c_double] + [vp] * 15
        _lib.oracle_ec_slots.argtypes = [ip, ip, ip, vp, vp, vp, vp, vp, vp]
        for f in ("oracle_route", "oracle_gates_for_ids", "oracle_group", "oracle_layer_tokens",
                  "oracle_load_stats", "oracle_num_threads", "oracle_bias_update", "oracle_ec_select",
                  "oracle_ec_slots", "oracle_load_stats_n", "oracle_e4m3_encode", "oracle_e4m3_decode",
                  "oracle_quantize_fp8", "oracle_dequant_fp8", "oracle_layer_backward"):
            getattr(_lib, f).restype = ctypes.c_int
    return _lib


def num_threads() -> int:
    return int(_L().oracle_num_threads())


def _p(a):
    return None if a is None else a.ctypes.data


def _dtype_of(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle takes float32, uint16 (bf16 bits) or float64, got {a.dtype}")


def _c(a, dt=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a if dt is None else a.astype(dt, copy=False))
    return a


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def route(x, w_gate, k, logit_bias=None, select_bias=None, renormalize=True):
    """Router, softmax, top-k and gates for every token.

    x: [T, d]; w_gate: [E, d]; both float32 or both bf16 bits.
    Returns dict(ids int32 [T,k], gates f64 [T,k], probs f64 [T,E], margin f64 [T]).
    """
    x, w_gate = _c(x), _c(w_gate)
    dt = _dtype_of(x)
    if _dtype_of(w_gate) != dt:
        raise TypeError("x and w_gate must share a dtype")
    T, d = x.shape
    E = w_gate.shape[0]
    assert w_gate.shape[1] == d
    lb, sb = _c(logit_bias, np.float32), _c(select_bias, np.float32)
    ids = np.empty((T, k), np.int32)
    gates = np.empty((T, k), np.float64)
    probs = np.empty((T, E), np.float64)
    margin = np.empty((T,), np.float64)
    _check(_L().oracle_route(T, d, E, k, dt, _p(x), _p(w_gate), _p(lb), _p(sb), int(bool(renormalize)),
                             _p(ids), _p(gates), _p(probs), _p(margin)), "route")
    return dict(ids=ids, gates=gates, probs=probs, margin=margin)


def gates_for_ids(probs, ids, renormalize=True):
    """Gates g_j = p[t, ids_j] (renormalised over the k chosen) for given ids."""
    probs, ids = _c(probs, np.float64), _c(ids, np.int32)
    T, E = probs.shape
    k = ids.shape[1]
    gates = np.empty((T, k), np.float64)
    _check(_L().oracle_gates_for_ids(T, E, k, _p(probs), _p(ids), int(bool(renormalize)), _p(gates)),
           "gates_for_ids")
    return gates


def group(ids, E, capacity=-1):
    """Grouping by expert: counts, capacity cut, offsets, permutation.

    ids: int32 [T, k].  capacity < 0 means unlimited.
    """
    ids = _c(ids, np.int32)
    T, k = ids.shape
    n = T * k
    out = dict(counts=np.empty(E, np.int32), kept=np.empty(E, np.int32),
               offsets=np.empty(E + 1, np.int32), rank=np.empty((T, k), np.int32),
               slot_pos=np.empty((T, k), np.int32), sorted_token_ids=np.empty(n, np.int32))
    nd = np.zeros(1, np.int32)
    _check(_L().oracle_group(T, E, k, int(capacity), _p(ids), _p(out["counts"]), _p(out["kept"]),
                             _p(out["offsets"]), _p(out["rank"]), _p(out["slot_pos"]),
                             _p(out["sorted_token_ids"]), _p(nd)), "group")
    out["n_dropped"] = int(nd[0])
    return out


def layer_tokens(x, w1, w3, w2, ids, gates, slot_pos=None, tokens=None, shared=None):
    """Layer output rows y_t for the listed tokens (all tokens when None).

    w1, w3: [E, F, d]; w2: [E, d, F]; shared: None or (ws1 [F_s, d], ws3 [F_s, d], ws2 [d, F_s]).
    ids int32 [T, k], gates f64 [T, k], slot_pos int32 [T, k] or None.
    Returns f64 [len(tokens), d].
    """
    x = _c(x)
    dt = _dtype_of(x)
    w1, w3, w2 = _c(w1), _c(w3), _c(w2)
    for w in (w1, w3, w2):
        if _dtype_of(w) != dt:
            raise TypeError("weights and x must share a dtype")
    T, d = x.shape
    E, F, _ = w1.shape
    ids = _c(ids, np.int32)
    k = ids.shape[1]
    gates = _c(gates, np.float64)
    slot_pos = _c(slot_pos, np.int32)
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    tokens = _c(tokens, np.int32)
    if shared is None:
        ns, Fs, s1, s3, s2 = 0, 0, None, None, None
    else:
        s1, s3, s2 = (_c(a) for a in shared)
        ns, Fs = 1, s1.shape[0]
    y = np.empty((len(tokens), d), np.float64)
    _check(_L().oracle_layer_tokens(T, d, E, k, F, ns, Fs, dt, _p(x), _p(w1), _p(w3), _p(w2),
                                    _p(s1), _p(s3), _p(s2), _p(ids), _p(gates), _p(slot_pos),
                                    _p(tokens), len(tokens), _p(y)), "layer_tokens")
    return y


def load_stats(counts, probs, k, alpha):
    """f_i, p_i and L_balance = alpha * E * sum f_i p_i."""
    counts, probs = _c(counts, np.int32), _c(probs, np.float64)
    T, E = probs.shape
    f = np.empty(E, np.float64)
    p = np.empty(E, np.float64)
    L = np.zeros(1, np.float64)
    _check(_L().oracle_load_stats(T, E, k, _p(counts), _p(probs), float(alpha), _p(f), _p(p), _p(L)),
           "load_stats")
    return dict(f=f, p=p, L=float(L[0]))


def bias_update(counts, bias, T, k, gamma):
    """Selection-bias step b_e - gamma * sign(load_e - T k / E); returns float64 [E]."""
    counts = _c(counts, np.int32)
    bias = _c(bias, np.float32)
    E = counts.shape[0]
    out = np.empty(E, np.float64)
    _check(_L().oracle_bias_update(int(T), E, int(k), _p(counts), float(gamma), _p(bias), _p(out)), "bias_update")
    return out


def forward(layer, k, renormalize=True, capacity=-1, alpha=0.01, ids=None, tokens=None):
    """The whole layer, composed from the steps above in the pages' order.

    layer: dict with x, w_gate, w1, w3, w2 and optionally logit_bias, select_bias,
    ws1, ws3, ws2 (numpy arrays as described above).
    ids: optional int32 [T, k] routing decisions to use instead of the oracle's
    own (gates are then recomputed from the oracle's probabilities for those ids).
    tokens: optional token subset for y (routing, grouping and statistics always
    cover every token).
    """
    r = route(layer["x"], layer["w_gate"], k, layer.get("logit_bias"), layer.get("select_bias"),
              renormalize)
    if ids is None:
        ids, gates = r["ids"], r["gates"]
    else:
        ids = np.ascontiguousarray(ids, np.int32)
        gates = gates_for_ids(r["probs"], ids, renormalize)
    E = layer["w_gate"].shape[0]
    g = group(ids, E, capacity)
    shared = None
    if layer.get("ws1") is not None:
        shared = (layer["ws1"], layer["ws3"], layer["ws2"])
    y = layer_tokens(layer["x"], layer["w1"], layer["w3"], layer["w2"], ids, gates, g["slot_pos"],
                     tokens, shared)
    st = load_stats(g["counts"], r["probs"], k, alpha)
    return dict(y=y, ids=ids, gates=gates, probs=r["probs"], margin=r["margin"], **g, **st)


# ---------------------------------------------------------------- expert choice

def ec_bucket(T, E, k, capacity=-1):
    """Bucket size C of expert-choice routing: `capacity` when positive, else
    floor(T k / E) (k read as the average number of experts per token), at
    least 1 and at most T."""
    if T == 0:
        return 0
    C = int(capacity) if capacity > 0 else (T * k) // E
    return max(1, min(C, T))


def ec_select(probs, C):
    """Each expert's C highest-scoring tokens (ties to the lower token index),
    ascending.  probs f64 [T, E].  Returns (sel int32 [E, C], margin f64 [E])."""
    probs = _c(probs, np.float64)
    T, E = probs.shape
    sel = np.empty((E, C), np.int32)
    margin = np.empty(E, np.float64)
    _check(_L().oracle_ec_select(T, E, int(C), _p(probs), _p(sel), _p(margin)), "ec_select")
    return sel, margin


def ec_slots(sel, probs):
    """[T, E] slot form of an expert-choice assignment: ids, gates (p or 0),
    slot_pos (e*C + i or -1) and the number of tokens no expert chose."""
    sel, probs = _c(sel, np.int32), _c(probs, np.float64)
    T, E = probs.shape
    C = sel.shape[1]
    ids = np.empty((T, E), np.int32)
    gates = np.empty((T, E), np.float64)
    slot_pos = np.empty((T, E), np.int32)
    ne = np.zeros(1, np.int32)
    _check(_L().oracle_ec_slots(T, E, C, _p(sel), _p(probs), _p(ids), _p(gates), _p(slot_pos), _p(ne)), "ec_slots")
    return dict(ids=ids, gates=gates, slot_pos=slot_pos, n_empty=int(ne[0]))


def forward_expert_choice(layer, C, alpha=0.01, sel=None, tokens=None):
    """The layer under expert-choice routing, from the steps above.

    The router scores are the token-choice softmax probabilities (one route
    call with k = 1 supplies them); every expert keeps C tokens; each chosen
    (token, expert) pair adds p[t, e] * Expert_e(x_t); the shared expert is
    added unweighted.  sel: optional int32 [E, C] selection to use instead of
    the oracle's own (gates still come from the oracle's probabilities).
    Statistics: counts_e = C, f_e = C / (E C), p_e = mean score, L as usual.
    """
    r = route(layer["x"], layer["w_gate"], 1, layer.get("logit_bias"), None, True)
    probs = r["probs"]
    T, E = probs.shape
    own_sel, margin = ec_select(probs, C)
    use = own_sel if sel is None else np.ascontiguousarray(sel, np.int32)
    sl = ec_slots(use, probs)
    shared = None
    if layer.get("ws1") is not None:
        shared = (layer["ws1"], layer["ws3"], layer["ws2"])
    y = layer_tokens(layer["x"], layer["w1"], layer["w3"], layer["w2"], sl["ids"], sl["gates"], sl["slot_pos"],
                     tokens, shared)
    counts = np.full(E, C, np.int32)
    f = np.zeros(E, np.float64)
    pm = np.zeros(E, np.float64)
    Lb = np.zeros(1, np.float64)
    if T > 0:
        _check(_L().oracle_load_stats_n(T, E, E * C, _p(counts), _p(probs), float(alpha), _p(f), _p(pm), _p(Lb)),
               "load_stats_n")
    st = dict(f=f, p=pm, L=float(Lb[0]))
    return dict(y=y, probs=probs, sel=use, own_sel=own_sel, margin=margin, counts=counts, **sl, **st)


# ------------------------------------------------------------ FP8 weights

def widen(a):
    """Exact float64 copy of a float32 array or of bf16 bits held as uint16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def e4m3_encode(v):
    """float32 values -> E4M3 codes (round to nearest even, saturating)."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    _check(_L().oracle_e4m3_encode(v.size, _p(v), _p(out)), "e4m3_encode")
    return out


def e4m3_decode(c):
    """E4M3 codes -> float64 values (NaN for the two NaN codes)."""
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    _check(_L().oracle_e4m3_decode(c.size, _p(c), _p(out)), "e4m3_decode")
    return out


def quantize_fp8(w):
    """Per-row E4M3 quantisation of a [..., cols] weight array (float32 or bf16
    bits): returns (codes uint8 of the same shape, scales float32 [rows])."""
    w = _c(w)
    dt = _dtype_of(w)
    cols = w.shape[-1]
    rows = w.size // cols
    q = np.empty(w.shape, np.uint8)
    sc = np.empty(w.shape[:-1], np.float32)
    _check(_L().oracle_quantize_fp8(rows, cols, dt, _p(w), _p(q), _p(sc)), "quantize_fp8")
    return q, sc


def dequant_fp8(q, scale):
    """value(q) * scale per row, exactly, as float64."""
    q, scale = _c(q, np.uint8), _c(scale, np.float32)
    cols = q.shape[-1]
    rows = q.size // cols
    out = np.empty(q.shape, np.float64)
    _check(_L().oracle_dequant_fp8(rows, cols, _p(q), _p(scale), _p(out)), "dequant_fp8")
    return out


# ---------------------------------------------------------------- backward

def backward(layer, k, ids, slot_pos, dy, renormalize=True, alpha=0.01, dL=0.0, magnitudes=False):
    """Gradients of <dy, y> + dL * L_balance with respect to x, W_g, W1, W3, W2
    (and the shared expert's weights), the routing decisions (ids, dropped
    slots) held fixed and f held constant.  layer: dict as for forward();
    ids int32 [T, k]; slot_pos int32 [T, k] or None (< 0 = dropped); dy [T, d]
    (converted to float64).  Returns a dict of float64 arrays: dx, dw_gate,
    dw1, dw3, dw2, dlogits (and dws1, dws3, dws2 with a shared expert).
    magnitudes=True adds, for every weight gradient "dwX", "sum_abs_dwX": the
    sum over the same terms of the products of absolute values (|da| |x|,
    |db| |x|, |g dy| |h|), the per-entry scale for comparing gradients
    computed from rounded operands."""
    x = _c(layer["x"])
    dt = _dtype_of(x)
    wg, w1, w3, w2 = (_c(layer[n]) for n in ("w_gate", "w1", "w3", "w2"))
    T, d = x.shape
    E, F, _ = w1.shape
    ids = _c(ids, np.int32)
    assert ids.shape == (T, k)
    sp = _c(slot_pos, np.int32)
    dy = _c(dy, np.float64)
    lb = _c(layer.get("logit_bias"), np.float32)
    shared = layer.get("ws1") is not None
    s1, s3, s2 = (_c(layer[n]) for n in ("ws1", "ws3", "ws2")) if shared else (None, None, None)
    Fs = s1.shape[0] if shared else 0
    out = dict(dx=np.empty((T, d)), dw_gate=np.empty((E, d)), dw1=np.empty((E, F, d)), dw3=np.empty((E, F, d)),
               dw2=np.empty((E, d, F)), dlogits=np.empty((T, E)))
    if shared:
        out.update(dws1=np.empty((Fs, d)), dws3=np.empty((Fs, d)), dws2=np.empty((d, Fs)))
    if magnitudes:
        for n in [n for n in out if n.startswith("dw") and n != "dw_gate"]:
            out["sum_abs_" + n] = np.empty_like(out[n])
    _check(_L().oracle_layer_backward(T, d, E, k, F, int(shared), Fs, dt, _p(x), _p(wg), _p(lb), _p(w1), _p(w3),
                                      _p(w2), _p(s1), _p(s3), _p(s2), _p(ids), _p(sp), int(bool(renormalize)),
                                      float(alpha), _p(dy), float(dL), _p(out["dx"]), _p(out["dw_gate"]),
                                      _p(out["dw1"]), _p(out["dw3"]), _p(out["dw2"]), _p(out.get("dws1")),
                                      _p(out.get("dws3")), _p(out.get("dws2")), _p(out["dlogits"]),
                                      *(_p(out.get("sum_abs_" + n)) for n in ("dw1", "dw3", "dw2", "dws1", "dws3", "dws2"))),
           "layer_backward")
    return out

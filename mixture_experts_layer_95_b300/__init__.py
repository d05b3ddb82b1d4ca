"""Python binding of libmoe_b300.so -- the MoE SwiGLU layer forward on a B300.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory (tensors) and streams; the functions
below check shapes/dtypes, allocate outputs with ``torch.empty`` and pass raw
pointers through ctypes to the C entry points of ``include/moe_b300.h`` of the
same names.  There is no CPU path: if the shared library is missing, importing
succeeds but every call raises ``MoeError``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_ROUTE_TOKEN_CHOICE, MOE_ROUTE_EXPERT_CHOICE = 0, 1
STATUS = {0: "MOE_OK", -1: "MOE_ERR_NULL", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_DTYPE", -4: "MOE_ERR_WORKSPACE",
          -5: "MOE_ERR_CUDA", -6: "MOE_ERR_DEVICE", -7: "MOE_ERR_TIMEOUT", -8: "MOE_ERR_DEVICE_BOUNDS",
          -9: "MOE_ERR_ALIGN"}

EXPORTED = ("moe_workspace_size", "moe_workspace_init", "moe_route", "moe_permute", "moe_expert_ffn",
            "moe_combine", "moe_load_stats", "moe_forward", "moe_last_device_status", "moe_strerror",
            "moe_version", "moe_set_stage_events", "moe_launch_count", "moe_permute_static", "moe_bias_update",
            "moe_plan_describe", "moe_route_expert_choice", "moe_quantize_fp8", "moe_forward_fp8",
            "moe_backward_workspace_size", "moe_backward", "moe_forward_train", "moe_backward_saved",
            "moe_test_stall_gemm")
STAGES = ("router", "group_scan", "gather", "up_gemm", "down_gemm", "combine")


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)} ({strerror(code) if _lib else ''})")


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("d_ff_shared", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("renormalize", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("y_fp32", ctypes.c_int32), ("h_split", ctypes.c_int32),
                ("routing", ctypes.c_int32), ("yperm_bf16", ctypes.c_int32)]


class MoeFp8Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w1", "w3", "w2", "s1", "s3", "s2", "ws1", "ws3", "ws2", "ss1", "ss3",
                                               "ss2")]


class MoeStats(ctypes.Structure):
    _fields_ = [("counts", ctypes.c_void_p), ("kept", ctypes.c_void_p), ("f", ctypes.c_void_p),
                ("p", ctypes.c_void_p), ("L", ctypes.c_void_p), ("n_dropped", ctypes.c_void_p)]


_lib = None


def lib():
    """The loaded shared library; raises MoeError if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoeError(-5, f"{LIB_PATH} is missing; build it with `python -m mixture_experts_layer_95_b300._build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        cfgp = ctypes.POINTER(MoeConfig)
        L.moe_workspace_size.argtypes = [cfgp]
        L.moe_workspace_size.restype = sz
        L.moe_workspace_init.argtypes = [cfgp, vp, sz, vp]
        L.moe_route.argtypes = [cfgp] + [vp] * 7 + [vp, sz, vp]
        L.moe_permute.argtypes = [cfgp] + [vp] * 11 + [vp, sz, vp]
        L.moe_permute_static.argtypes = [cfgp] + [vp] * 11 + [vp]
        L.moe_permute_static.restype = i32
        L.moe_bias_update.argtypes = [cfgp, vp, ctypes.c_float, vp, vp]
        L.moe_bias_update.restype = i32
        L.moe_expert_ffn.argtypes = [cfgp] + [vp] * 12 + [vp, sz, vp]
        L.moe_combine.argtypes = [cfgp] + [vp] * 4 + [vp]
        L.moe_load_stats.argtypes = [cfgp] + [vp] * 4 + [vp]
        L.moe_forward.argtypes = [cfgp] + [vp] * 10 + [vp, ctypes.POINTER(MoeStats), vp, sz, vp]
        L.moe_last_device_status.argtypes = [cfgp, vp, vp]
        L.moe_strerror.argtypes = [i32]
        L.moe_strerror.restype = ctypes.c_char_p
        L.moe_version.restype = ctypes.c_char_p
        L.moe_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
        L.moe_set_stage_events.restype = i32
        L.moe_launch_count.restype = ctypes.c_uint64
        L.moe_test_stall_gemm.argtypes = [i32]
        L.moe_test_stall_gemm.restype = i32
        L.moe_route_expert_choice.argtypes = [cfgp] + [vp] * 10 + [vp, sz, vp]
        L.moe_quantize_fp8.argtypes = [vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, vp, vp, vp]
        L.moe_quantize_fp8.restype = i32
        L.moe_forward_fp8.argtypes = [cfgp, vp, vp, vp, vp, ctypes.POINTER(MoeFp8Weights), vp,
                                      ctypes.POINTER(MoeStats), vp, sz, vp]
        L.moe_forward_fp8.restype = i32
        L.moe_backward_workspace_size.argtypes = [cfgp]
        L.moe_backward_workspace_size.restype = sz
        L.moe_backward.argtypes = [cfgp] + [vp] * 11 + [ctypes.c_float] + [vp] * 8 + [vp, sz, vp]
        L.moe_backward.restype = i32
        L.moe_backward_saved.argtypes = L.moe_backward.argtypes
        L.moe_backward_saved.restype = i32
        L.moe_forward_train.argtypes = L.moe_forward.argtypes
        L.moe_forward_train.restype = i32
        L.moe_route_expert_choice.restype = i32
        L.moe_plan_describe.argtypes = [cfgp, ctypes.c_char_p, sz]
        L.moe_plan_describe.restype = i32
        for f in ("moe_workspace_init", "moe_route", "moe_permute", "moe_expert_ffn", "moe_combine",
                  "moe_load_stats", "moe_forward", "moe_last_device_status"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().moe_strerror(int(code)).decode()


def version() -> str:
    return lib().moe_version().decode()


def plan_describe(cfg: MoeConfig) -> dict:
    """The kernels moe_forward picks for `cfg`, as a dict of the library's
    "key=value" words (router, up, down, ksplit_up, ksplit_down, gather_a, h)."""
    buf = ctypes.create_string_buffer(256)
    _check(lib().moe_plan_describe(ctypes.byref(cfg), buf, 256), "moe_plan_describe")
    return dict(w.split("=", 1) for w in buf.value.decode().split())


def launch_count() -> int:
    """Kernels launched by the library in this process so far."""
    return int(lib().moe_launch_count())


def test_stall_gemm(on: bool) -> bool:
    """moe_test_stall_gemm: the failure-detection test switch (tensor-core GEMMs
    launched while it is on issue no loads and time out after 20 ms).
    Returns the previous setting."""
    return bool(lib().moe_test_stall_gemm(1 if on else 0))


# True while a StageTimer has stage events set for the next library calls
# (Forward then enqueues eagerly, so that the events record this call).
_STAGE_EVENTS_SET = [False]


class StageTimer:
    """Per-stage CUDA-event timing of the library's launches (diagnostics).

    Inside ``with StageTimer() as st:``, call ``st.begin_call()`` before each
    library call; the call then records a start/stop event pair around each
    stage's launches (``moe_set_stage_events``) on its own stream.  ``st.ms()``
    returns the summed milliseconds per stage and how many calls recorded it.
    The events are plain cudart events owned by this object.
    """

    def __init__(self, n_calls: int = 0, stages=STAGES):
        from cuda.bindings import runtime as cudart
        self._rt = cudart
        self._events = []
        self._used = 0
        self._want = set(stages)  # stages not listed get no events (their launches stay back to back)
        for _ in range(n_calls):  # create up front so timed loops pay no creation cost
            self._events.append(self._new_set())

    def _new_set(self):
        rt = self._rt
        ev = []
        for _ in range(2 * len(STAGES)):
            err, e = rt.cudaEventCreate()
            if err != rt.cudaError_t.cudaSuccess:
                raise MoeError(-5, f"cudaEventCreate: {err}")
            ev.append(e)
        return ev

    def begin_call(self):
        _STAGE_EVENTS_SET[0] = True
        if self._used == len(self._events):
            self._events.append(self._new_set())
        ev = self._events[self._used]
        self._used += 1
        handles = [int(e) if STAGES[i // 2] in self._want else None for i, e in enumerate(ev)]
        self._arr = (ctypes.c_void_p * len(ev))(*handles)  # kept alive while set
        _check(lib().moe_set_stage_events(self._arr, len(ev)), "moe_set_stage_events")

    def skip_call(self):
        """The next library call records no events (its launches keep their
        programmatic overlap)."""
        _check(lib().moe_set_stage_events(None, 0), "moe_set_stage_events")
        _STAGE_EVENTS_SET[0] = False

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        lib().moe_set_stage_events(None, 0)
        _STAGE_EVENTS_SET[0] = False
        return False

    def ms(self):
        """(summed ms per stage, number of calls that recorded the stage)."""
        rt = self._rt
        torch.cuda.synchronize()
        out = {s: 0.0 for s in STAGES}
        counts = {s: 0 for s in STAGES}
        for ev in self._events[:self._used]:
            for i, s in enumerate(STAGES):
                if s not in self._want:
                    continue
                err, ms = rt.cudaEventElapsedTime(ev[2 * i], ev[2 * i + 1])
                if err == rt.cudaError_t.cudaSuccess:  # stages a call did not run stay unrecorded
                    out[s] += ms
                    counts[s] += 1
        return out, counts

    def close(self):
        for ev in self._events:
            for e in ev:
                self._rt.cudaEventDestroy(e)
        self._events = []


def _check(rc: int, what: str):
    if rc != 0:
        raise MoeError(rc, what)


@dataclass
class Layer:
    """Static description of a layer (sizes and routing options)."""
    T: int
    d: int
    E: int
    k: int
    d_ff: int
    n_shared: int = 0
    d_ff_shared: int = 0
    dtype: str = "bf16"
    renormalize: bool = True
    capacity: int = -1
    alpha: float = 0.01
    y_fp32: bool = False  # return y in fp32 (before rounding to the layer dtype)
    h_split: bool = False  # bf16: keep H as a hi + lo bf16 pair (heavy-tailed layers)
    routing: str = "token"  # "token": tokens choose top-k experts; "expert": experts choose C tokens
    yperm_bf16: bool = False  # bf16: keep the expert rows (y_perm, y_shared) in bf16 for the combine

    def cfg(self) -> MoeConfig:
        if self.routing not in ("token", "expert"):
            raise ValueError(f"routing must be 'token' or 'expert', got {self.routing!r}")
        return MoeConfig(self.T, self.d, self.E, self.k, self.d_ff, self.n_shared, self.d_ff_shared,
                         MOE_BF16 if self.dtype == "bf16" else MOE_F32, int(bool(self.renormalize)),
                         int(self.capacity), float(self.alpha), int(bool(self.y_fp32)), int(bool(self.h_split)),
                         MOE_ROUTE_EXPERT_CHOICE if self.routing == "expert" else MOE_ROUTE_TOKEN_CHOICE,
                         int(bool(self.yperm_bf16)))

    @property
    def yperm_dtype(self):
        """Storage of the expert rows y_perm / y_shared of the step API."""
        return torch.bfloat16 if self.yperm_bf16 else torch.float32

    @property
    def bucket(self) -> int:
        """Expert choice: tokens per expert, C (the header's rule); 0 for token choice."""
        if self.routing != "expert" or self.T == 0:
            return 0
        C = self.capacity if self.capacity > 0 else (self.T * self.k) // self.E
        return max(1, min(C, self.T))

    @property
    def perm_rows(self) -> int:
        """Rows of the permuted layout: T*k, or E*C under expert choice."""
        return self.E * self.bucket if self.routing == "expert" else self.T * self.k

    @property
    def slots(self) -> int:
        """Slots per token in slot_pos: k, or E under expert choice."""
        return self.E if self.routing == "expert" else self.k

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def y_dtype(self):
        return torch.float32 if self.y_fp32 else self.torch_dtype


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, shape, dtype, name):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name}: expected {tuple(shape)} {dtype}, got {tuple(t.shape)} {t.dtype}")
    return t


def workspace_size(layer: Layer) -> int:
    c = layer.cfg()
    n = lib().moe_workspace_size(ctypes.byref(c))
    if n == 0:
        raise MoeError(-2, "moe_workspace_size")
    return int(n)


def workspace(layer: Layer, device=None, stream=None) -> torch.Tensor:
    """Allocates (with torch) and initialises a workspace for `layer`."""
    ws = torch.empty(workspace_size(layer), dtype=torch.uint8, device=device or "cuda")
    c = layer.cfg()
    _check(lib().moe_workspace_init(ctypes.byref(c), _ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")
    return ws


def last_device_status(layer: Layer, ws: torch.Tensor, stream=None) -> int:
    c = layer.cfg()
    return int(lib().moe_last_device_status(ctypes.byref(c), _ptr(ws), _stream(stream)))


def route(layer: Layer, x, w_gate, logit_bias=None, select_bias=None, ws=None, stream=None):
    """moe_route: returns (topk_ids int32 [T,k], gates fp32 [T,k], p_mean fp32 [E])."""
    dt, dev = layer.torch_dtype, x.device
    _need(x, (layer.T, layer.d), dt, "x")
    _need(w_gate, (layer.E, layer.d), dt, "w_gate")
    if logit_bias is not None:
        _need(logit_bias, (layer.E,), torch.float32, "logit_bias")
    if select_bias is not None:
        _need(select_bias, (layer.E,), torch.float32, "select_bias")
    ws = ws if ws is not None else workspace(layer, dev, stream)
    ids = torch.empty((layer.T, layer.k), dtype=torch.int32, device=dev)
    gates = torch.empty((layer.T, layer.k), dtype=torch.float32, device=dev)
    p_mean = torch.empty((layer.E,), dtype=torch.float32, device=dev)
    c = layer.cfg()
    _check(lib().moe_route(ctypes.byref(c), _ptr(x), _ptr(w_gate), _ptr(logit_bias), _ptr(select_bias), _ptr(ids),
                           _ptr(gates), _ptr(p_mean), _ptr(ws), ws.numel(), _stream(stream)), "moe_route")
    return ids, gates, p_mean


def route_expert_choice(layer: Layer, x, w_gate, logit_bias=None, ws=None, stream=None, gather=True):
    """moe_route_expert_choice: every expert takes its C tokens.  Returns a dict
    with probs [T,E], sorted_token_ids / gates_perm [E*C], slot_pos [T,E],
    offsets [E+1], p_mean [E] and (gather=True) x_perm [E*C, d]."""
    dt, dev = layer.torch_dtype, x.device
    _need(x, (layer.T, layer.d), dt, "x")
    _need(w_gate, (layer.E, layer.d), dt, "w_gate")
    if logit_bias is not None:
        _need(logit_bias, (layer.E,), torch.float32, "logit_bias")
    ws = ws if ws is not None else workspace(layer, dev, stream)
    n = layer.perm_rows
    i32 = dict(dtype=torch.int32, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    out = dict(probs=torch.empty((layer.T, layer.E), **f32), sorted_token_ids=torch.empty(n, **i32),
               gates_perm=torch.empty(n, **f32), slot_pos=torch.empty((layer.T, layer.E), **i32),
               offsets=torch.empty(layer.E + 1, **i32), p_mean=torch.empty(layer.E, **f32),
               x_perm=torch.empty((n, layer.d), dtype=dt, device=dev) if gather else None)
    c = layer.cfg()
    _check(lib().moe_route_expert_choice(ctypes.byref(c), _ptr(x), _ptr(w_gate), _ptr(logit_bias),
                                         _ptr(out["probs"]), _ptr(out["sorted_token_ids"]), _ptr(out["gates_perm"]),
                                         _ptr(out["slot_pos"]), _ptr(out["offsets"]), _ptr(out["p_mean"]),
                                         _ptr(out["x_perm"]), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_route_expert_choice")
    return out


def permute(layer: Layer, topk_ids, gates, x, ws=None, stream=None):
    """moe_permute: returns a dict of the grouping outputs and x_perm."""
    dev = x.device
    n = layer.T * layer.k
    _need(topk_ids, (layer.T, layer.k), torch.int32, "topk_ids")
    _need(gates, (layer.T, layer.k), torch.float32, "gates")
    _need(x, (layer.T, layer.d), layer.torch_dtype, "x")
    ws = ws if ws is not None else workspace(layer, dev, stream)
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(counts=torch.empty(layer.E, **i32), kept=torch.empty(layer.E, **i32),
               offsets=torch.empty(layer.E + 1, **i32), sorted_token_ids=torch.empty(n, **i32),
               slot_pos=torch.empty((layer.T, layer.k), **i32),
               gates_perm=torch.empty(n, dtype=torch.float32, device=dev),
               x_perm=torch.empty((n, layer.d), dtype=layer.torch_dtype, device=dev),
               n_dropped=torch.empty(1, **i32))
    c = layer.cfg()
    _check(lib().moe_permute(ctypes.byref(c), _ptr(topk_ids), _ptr(gates), _ptr(x), _ptr(out["counts"]),
                             _ptr(out["kept"]), _ptr(out["offsets"]), _ptr(out["sorted_token_ids"]),
                             _ptr(out["slot_pos"]), _ptr(out["gates_perm"]), _ptr(out["x_perm"]),
                             _ptr(out["n_dropped"]), _ptr(ws), ws.numel(), _stream(stream)), "moe_permute")
    return out


def permute_static(layer: Layer, topk_ids, gates, x, stream=None):
    """moe_permute_static: moe_permute without a workspace (fixed library scratch).

    For callers that cannot allocate device memory; see include/moe_b300.h for
    the size limit and the rule that concurrent calls on one device race.
    """
    dev = x.device
    n = layer.T * layer.k
    _need(topk_ids, (layer.T, layer.k), torch.int32, "topk_ids")
    _need(gates, (layer.T, layer.k), torch.float32, "gates")
    _need(x, (layer.T, layer.d), layer.torch_dtype, "x")
    i32 = dict(dtype=torch.int32, device=dev)
    out = dict(counts=torch.empty(layer.E, **i32), kept=torch.empty(layer.E, **i32),
               offsets=torch.empty(layer.E + 1, **i32), sorted_token_ids=torch.empty(n, **i32),
               slot_pos=torch.empty((layer.T, layer.k), **i32),
               gates_perm=torch.empty(n, dtype=torch.float32, device=dev),
               x_perm=torch.empty((n, layer.d), dtype=layer.torch_dtype, device=dev),
               n_dropped=torch.empty(1, **i32))
    c = layer.cfg()
    _check(lib().moe_permute_static(ctypes.byref(c), _ptr(topk_ids), _ptr(gates), _ptr(x), _ptr(out["counts"]),
                                    _ptr(out["kept"]), _ptr(out["offsets"]), _ptr(out["sorted_token_ids"]),
                                    _ptr(out["slot_pos"]), _ptr(out["gates_perm"]), _ptr(out["x_perm"]),
                                    _ptr(out["n_dropped"]), _stream(stream)), "moe_permute_static")
    return out


def expert_ffn(layer: Layer, x_perm, offsets, gates_perm, w1, w3, w2, x=None, ws1=None, ws3=None, ws2=None,
               ws=None, stream=None):
    """moe_expert_ffn: returns (y_perm [rows, d], y_shared [T, d] or None), fp32 or,
    with layer.yperm_bf16, bf16; rows = T*k (token choice) or E*C (expert choice)."""
    dt, dev = layer.torch_dtype, x_perm.device
    n = layer.perm_rows
    _need(x_perm, (n, layer.d), dt, "x_perm")
    _need(offsets, (layer.E + 1,), torch.int32, "offsets")
    _need(gates_perm, (n,), torch.float32, "gates_perm")
    _need(w1, (layer.E, layer.d_ff, layer.d), dt, "w1")
    _need(w3, (layer.E, layer.d_ff, layer.d), dt, "w3")
    _need(w2, (layer.E, layer.d, layer.d_ff), dt, "w2")
    y_shared = None
    if layer.n_shared:
        _need(x, (layer.T, layer.d), dt, "x")
        _need(ws1, (layer.d_ff_shared, layer.d), dt, "ws1")
        _need(ws3, (layer.d_ff_shared, layer.d), dt, "ws3")
        _need(ws2, (layer.d, layer.d_ff_shared), dt, "ws2")
        y_shared = torch.empty((layer.T, layer.d), dtype=layer.yperm_dtype, device=dev)
    ws = ws if ws is not None else workspace(layer, dev, stream)
    y_perm = torch.empty((n, layer.d), dtype=layer.yperm_dtype, device=dev)
    c = layer.cfg()
    _check(lib().moe_expert_ffn(ctypes.byref(c), _ptr(x_perm), _ptr(offsets), _ptr(gates_perm), _ptr(w1), _ptr(w3),
                                _ptr(w2), _ptr(x), _ptr(ws1), _ptr(ws3), _ptr(ws2), _ptr(y_perm), _ptr(y_shared),
                                _ptr(ws), ws.numel(), _stream(stream)), "moe_expert_ffn")
    return y_perm, y_shared


def combine(layer: Layer, y_perm, slot_pos, y_shared=None, stream=None):
    """moe_combine: returns y [T, d] in the layer dtype."""
    dev = y_perm.device
    _need(y_perm, (layer.perm_rows, layer.d), layer.yperm_dtype, "y_perm")
    _need(slot_pos, (layer.T, layer.slots), torch.int32, "slot_pos")
    if y_shared is not None:
        _need(y_shared, (layer.T, layer.d), layer.yperm_dtype, "y_shared")
    y = torch.empty((layer.T, layer.d), dtype=layer.y_dtype, device=dev)
    c = layer.cfg()
    _check(lib().moe_combine(ctypes.byref(c), _ptr(y_perm), _ptr(slot_pos), _ptr(y_shared), _ptr(y),
                             _stream(stream)), "moe_combine")
    return y


def load_stats(layer: Layer, counts, p_mean, stream=None):
    """moe_load_stats: returns (f fp32 [E], L fp32 [1])."""
    dev = counts.device
    _need(counts, (layer.E,), torch.int32, "counts")
    _need(p_mean, (layer.E,), torch.float32, "p_mean")
    f = torch.empty(layer.E, dtype=torch.float32, device=dev)
    L = torch.empty(1, dtype=torch.float32, device=dev)
    c = layer.cfg()
    _check(lib().moe_load_stats(ctypes.byref(c), _ptr(counts), _ptr(p_mean), _ptr(f), _ptr(L), _stream(stream)),
           "moe_load_stats")
    return f, L


def bias_update(layer: Layer, counts, select_bias, gamma: float, stream=None):
    """moe_bias_update: select_bias[e] -= gamma * sign(counts[e] - T k / E), in place."""
    _need(counts, (layer.E,), torch.int32, "counts")
    _need(select_bias, (layer.E,), torch.float32, "select_bias")
    c = layer.cfg()
    _check(lib().moe_bias_update(ctypes.byref(c), _ptr(counts), ctypes.c_float(gamma), _ptr(select_bias),
                                 _stream(stream)), "moe_bias_update")
    return select_bias


def quantize_fp8(w, stream=None):
    """moe_quantize_fp8 over the last axis of w (bf16 or fp32, last dim a
    multiple of 16): returns (codes uint8 of w's shape, scales fp32 w.shape[:-1])."""
    if not w.is_cuda or not w.is_contiguous() or w.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("w must be a contiguous bf16 or fp32 CUDA tensor")
    cols = w.shape[-1]
    rows = w.numel() // cols
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    sc = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    _check(lib().moe_quantize_fp8(_ptr(w), MOE_BF16 if w.dtype == torch.bfloat16 else MOE_F32, rows, cols, _ptr(q),
                                  _ptr(sc), _stream(stream)), "moe_quantize_fp8")
    return q, sc


def quantize_experts_fp8(layer: "Layer", w1, w3, w2, ws1=None, ws3=None, ws2=None, stream=None) -> dict:
    """FP8 weight set for moe_forward_fp8: codes and per-row scales of W1, W3,
    W2 (and of the shared expert when the layer has one)."""
    out = {}
    for n, t in (("w1", w1), ("w3", w3), ("w2", w2), ("ws1", ws1), ("ws3", ws3), ("ws2", ws2)):
        if t is None:
            continue
        q, sc = quantize_fp8(t, stream)
        out[n] = q
        out["s" + n[1:]] = sc  # w1 -> s1, ws1 -> ss1
    return out


def backward(layer: Layer, x, w_gate, w1, w3, w2, dy, logit_bias=None, select_bias=None, ws1=None, ws3=None,
             ws2=None, dL: float = 0.0, stream=None) -> dict:
    """moe_backward: gradients (fp32) of <dy, y> + dL * L_balance for every
    input of the layer, routing held fixed.  Returns a dict with dx, dw_gate,
    dw1, dw3, dw2 (and dws1, dws3, dws2 with a shared expert)."""
    dt, dev = layer.torch_dtype, x.device
    E, F, d, T, Fs = layer.E, layer.d_ff, layer.d, layer.T, layer.d_ff_shared
    _need(x, (T, d), dt, "x")
    _need(dy, (T, d), dt, "dy")
    _need(w_gate, (E, d), dt, "w_gate")
    _need(w1, (E, F, d), dt, "w1")
    _need(w3, (E, F, d), dt, "w3")
    _need(w2, (E, d, F), dt, "w2")
    f32 = dict(dtype=torch.float32, device=dev)
    out = dict(dx=torch.empty((T, d), **f32), dw_gate=torch.empty((E, d), **f32),
               dw1=torch.empty((E, F, d), **f32), dw3=torch.empty((E, F, d), **f32),
               dw2=torch.empty((E, d, F), **f32))
    if layer.n_shared:
        _need(ws1, (Fs, d), dt, "ws1")
        _need(ws3, (Fs, d), dt, "ws3")
        _need(ws2, (d, Fs), dt, "ws2")
        out.update(dws1=torch.empty((Fs, d), **f32), dws3=torch.empty((Fs, d), **f32),
                   dws2=torch.empty((d, Fs), **f32))
    c = layer.cfg()
    nbytes = lib().moe_backward_workspace_size(ctypes.byref(c))
    if nbytes == 0:
        raise MoeError(-2, "moe_backward_workspace_size")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _check(lib().moe_workspace_init(ctypes.byref(c), _ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")
    _check(lib().moe_backward(ctypes.byref(c), _ptr(x), _ptr(w_gate), _ptr(logit_bias), _ptr(select_bias), _ptr(w1),
                              _ptr(w3), _ptr(w2), _ptr(ws1), _ptr(ws3), _ptr(ws2), _ptr(dy), ctypes.c_float(dL),
                              _ptr(out["dx"]), _ptr(out["dw_gate"]), _ptr(out["dw1"]), _ptr(out["dw3"]),
                              _ptr(out["dw2"]), _ptr(out.get("dws1")), _ptr(out.get("dws3")), _ptr(out.get("dws2")),
                              _ptr(ws), ws.numel(), _stream(stream)), "moe_backward")
    rc = last_device_status(layer, ws, stream)
    if rc != 0:
        raise MoeError(rc, "moe_backward (device status)")
    return out


class Backward:
    """Reusable moe_backward call (preallocated workspace and gradient
    buffers): the form the benchmark times."""

    def __init__(self, layer: Layer, w_gate, w1, w3, w2, logit_bias=None, select_bias=None, ws1=None, ws3=None,
                 ws2=None, device=None):
        dev = device or w1.device
        self.layer, self.cfg = layer, layer.cfg()
        E, F, d, T, Fs = layer.E, layer.d_ff, layer.d, layer.T, layer.d_ff_shared
        nbytes = lib().moe_backward_workspace_size(ctypes.byref(self.cfg))
        if nbytes == 0:
            raise MoeError(-2, "moe_backward_workspace_size")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        _check(lib().moe_workspace_init(ctypes.byref(self.cfg), _ptr(self.ws), self.ws.numel(), _stream(None)),
               "moe_workspace_init")
        f32 = dict(dtype=torch.float32, device=dev)
        self.grads = dict(dx=torch.empty((T, d), **f32), dw_gate=torch.empty((E, d), **f32),
                          dw1=torch.empty((E, F, d), **f32), dw3=torch.empty((E, F, d), **f32),
                          dw2=torch.empty((E, d, F), **f32))
        if layer.n_shared:
            self.grads.update(dws1=torch.empty((Fs, d), **f32), dws3=torch.empty((Fs, d), **f32),
                              dws2=torch.empty((d, Fs), **f32))
        self.w = (w_gate, logit_bias, select_bias, w1, w3, w2, ws1, ws3, ws2)

    def forward_train(self, x, y=None, stream=None, stats: bool = False):
        """moe_forward_train: y of the layer, with the activations the next
        __call__(..., saved=True) reads kept in this object's workspace.
        stats=True returns (y, stats) with the same statistics as Forward."""
        L = self.layer
        _need(x, (L.T, L.d), L.torch_dtype, "x")
        if y is None:
            y = torch.empty((L.T, L.d), dtype=L.y_dtype, device=x.device)
        else:
            _need(y, (L.T, L.d), L.y_dtype, "y")
        st, st_struct = None, None
        if stats:
            i32 = dict(dtype=torch.int32, device=x.device)
            f32 = dict(dtype=torch.float32, device=x.device)
            E = L.E
            st = dict(counts=torch.zeros(E, **i32), kept=torch.zeros(E, **i32), f=torch.zeros(E, **f32),
                      p=torch.zeros(E, **f32), L=torch.zeros(1, **f32), n_dropped=torch.zeros(1, **i32))
            st_struct = MoeStats(st["counts"].data_ptr(), st["kept"].data_ptr(), st["f"].data_ptr(),
                                 st["p"].data_ptr(), st["L"].data_ptr(), st["n_dropped"].data_ptr())
        wg, lb, sb, w1, w3, w2, s1, s3, s2 = (_ptr(t) for t in self.w)
        _check(lib().moe_forward_train(ctypes.byref(self.cfg), _ptr(x), wg, lb, sb, w1, w3, w2, s1, s3, s2, _ptr(y),
                                       ctypes.byref(st_struct) if st_struct is not None else None, _ptr(self.ws),
                                       self.ws.numel(), _stream(stream)), "moe_forward_train")
        return (y, st) if stats else y

    def __call__(self, x, dy, dL: float = 0.0, stream=None, saved: bool = False):
        """saved=True: moe_backward_saved on the activations of the last
        forward_train(x) (same x); otherwise moe_backward recomputes them."""
        wg, lb, sb, w1, w3, w2, s1, s3, s2 = (_ptr(t) for t in self.w)
        g = self.grads
        fn, name = (lib().moe_backward_saved, "moe_backward_saved") if saved else (lib().moe_backward, "moe_backward")
        _check(fn(ctypes.byref(self.cfg), _ptr(x), wg, lb, sb, w1, w3, w2, s1, s3, s2, _ptr(dy), ctypes.c_float(dL),
                  _ptr(g["dx"]), _ptr(g["dw_gate"]), _ptr(g["dw1"]), _ptr(g["dw3"]), _ptr(g["dw2"]),
                  _ptr(g.get("dws1")), _ptr(g.get("dws3")), _ptr(g.get("dws2")), _ptr(self.ws), self.ws.numel(),
                  _stream(stream)), name)
        return g

    def device_status(self, stream=None) -> int:
        return last_device_status(self.layer, self.ws, stream)


class Forward:
    """Reusable moe_forward call: checks the weights once, owns the workspace,
    and enqueues the whole layer per call (the form the benchmark times).

    graph=True replays the layer from a CUDA graph: the first call on a given
    pair of x / y buffers runs eagerly and records the library's launches
    (every pointer, the workspace and the statistics buffers included) into a
    graph; later calls on the same buffers only replay it, which costs the
    host one graph launch instead of the library's argument checks, tensor
    map set-up and one launch per kernel.  The layer's configuration and
    weights are fixed per Forward, so a replay computes exactly what an eager
    call would."""

    def __init__(self, layer: Layer, w_gate, w1, w3, w2, logit_bias=None, select_bias=None, ws1=None, ws3=None,
                 ws2=None, stats: bool = False, device=None, stream=None, fp8: dict | None = None,
                 graph: bool = False):
        """fp8: an FP8 weight set from quantize_experts_fp8 (then w1/w3/w2 and
        ws1/ws3/ws2 are ignored and may be None; the call is moe_forward_fp8)."""
        self.graph = graph
        self._graphs = {}
        dt = layer.torch_dtype
        self.layer = layer
        self.cfg = layer.cfg()
        E, F, d, Fs = layer.E, layer.d_ff, layer.d, layer.d_ff_shared
        self.fp8 = None
        if fp8 is not None:
            u8, f32 = torch.uint8, torch.float32
            for n, shape, t in (("w1", (E, F, d), u8), ("w3", (E, F, d), u8), ("w2", (E, d, F), u8),
                                ("s1", (E, F), f32), ("s3", (E, F), f32), ("s2", (E, d), f32)):
                _need(fp8.get(n), shape, t, "fp8 " + n)
            if layer.n_shared:
                for n, shape, t in (("ws1", (Fs, d), u8), ("ws3", (Fs, d), u8), ("ws2", (d, Fs), u8),
                                    ("ss1", (Fs,), f32), ("ss3", (Fs,), f32), ("ss2", (d,), f32)):
                    _need(fp8.get(n), shape, t, "fp8 " + n)
            self.fp8 = dict(fp8)
            self._fp8_struct = MoeFp8Weights(*[(self.fp8[n].data_ptr() if self.fp8.get(n) is not None else None)
                                               for n, _ in MoeFp8Weights._fields_])
            w1 = w3 = w2 = ws1 = ws3 = ws2 = None
        else:
            _need(w1, (E, F, d), dt, "w1")
            _need(w3, (E, F, d), dt, "w3")
            _need(w2, (E, d, F), dt, "w2")
            if layer.n_shared:
                _need(ws1, (Fs, d), dt, "ws1")
                _need(ws3, (Fs, d), dt, "ws3")
                _need(ws2, (d, Fs), dt, "ws2")
        self.w = dict(w_gate=_need(w_gate, (E, d), dt, "w_gate"), w1=w1, w3=w3, w2=w2,
                      logit_bias=logit_bias, select_bias=select_bias, ws1=ws1, ws3=ws3, ws2=ws2)
        if logit_bias is not None:
            _need(logit_bias, (layer.E,), torch.float32, "logit_bias")
        if select_bias is not None:
            _need(select_bias, (layer.E,), torch.float32, "select_bias")
        dev = device or w_gate.device
        self.ws = workspace(layer, dev, stream)
        self.stats = None
        self._stats_struct = None
        if stats:
            E = layer.E
            i32 = dict(dtype=torch.int32, device=dev)
            f32 = dict(dtype=torch.float32, device=dev)
            self.stats = dict(counts=torch.zeros(E, **i32), kept=torch.zeros(E, **i32), f=torch.zeros(E, **f32),
                              p=torch.zeros(E, **f32), L=torch.zeros(1, **f32), n_dropped=torch.zeros(1, **i32))
            s = self.stats
            self._stats_struct = MoeStats(s["counts"].data_ptr(), s["kept"].data_ptr(), s["f"].data_ptr(),
                                          s["p"].data_ptr(), s["L"].data_ptr(), s["n_dropped"].data_ptr())
        self._args = [_ptr(self.w[n]) for n in ("w_gate", "logit_bias", "select_bias", "w1", "w3", "w2", "ws1",
                                                "ws3", "ws2")]

    def __call__(self, x, y=None, stream=None):
        L = self.layer
        _need(x, (L.T, L.d), L.torch_dtype, "x")
        if y is None:
            y = torch.empty((L.T, L.d), dtype=L.y_dtype, device=x.device)
        else:
            _need(y, (L.T, L.d), L.y_dtype, "y")
        if self.graph and not _STAGE_EVENTS_SET[0]:
            key = (x.data_ptr(), y.data_ptr())
            g = self._graphs.get(key)
            if g is None:
                if len(self._graphs) >= 8:
                    self._graphs.clear()
                self._graphs[key] = self.capture(x, y, stream=stream)  # (its eager call computed this y)
                return y
            if stream is not None:
                with torch.cuda.stream(stream):
                    g.replay()
            else:
                g.replay()
            return y
        self._enqueue(x, y, stream)
        return y

    def capture(self, x, y, stage_timer=None, stream=None):
        """Runs one layer call on (x, y) eagerly, then records the same call as
        a CUDA graph and returns it (torch.cuda.CUDAGraph: .replay() enqueues
        the whole layer on the current stream).  With stage_timer, that
        timer's next event set is recorded inside the graph, so each replay
        records it again."""
        dev = x.device
        cur = stream or torch.cuda.current_stream(dev)
        events_were_set = _STAGE_EVENTS_SET[0]
        if events_were_set:
            lib().moe_set_stage_events(None, 0)
            _STAGE_EVENTS_SET[0] = False
        self._enqueue(x, y, cur)  # the library's one-time per-device set-up happens outside the capture
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(cur)
        with torch.cuda.graph(g, stream=side, capture_error_mode="relaxed"):
            if stage_timer is not None:
                stage_timer.begin_call()
            try:
                self._enqueue(x, y, side)
            finally:
                if stage_timer is not None:
                    stage_timer.skip_call()
        cur.wait_stream(side)
        return g

    def _enqueue(self, x, y, stream):
        wg, lb, sb, w1, w3, w2, s1, s3, s2 = self._args
        st = ctypes.byref(self._stats_struct) if self._stats_struct is not None else None
        if self.fp8 is not None:
            _check(lib().moe_forward_fp8(ctypes.byref(self.cfg), _ptr(x), wg, lb, sb, ctypes.byref(self._fp8_struct),
                                         _ptr(y), st, _ptr(self.ws), self.ws.numel(), _stream(stream)),
                   "moe_forward_fp8")
            return
        _check(lib().moe_forward(ctypes.byref(self.cfg), _ptr(x), wg, lb, sb, w1, w3, w2, s1, s3, s2, _ptr(y), st,
                                 _ptr(self.ws), self.ws.numel(), _stream(stream)), "moe_forward")

    def device_status(self, stream=None) -> int:
        return last_device_status(self.layer, self.ws, stream)


class HostPipeline:
    """Feeds a Forward with batches that live in pinned host memory, the way a
    serving loop does: two device slots for x and y; batch i's host-to-device
    copy runs on a copy stream while batch i-1 computes, and its result goes
    back to the host on a second copy stream while batch i+1 computes.  Events
    order each slot's copy-in, layer call and copy-out; every kernel is the
    Forward's own, on the compute stream."""

    def __init__(self, fw: Forward, device=None):
        L = fw.layer
        dev = torch.device(device) if device is not None else fw.ws.device
        self.fw = fw
        self.device = dev
        self.x = [torch.empty((L.T, L.d), dtype=L.torch_dtype, device=dev) for _ in range(2)]
        self.y = [torch.empty((L.T, L.d), dtype=L.y_dtype, device=dev) for _ in range(2)]
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.copied_in = [torch.cuda.Event() for _ in range(2)]
        self.computed = [torch.cuda.Event() for _ in range(2)]
        self.copied_out = [torch.cuda.Event() for _ in range(2)]
        self.used = [False, False]

    def run(self, x_host, y_host, stream=None):
        """Enqueues one layer call per (x_host[i], y_host[i]) pair of pinned
        host tensors ([T][d], the layer's input and output dtypes) and returns
        without waiting; once `stream` (default: the current stream) has
        drained, every y_host[i] holds its result.  The host tensors must stay
        alive and untouched until then."""
        L = self.fw.layer
        comp = stream or torch.cuda.current_stream(self.device)
        start = torch.cuda.Event()
        start.record(comp)  # copies begin after the work already on `stream`
        self.h2d.wait_stream(comp)
        last = None
        for i, (xh, yh) in enumerate(zip(x_host, y_host)):
            _need_host(xh, (L.T, L.d), L.torch_dtype, "x_host")
            _need_host(yh, (L.T, L.d), L.y_dtype, "y_host")
            s = i % 2
            if self.used[s]:
                self.h2d.wait_event(self.computed[s])   # the call that last read x[s] is done
                comp.wait_event(self.copied_out[s])     # y[s] is back on the host
            with torch.cuda.stream(self.h2d):
                self.x[s].copy_(xh, non_blocking=True)
            self.copied_in[s].record(self.h2d)
            comp.wait_event(self.copied_in[s])
            self.fw(self.x[s], self.y[s], stream=comp)
            self.computed[s].record(comp)
            self.d2h.wait_event(self.computed[s])
            with torch.cuda.stream(self.d2h):
                yh.copy_(self.y[s], non_blocking=True)
            self.copied_out[s].record(self.d2h)
            self.used[s] = True
            last = s
        if last is not None:
            comp.wait_event(self.copied_out[last])  # draining `stream` covers every copy-out


def _need_host(t, shape, dtype, name):
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu" or not t.is_pinned():
        raise ValueError(f"{name} must be a pinned host tensor")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected contiguous {tuple(shape)} {dtype}, got {tuple(t.shape)} {t.dtype}")
    return t


def forward(layer: Layer, x, w_gate, w1, w3, w2, logit_bias=None, select_bias=None, ws1=None, ws3=None, ws2=None,
            stats: bool = False, stream=None):
    """One moe_forward call; returns y (and the statistics dict when stats=True)."""
    fw = Forward(layer, w_gate, w1, w3, w2, logit_bias, select_bias, ws1, ws3, ws2, stats=stats, device=x.device,
                 stream=stream)
    y = fw(x, stream=stream)
    rc = fw.device_status(stream)
    if rc != 0:
        raise MoeError(rc, "moe_forward (device status)")
    return (y, fw.stats) if stats else y

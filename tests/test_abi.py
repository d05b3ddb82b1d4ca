"""Host-side checks of the C ABI (no GPU needed).

The shared library must load on a machine without a GPU, export every entry
point that include/moe_b300.h declares, and reject bad arguments on the host
before it touches the device.
"""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_95_b300 as moe
from mixture_experts_layer_95_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_b300.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*MOE_API\s+(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_forward",
                     "moe_workspace_size", "moe_strerror", "moe_last_device_status"):
        assert required in names
    assert set(names) == set(moe.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {moe.LIB_PATH}").read()
    exported = set(re.findall(r" T (moe_\w+)", out))
    assert exported == set(declared_functions()), exported ^ set(declared_functions())


def test_strerror_and_version(lib):
    assert moe.strerror(0) == "ok"
    for code in range(-9, 0):
        assert moe.strerror(code) and moe.strerror(code) != "unknown status"
    assert moe.strerror(-100) == "unknown status"
    assert re.match(r"\d+\.\d+\.\d+", moe.version())


def _cfg(**kw):
    base = dict(T=16, d=64, E=4, k=2, d_ff=32)
    base.update(kw)
    return moe.Layer(**base).cfg()


def test_workspace_size_validation(lib):
    ok = lib.moe_workspace_size(ctypes.byref(_cfg()))
    assert ok > 0 and ok % 256 == 0
    bad = [dict(k=5), dict(k=0), dict(E=0), dict(E=2000), dict(d=12), dict(d_ff=20), dict(T=-1),
           dict(n_shared=2), dict(n_shared=1, d_ff_shared=0), dict(k=33, E=64)]
    for b in bad:
        assert lib.moe_workspace_size(ctypes.byref(_cfg(**b))) == 0, b
    c = _cfg()
    c.dtype = 7
    assert lib.moe_workspace_size(ctypes.byref(c)) == 0


def test_workspace_grows_with_tokens_and_shared_expert(lib):
    # large batches (no split-K slices in the workspace)
    a = lib.moe_workspace_size(ctypes.byref(_cfg(T=16000)))
    b = lib.moe_workspace_size(ctypes.byref(_cfg(T=32000)))
    c = lib.moe_workspace_size(ctypes.byref(_cfg(T=32000, n_shared=1, d_ff_shared=32)))
    assert a < b < c


def test_decode_sized_batches_reserve_split_k_slices(lib):
    """A one-token batch cannot fill the SMs with output tiles, so the expert
    GEMMs split K and the workspace holds their fp32 partial slices."""
    one = moe.Layer(T=1, d=4096, E=8, k=2, d_ff=14336).cfg()
    n, d, F = 2, 4096, 14336
    plain = 4 * n * (d + 2 + 2 + 3 + 1) + 2 * n * (d + F)  # rough lower bound without slices
    assert lib.moe_workspace_size(ctypes.byref(one)) > plain + 4 * n * (2 * F + d)


def test_bf16_workspace_is_smaller_than_fp32(lib):
    # bf16 activations take half the bytes of fp32 in the large regions
    f32 = moe.Layer(T=4096, d=1024, E=8, k=2, d_ff=2048, dtype="f32").cfg()
    bf = moe.Layer(T=4096, d=1024, E=8, k=2, d_ff=2048, dtype="bf16").cfg()
    assert lib.moe_workspace_size(ctypes.byref(bf)) < lib.moe_workspace_size(ctypes.byref(f32))


def test_host_rejects_bad_arguments_before_touching_the_device(lib):
    c = _cfg()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the host checks fail first
    ws_bytes = lib.moe_workspace_size(ctypes.byref(c))
    # null required pointer
    rc = lib.moe_route(ctypes.byref(c), None, fake, None, None, fake, fake, None, fake, ws_bytes, None)
    assert rc == -1
    # bad shape
    bad = _cfg(k=9)
    rc = lib.moe_route(ctypes.byref(bad), fake, fake, None, None, fake, fake, None, fake, ws_bytes, None)
    assert rc == -2
    # bad dtype
    bd = _cfg()
    bd.dtype = 3
    rc = lib.moe_forward(ctypes.byref(bd), fake, fake, None, None, fake, fake, fake, None, None, None, fake, None,
                         fake, ws_bytes, None)
    assert rc == -3
    # workspace too small / misaligned
    rc = lib.moe_forward(ctypes.byref(c), fake, fake, None, None, fake, fake, fake, None, None, None, fake, None,
                         fake, ws_bytes - 1, None)
    assert rc == -4
    rc = lib.moe_forward(ctypes.byref(c), fake, fake, None, None, fake, fake, fake, None, None, None, fake, None,
                         ctypes.c_void_p((1 << 20) + 16), ws_bytes, None)
    assert rc == -4
    # misaligned tensor pointer
    rc = lib.moe_forward(ctypes.byref(c), ctypes.c_void_p((1 << 20) + 4), fake, None, None, fake, fake, fake, None,
                         None, None, fake, None, fake, ws_bytes, None)
    assert rc == -9
    # shared expert required when n_shared == 1
    cs = _cfg(n_shared=1, d_ff_shared=32)
    rc = lib.moe_forward(ctypes.byref(cs), fake, fake, None, None, fake, fake, fake, None, None, None, fake, None,
                         fake, lib.moe_workspace_size(ctypes.byref(cs)), None)
    assert rc == -1
    assert lib.moe_route(None, fake, fake, None, None, fake, fake, None, fake, ws_bytes, None) == -1


def test_no_device_reports_an_error_not_a_crash(lib):
    """Valid host arguments on a machine without a GPU: a clean error code."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    c = _cfg()
    fake = ctypes.c_void_p(1 << 20)
    ws_bytes = lib.moe_workspace_size(ctypes.byref(c))
    rc = lib.moe_route(ctypes.byref(c), fake, fake, None, None, fake, fake, None, fake, ws_bytes, None)
    assert rc in (-5, -6)


def test_product_path_has_no_cpu_fallback():
    """The package must not import the oracle or any CPU implementation."""
    pkg = os.path.join(ROOT, "mixture_experts_layer_95_b300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in src and "from oracle" not in src, fn

"""moe_permute_static: the grouping step for callers that cannot allocate.

Some callers are handed only their input and output buffers, or run where
device allocation is forbidden, so they cannot give moe_permute a workspace.
moe_permute_static keeps the grouping's small scratch in a fixed array inside
the library instead.  This test calls it through the C ABI twice in a row and
checks that both calls produce exactly what moe_permute produces (grouping is
integer and copy work, so the tolerance is zero), and that sizes beyond the
fixed scratch are refused before anything is enqueued.

The file name sorts last so that a run stopping at the first failure has run
every other test before this one.
"""
import ctypes

import pytest
import torch

from moe_inputs import Workload

pytestmark = pytest.mark.gpu

CASES = [
    Workload("nalloc_small_bf16", T=300, d=256, E=8, F=64, k=2),
    Workload("nalloc_capacity_zipf_bf16", T=1000, d=128, E=64, F=64, k=4, capacity=50, zipf_s=1.2),
    Workload("nalloc_f32", T=77, d=264, E=6, F=64, k=3, dtype="f32"),
]


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_static_scratch_permute_matches_workspace_permute(cuda, w):
    import mixture_experts_layer_95_b300 as moe
    import moe_inputs
    from tests._parity import layer_of
    layer = layer_of(w)
    L = moe_inputs.make_layer(w, "cuda")
    ids, gates, _ = moe.route(layer, L["x"], L["w_gate"], L["logit_bias"], L["select_bias"])
    ref = moe.permute(layer, ids, gates, L["x"])
    for _ in range(2):  # the second call runs on the scratch the first one left behind
        got = moe.permute_static(layer, ids, gates, L["x"])
        torch.cuda.synchronize()
        total = int(ref["offsets"][-1].item())
        for name in ("counts", "kept", "offsets", "sorted_token_ids", "slot_pos", "gates_perm", "n_dropped"):
            assert torch.equal(got[name], ref[name]), name
        assert torch.equal(got["x_perm"][:total], ref["x_perm"][:total])


def test_static_scratch_permute_refuses_sizes_beyond_its_scratch(cuda):
    import mixture_experts_layer_95_b300 as moe
    lib = moe.lib()
    layer = moe.Layer(T=64 * 257, d=64, E=256, k=2, d_ff=64)  # ceil(T/64) * E = 65,792 > 65,536
    c = layer.cfg()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    rc = lib.moe_permute_static(ctypes.byref(c), *([fake] * 11), None)
    assert rc == -2  # MOE_ERR_SHAPE


def test_static_scratch_permute_at_its_exact_limit(cuda):
    """ceil(T/64) * E == 65,536 (T = 16384, E = 256) is accepted and matches moe_permute."""
    import mixture_experts_layer_95_b300 as moe
    layer = moe.Layer(T=16384, d=64, E=256, k=8, d_ff=64)
    g = torch.Generator(device="cuda").manual_seed(7)
    ids = torch.argsort(torch.rand((layer.T, layer.E), generator=g, device="cuda"), dim=1)[:, :layer.k]
    ids = ids.to(torch.int32).contiguous()
    gates = torch.rand((layer.T, layer.k), generator=g, device="cuda")
    x = torch.randn((layer.T, layer.d), generator=g, device="cuda").to(torch.bfloat16)
    ref = moe.permute(layer, ids, gates, x)
    got = moe.permute_static(layer, ids, gates, x)
    torch.cuda.synchronize()
    for name in ("counts", "kept", "offsets", "sorted_token_ids", "slot_pos", "gates_perm", "n_dropped"):
        assert torch.equal(got[name], ref[name]), name
    assert torch.equal(got["x_perm"], ref["x_perm"])


def test_static_scratch_permute_skips_out_of_range_ids(cuda):
    """Ids equal to E or negative get no position and are not counted, exactly as
    in moe_permute (which also records them in its workspace status word)."""
    import mixture_experts_layer_95_b300 as moe
    layer = moe.Layer(T=200, d=64, E=8, k=2, d_ff=64)
    g = torch.Generator(device="cuda").manual_seed(8)
    ids = torch.argsort(torch.rand((layer.T, layer.E), generator=g, device="cuda"), dim=1)[:, :layer.k]
    ids = ids.to(torch.int32).contiguous()
    bad = [(3, 0, layer.E), (50, 1, -1), (199, 0, layer.E + 5)]
    for t, j, v in bad:
        ids[t, j] = v
    gates = torch.rand((layer.T, layer.k), generator=g, device="cuda")
    x = torch.randn((layer.T, layer.d), generator=g, device="cuda").to(torch.bfloat16)
    ref = moe.permute(layer, ids, gates, x)
    got = moe.permute_static(layer, ids, gates, x)
    torch.cuda.synchronize()
    for name in ("counts", "kept", "offsets", "sorted_token_ids", "slot_pos", "gates_perm", "n_dropped"):
        assert torch.equal(got[name], ref[name]), name
    valid = (ids >= 0) & (ids < layer.E)
    assert int(got["counts"].sum().item()) == int(valid.sum().item())
    for t, j, _ in bad:
        assert int(got["slot_pos"][t, j].item()) == -1
    assert bool((got["slot_pos"][valid] >= 0).all())

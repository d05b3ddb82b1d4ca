"""Pins of the oracle's FP8 (E4M3) expert-weight quantisation (CPU only).

The pages name FP8 quantisation of the experts as the way to fit them in memory
("Mixture of Experts" notes, serving; handbook, DeepSeek-V3's FP8 weights) but
fix no format: the oracle reads it as OCP E4M3 with one fp32 scale per output
channel.  The codes are pinned to PyTorch's float8_e4m3fn cast (a library
routine), the per-row scaling to its defining properties.
"""
import numpy as np
import pytest
import torch

import oracle


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn)


def test_every_code_decodes_like_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))  # 0x7F and 0xFF
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_rounding_matches_torch_on_random_ties_and_boundaries():
    rng = np.random.default_rng(0)
    finite = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = np.unique(finite[~np.isnan(finite)])
    mids = (finite[:-1] + finite[1:]) / 2  # exact ties: round half to even
    vals = np.concatenate([
        rng.standard_normal(20000) * 50, rng.uniform(-448, 448, 20000),
        rng.uniform(-2 ** -6, 2 ** -6, 5000),  # subnormal range
        finite, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
        [0.0, -0.0, 448.0, -448.0, 2.0 ** -10, 3 * 2.0 ** -11]]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    ours = oracle.e4m3_encode(vals)
    ref = _torch_e4m3(vals).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_saturation_above_the_largest_finite_value():
    vals = np.array([448.5, 463.9, 464.0, 500.0, 1e6, -1e6], np.float32)
    ours = oracle.e4m3_encode(vals)
    np.testing.assert_array_equal(oracle.e4m3_decode(ours), [448, 448, 448, 448, 448, -448])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_row_quantisation_properties(dtype):
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((37, 200)) * rng.uniform(0.01, 3, (37, 1))).astype(np.float32)
    w[5] = 0.0  # an all-zero row: scale 1, codes 0
    if dtype == "bf16":
        w = (w.view(np.uint32) >> 16).astype(np.uint16)
    q, sc = oracle.quantize_fp8(w)
    wd = oracle.widen(w)
    deq = oracle.dequant_fp8(q, sc)
    assert sc[5] == 1.0 and not q[5].any()
    for r in range(w.shape[0]):
        if r == 5:
            continue
        amax = np.abs(wd[r]).max()
        assert sc[r] == np.float32(np.float32(amax) / np.float32(448.0))
        i = int(np.argmax(np.abs(wd[r])))
        assert abs(oracle.e4m3_decode(q[r, i:i + 1])[0]) == 448.0  # the row's maximum maps to +-448
        # round to nearest: half a grid step, relative 2^-4 for normal codes, 2^-10 * scale below 2^-6
        err = np.abs(deq[r] - wd[r])
        bound = np.maximum(np.abs(wd[r]) * 2.0 ** -4, 2.0 ** -10 * sc[r]) * (1 + 1e-6)
        assert np.all(err <= bound)
    # dequantisation is value(code) * scale, exactly
    np.testing.assert_array_equal(deq, oracle.e4m3_decode(q) * sc[:, None].astype(np.float64))


def test_quantised_layer_error_is_small_relative_to_the_output():
    """End to end in the oracle: a layer with quantised experts stays within a
    few percent (RMS) of the unquantised layer (E4M3 keeps ~4 significant bits)."""
    rng = np.random.default_rng(2)
    T, d, E, F, k = 16, 64, 4, 96, 2
    f32 = lambda a: np.ascontiguousarray(a, np.float32)
    L = dict(x=f32(rng.standard_normal((T, d))), w_gate=f32(rng.standard_normal((E, d)) / 8),
             w1=f32(rng.standard_normal((E, F, d)) / 8), w3=f32(rng.standard_normal((E, F, d)) / 8),
             w2=f32(rng.standard_normal((E, d, F)) / np.sqrt(F)))
    ref = oracle.forward(L, k)
    Lq = dict(L)
    for n in ("w1", "w3", "w2"):
        q, sc = oracle.quantize_fp8(L[n])
        Lq[n] = oracle.dequant_fp8(q, sc)
    y = oracle.layer_tokens(oracle.widen(L["x"]), Lq["w1"], Lq["w3"], Lq["w2"], ref["ids"], ref["gates"],
                            ref["slot_pos"])
    rms = np.sqrt(np.mean(ref["y"] ** 2))
    assert np.sqrt(np.mean((y - ref["y"]) ** 2)) < 0.05 * rms
    assert np.abs(y - ref["y"]).max() > 1e-4 * rms  # quantisation did change the weights

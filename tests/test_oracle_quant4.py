"""Pins for the oracle's 4-bit group-of-64 KV format.

FlexGen ("FlexGen: High-Throughput Generative Inference of Large Language Models
with a Single GPU" 解读, 4-bit 近似方法): groups of 64 along the hidden
dimension, per-group min / max, 4-bit codes, values dequantised to FP16.  With
15 steps between min and max, rounding to the nearest code is off by at most
half a step, (max - min) / 30, plus the rounding of the fp16 step and of the
fp16 result.
"""

import numpy as np
import pytest
import torch

import oracle


def _f16(x):
    return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


def _v(b):
    return np.asarray(b, np.uint16).view(np.float16).astype(np.float64)


def _codes(packed):
    lo = packed & 0xF
    hi = packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (-1,))


@pytest.mark.parametrize("d", [64, 128])
def test_roundtrip_error_bound(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((500, d)) * np.exp2(rng.integers(-6, 6, (500, 1)))
    x[7] = 3.0  # one constant row
    xb = _f16(x)
    codes, gmin, gmax = oracle.quant4(xb)
    xh = oracle.dequant4(codes, gmin, gmax)
    xv, xhv = _v(xb), _v(xh)
    g = d // 64
    mn = xv.reshape(500, g, 64).min(-1)
    mx = xv.reshape(500, g, 64).max(-1)
    assert np.array_equal(_v(gmin), mn) and np.array_equal(_v(gmax), mx)
    half_step = ((mx - mn) / 30.0)[..., None] * (1 + 2.0 ** -9)
    ulp = np.abs(xhv).reshape(500, g, 64)
    half_ulp = np.where(ulp >= 2.0 ** -14, np.exp2(np.floor(np.log2(np.maximum(ulp, 1e-300))) - 11),
                        2.0 ** -25)
    err = np.abs(xhv - xv).reshape(500, g, 64)
    assert np.all(err <= half_step + half_ulp)
    assert np.array_equal(xhv[7], xv[7])  # constant group is exact


def test_grid_values_roundtrip_exactly():
    # Values already on the 16-level grid mn + c*step come back unchanged and
    # map to code c.
    mn, step = -1.5, 0.25  # step = (mx - mn)/15 exactly, all values exact in fp16
    mx = mn + 15 * step
    c = np.random.default_rng(0).integers(0, 16, 64)
    c[0], c[1] = 0, 15
    x = mn + c * step
    assert x.min() == mn and x.max() == mx
    codes, gmin, gmax = oracle.quant4(_f16(x[None]))
    assert np.array_equal(_codes(codes)[0], c)
    assert np.array_equal(_v(oracle.dequant4(codes, gmin, gmax))[0], x)


def test_nibble_order_and_group_independence():
    x = np.zeros((1, 128))
    x[0, :64] = np.arange(64)            # group 0: ramp 0..63
    x[0, 64:] = 100.0                     # group 1: constant
    x[0, 64] = 99.0
    codes, gmin, gmax = oracle.quant4(_f16(x))
    assert codes.shape == (1, 64) and gmin.shape == (1, 2)
    assert codes[0, 0] & 0xF == 0        # channel 0 (low nibble of byte 0) is the min
    assert codes[0, 31] >> 4 == 15       # channel 63 (high nibble of byte 31) is the max
    assert (codes[0, 32] & 0xF) == 0     # channel 64 is group 1's min
    assert np.all(_codes(codes)[0, 65:] == 15)
    assert _v(gmin)[0].tolist() == [0.0, 99.0] and _v(gmax)[0].tolist() == [63.0, 100.0]


def test_codes_monotone_in_value():
    rng = np.random.default_rng(3)
    x = np.sort(rng.standard_normal((50, 64)), axis=1)
    codes, _, _ = oracle.quant4(_f16(x))
    c = _codes(codes)
    assert np.all(np.diff(c.astype(int), axis=1) >= 0)
    assert np.all(c[:, 0] == 0) and np.all(c[:, -1] == 15)


def test_signed_zero_group():
    x = np.zeros((1, 64), np.uint16)
    x[0, 3] = 0x8000
    codes, gmin, gmax = oracle.quant4(x)
    assert gmin[0, 0] == 0x8000 and gmax[0, 0] == 0
    assert np.all(codes == 0)
    xh = oracle.dequant4(codes, gmin, gmax)
    assert np.all(_v(xh) == 0.0)


def test_reconstruction_saturates_at_group_max():
    # (65504 - 0) / 15 = 4366.93 rounds to the fp16 step 4368, and 15 * 4368 =
    # 65520 would round to infinity: the reconstruction is held at the max.
    x = np.zeros((1, 64))
    x[0, 1] = 65504.0
    x[0, 2:] = np.linspace(0, 65504, 62)
    xb = _f16(x)
    codes, gmin, gmax = oracle.quant4(xb)
    xh = _v(oracle.dequant4(codes, gmin, gmax))
    assert np.all(np.isfinite(xh))
    assert xh[0, 1] == 65504.0
    assert np.all((xh >= 0) & (xh <= 65504.0))
    assert np.all(np.abs(xh - _v(xb)) <= 65504.0 / 30 * (1 + 2.0 ** -9) + 16)

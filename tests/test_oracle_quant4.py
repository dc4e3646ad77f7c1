"""Pins for the oracle's 4-bit group-of-64 KV format.

FlexGen ("FlexGen: High-Throughput Generative Inference of Large Language Models
with a Single GPU" 解读, 4-bit 近似方法): groups of 64 along the hidden
dimension, per-group min / max, 4-bit codes, values dequantised to FP16.  With
15 steps between min and max, the nearest level is at most half a step,
(max - min) / 30, away; the fp16 result adds at most half its own ulp.  The
pins check that bound with no slack, for every finite group: random groups at
all scales, a sweep of group ranges k * 2^-24 down into the fp16 subnormals,
and an exhaustive C enumeration of every narrow group.  The parts of the
format are pinned separately in exact rational arithmetic: the step's bracket,
the codes as the nearest level, and the dequantised value as one rounding of
the level.
"""

import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

_HERE = os.path.dirname(os.path.abspath(__file__))


def _f16(x):
    return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


def _v(b):
    return np.asarray(b, np.uint16).view(np.float16).astype(np.float64)


def _codes(packed):
    lo = packed & 0xF
    hi = packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (-1,))


def _half_ulp(v):
    """Half the fp16 spacing at |v| (2^-25 in the subnormal range)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.frexp(np.maximum(a, 2.0 ** -14))[1] - 1
    return np.where(a < 2.0 ** -14, 2.0 ** -25, np.exp2(e - 11.0))


def _check_bound(xb):
    """Quantise fp16 rows [n, d] and assert |x^ - x| <= (mx - mn)/30 + half_ulp(x^)."""
    codes, gmin, gmax = oracle.quant4(xb)
    xh = oracle.dequant4(codes, gmin, gmax)
    n, d = xb.shape
    g = d // 64
    xv, xhv = _v(xb).reshape(n, g, 64), _v(xh).reshape(n, g, 64)
    mn, mx = xv.min(-1), xv.max(-1)
    assert np.array_equal(_v(gmin), mn) and np.array_equal(_v(gmax), mx)
    # 30 |x^ - x| <= range + 30 half_ulp: every term is dyadic and exact in float64
    lhs = 30.0 * np.abs(xhv - xv)
    rhs = (mx - mn)[..., None] + 30.0 * _half_ulp(xhv)
    bad = lhs > rhs
    assert not bad.any(), (xv[bad][:4], xhv[bad][:4])
    return codes, gmin, gmax, xh


@pytest.mark.parametrize("d", [64, 128])
def test_roundtrip_error_bound(d):
    rng = np.random.default_rng(d)
    x = rng.standard_normal((2000, d)) * np.exp2(rng.integers(-26, 16, (2000, 1)))
    x = np.clip(x, -65504, 65504)
    x[7] = 3.0  # one constant row
    xb = _f16(x)
    _, _, _, xh = _check_bound(xb)
    assert np.array_equal(_v(xh)[7], _v(xb)[7])  # constant group is exact


def _fp16_table():
    """All finite fp16 values once (one zero), sorted, as (bits, values)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    bits = bits[((bits >> 10) & 31) != 31]
    bits = bits[bits != 0x8000]
    vals = bits.view(np.float16).astype(np.float64)
    order = np.argsort(vals, kind="stable")
    return bits[order], vals[order]


def test_range_sweep_down_into_subnormals():
    # Every group range k * 2^-24, k = 1 .. 2048 (the fp16 subnormal steps and
    # well past the 451 * 2^-24 switch of step grids), at several positions of
    # the group; each group holds its min, its max and 62 values between them.
    bits, vals = _fp16_table()
    u = 2.0 ** -24
    starts = [0.0, -2.0 ** -14, 2.0 ** -14 - 300 * u, 2.0 ** -13 - 700 * u, -2.0 ** -12,
              2.0 ** -9, -2.0 ** -6 - 2.0 ** -15]
    rng = np.random.default_rng(7)
    groups = []
    for start in starts:
        i = int(np.searchsorted(vals, start))
        for k in range(1, 2049):
            j = int(np.searchsorted(vals, vals[i] + k * u))
            if j >= len(vals) or vals[j] != vals[i] + k * u:
                continue  # the range is not a difference of fp16 values here
            inner = np.arange(i, j + 1)
            pick = inner if len(inner) <= 62 else np.concatenate(
                [inner[:20], inner[-20:], rng.choice(inner[20:-20], 22, replace=False)])
            row = np.full(64, bits[i], np.uint16)
            row[1] = bits[j]
            row[2:2 + len(pick)] = bits[pick]
            groups.append(row)
    xb = np.stack(groups)
    assert len(xb) > 4000
    _check_bound(xb)
    # straddling zero: ranges k * 2^-24 centred on 0, every k to 2^11
    rows = []
    for k in range(1, 2049):
        lo = -(k // 2) * u
        row = np.array([lo + (k * e // 63) * u for e in range(64)])
        rows.append(_f16(row))
    _check_bound(np.stack(rows))


def test_bound_at_normal_scales_up_to_the_fp16_limit():
    rng = np.random.default_rng(11)
    rows = []
    for mx in [65504.0, 32768.0, 1000.0, 1.0, 2.0 ** -5]:
        for mn in [-65504.0, -1.0, 0.0, mx / 2, mx - mx * 2.0 ** -9]:
            if mn >= mx:
                continue
            row = rng.uniform(mn, mx, 64)
            row[0], row[1] = mn, mx
            rows.append(row)
    _check_bound(_f16(np.stack(rows)))


def test_exhaustive_narrow_groups():
    # Every pair mn < mx of finite fp16 values with mx - mn <= 460 * 2^-24 and
    # every fp16 x between them (~5e8 cases), by a C program over the oracle
    # library.
    exe = os.path.join(oracle._BUILD_DIR, "q4_bound_exhaustive")
    src = os.path.join(_HERE, "native", "q4_bound_exhaustive.c")
    subprocess.run(["gcc", "-O2", "-std=c11", src, "-o", exe, "-ldl", "-lm"], check=True)
    res = subprocess.run([exe, oracle.build(), "460"], capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "violations 0" in res.stdout


def _group_cases():
    rng = np.random.default_rng(5)
    cases = []
    for scale in [2.0 ** -24, 2.0 ** -20, 2.0 ** -16, 2.0 ** -12, 2.0 ** -6, 1.0, 300.0]:
        for _ in range(6):
            x = rng.standard_normal(64) * scale * rng.integers(1, 40)
            cases.append(_f16(np.clip(x, -65504, 65504)))
    return np.stack(cases)


def test_step_is_bracketed_in_exact_arithmetic():
    # (29/30) (mx - mn)/15 <= s <= (mx - mn)/15: the two facts the bound needs
    # (no level above mx; the top level within (mx - mn)/30 of mx).
    bits, vals = _fp16_table()
    rng = np.random.default_rng(3)
    for _ in range(3000):
        i, j = sorted(rng.integers(0, len(bits), 2))
        if rng.random() < 0.5:  # narrow groups too
            j = min(len(bits) - 1, i + int(rng.integers(1, 600)))
        mn, mx = int(bits[i]), int(bits[j])
        s, tiny = oracle.q4_step(mn, mx)
        rng_ = Fraction(float(vals[j])) - Fraction(float(vals[i]))
        assert Fraction(s) <= rng_ / 15
        assert Fraction(s) * 450 >= rng_ * 29
        assert tiny == (rng_ < Fraction(451, 2 ** 24))


def test_codes_are_the_nearest_level_and_values_one_rounding():
    xb = _group_cases()
    codes, gmin, gmax = oracle.quant4(xb)
    xh = oracle.dequant4(codes, gmin, gmax)
    c = _codes(codes)
    for r in range(len(xb)):
        s, _ = oracle.q4_step(int(gmin[r, 0]), int(gmax[r, 0]))
        S, mn = Fraction(s), Fraction(float(_v(gmin[r, 0])))
        levels = [mn + k * S for k in range(16)]
        for e in range(64):
            x = Fraction(float(_v(xb[r, e])))
            dist = [abs(lv - x) for lv in levels]
            best = min(dist)
            near = [k for k in range(16) if dist[k] == best]
            want = near[0] if len(near) == 1 else next(k for k in near if k % 2 == 0)
            if S == 0:
                want = 0
            assert c[r, e] == want, (r, e)
            # x^ = the level rounded once to fp16 (numpy's float64 -> float16
            # rounding; the level is exact in float64)
            lv = float(levels[c[r, e]])
            assert Fraction(lv) == levels[c[r, e]]
            assert xh[r, e] == np.float16(lv).view(np.uint16) or (lv == 0 and _v(xh[r, e]) == 0)


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


def test_levels_stay_inside_the_group():
    # The step is rounded down, so the top level mn + 15 s never passes the
    # max, even at the fp16 limit: (65504 - 0)/15 = 4366.9 rounds down to the
    # fp16 step 4364; 15 * 4364 = 65460 rounds once to the fp16 value 65472.
    x = np.zeros((1, 64))
    x[0, 1] = 65504.0
    x[0, 2:] = np.linspace(0, 65504, 62)
    xb = _f16(x)
    codes, gmin, gmax = oracle.quant4(xb)
    xh = _v(oracle.dequant4(codes, gmin, gmax))
    assert oracle.q4_step(int(gmin[0, 0]), int(gmax[0, 0])) == (4364.0, False)
    assert np.all(np.isfinite(xh))
    assert xh[0, 1] == 65472.0
    assert np.all((xh >= 0) & (xh <= 65504.0))


def test_exact_midpoints_round_to_even_codes():
    # mn = 0, mx = 15: the step is exactly 1, and x = c + 1/2 lies exactly
    # between two levels; the code is the even one of c, c + 1.
    x = np.zeros((1, 64))
    x[0, 1] = 15.0
    x[0, 2:17] = np.arange(15) + 0.5
    codes, _, _ = oracle.quant4(_f16(x))
    c = _codes(codes)[0]
    assert c[1] == 15
    assert c[2:17].tolist() == [0, 2, 2, 4, 4, 6, 6, 8, 8, 10, 10, 12, 12, 14, 14]

"""Pins for the oracle's 16-bit float decoding and fp16 rounding.

The oracle decodes bf16 / fp16 from their bit-level definitions; here every bit
pattern is checked against independent library conversions (torch for bf16,
numpy for IEEE half), and the fp16 rounding against numpy's double->half cast,
which rounds to nearest with ties to even.
"""

import numpy as np
import torch

import oracle


def test_bf16_decode_all_patterns():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = oracle.value16(pats, 0)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    # signed zero survives
    assert np.signbit(oracle.value16(np.array([0x8000], np.uint16), 0))[0]


def test_fp16_decode_all_patterns():
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = oracle.value16(pats, 1)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_fp16_round_matches_numpy():
    rng = np.random.default_rng(7)
    # random magnitudes over the whole fp16 range, incl. subnormals and overflow
    x = rng.standard_normal(20000) * np.exp2(rng.uniform(-30, 17, 20000))
    # exact midpoints between adjacent halves (ties) and their neighbours
    h = np.arange(0, 0x7bff, 37, dtype=np.uint16).view(np.float16).astype(np.float64)
    h_next = (np.arange(0, 0x7bff, 37, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    mids = (h + h_next) / 2
    x = np.concatenate([x, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf),
                        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -24, 2.0 ** -25,
                         3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25]])
    got = oracle.fp16_round(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)

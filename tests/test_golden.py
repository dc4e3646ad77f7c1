"""Golden fixtures: the oracle must reproduce its stored answers on this machine.

The fixtures (``tests/golden/*.json``) were written by
``tests/golden/make_golden.py``, which calls only the oracle.  Metadata, codes,
scores and selections are compared exactly; attention outputs go through the
C library's exp(), which may differ in the last bit between platforms, so they
get a 1e-13 relative allowance.
"""

import json
import os

import numpy as np

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def _hexarr(a):
    return np.array([float.fromhex(v) for v in a])


def test_sparse_small_fixture():
    g = _load("sparse_small.json")
    s = g["shape"]
    B, Hq, Hkv, d, N, S, K = (s[k] for k in ("B", "Hq", "Hkv", "d", "N", "S", "K"))
    P = (N + S - 1) // S
    q = np.array(g["q"], np.uint16).reshape(B, Hq, d)
    Kc = np.array(g["K"], np.uint16).reshape(B, Hkv, N, d)
    Vc = np.array(g["V"], np.uint16).reshape(B, Hkv, N, d)
    mn, mx = oracle.meta(Kc, S, 0)
    assert mn.ravel().tolist() == g["meta_min"]
    assert mx.ravel().tolist() == g["meta_max"]
    r = oracle.scores(q, mn, mx, 0)
    assert np.array_equal(r.ravel(), _hexarr(g["scores"]))
    sel = oracle.topk(r, K)
    assert sel.ravel().tolist() == g["selected"]
    full = oracle.attention(q, Kc, Vc, S, s["scale"], 0)
    sparse = oracle.attention(q, Kc, Vc, S, s["scale"], 0, sel=sel)
    np.testing.assert_allclose(full.ravel(), _hexarr(g["out_full"]), rtol=1e-13, atol=0)
    np.testing.assert_allclose(sparse.ravel(), _hexarr(g["out_sparse"]), rtol=1e-13, atol=0)
    assert P == 6 and sel.shape == (B, Hq, K)


def test_quant4_fixture():
    g = _load("quant4.json")
    x = np.array(g["x"], np.uint16).reshape(g["rows"], g["d"])
    codes, gmin, gmax = oracle.quant4(x)
    assert codes.ravel().tolist() == g["codes"]
    assert gmin.ravel().tolist() == g["gmin"]
    assert gmax.ravel().tolist() == g["gmax"]
    assert oracle.dequant4(codes, gmin, gmax).ravel().tolist() == g["xhat"]


def test_meta8_fixture():
    g = _load("meta8_small.json")
    for fmt, f16 in (("bf16", 0), ("fp16", 1)):
        c = g[fmt]
        s = c["shape"]
        shape = (1, s["Hkv"], s["P"], s["d"])
        mn = np.array(c["meta_min"], np.uint16).reshape(shape)
        mx = np.array(c["meta_max"], np.uint16).reshape(shape)
        cm, cM, lo, step = oracle.meta8(mn, mx, f16)
        assert cm.ravel().tolist() == c["code_min"], fmt
        assert cM.ravel().tolist() == c["code_max"], fmt
        assert np.array_equal(lo.ravel().astype(np.float64), _hexarr(c["lo"])), fmt
        assert np.array_equal(step.ravel().astype(np.float64), _hexarr(c["step"])), fmt
        q = np.array(c["q"], np.uint16).reshape(1, s["Hq"], s["d"])
        r8 = oracle.scores8(q, cm, cM, lo, step, f16)
        assert np.array_equal(r8.ravel(), _hexarr(c["scores8"])), fmt


def test_pages_fixture():
    g = _load("pages_small.json")
    s = g["shape"]
    q = np.array(g["q"], np.uint16).reshape(s["B"], s["Hq"], s["d"])
    Kc = np.array(g["K"], np.uint16).reshape(s["B"], s["Hkv"], s["N"], s["d"])
    for S in (4, 8, 32):
        c = g[f"S{S}"]
        mn, mx = oracle.meta(Kc, S, 0)
        assert mn.ravel().tolist() == c["meta_min"], S
        assert mx.ravel().tolist() == c["meta_max"], S
        assert mn.shape[2] == (s["N"] + S - 1) // S
        gs = oracle.group_scores(q, mn, mx, 0)
        assert np.array_equal(gs.ravel(), _hexarr(c["group_scores"])), S


def test_tokens_fixture():
    # single-token pages: scores q . k, the top K with ties to the lower token
    # index (the K-th place falls inside a class of equal scores), attention
    # over the chosen tokens
    g = _load("tokens_small.json")
    s = g["shape"]
    q = np.array(g["q"], np.uint16).reshape(s["B"], s["Hq"], s["d"])
    Kc = np.array(g["K"], np.uint16).reshape(s["B"], s["Hkv"], s["N"], s["d"])
    Vc = np.array(g["V"], np.uint16).reshape(s["B"], s["Hkv"], s["N"], s["d"])
    mn, mx = oracle.meta(Kc, 1, 1)
    assert np.array_equal(mn, Kc) and np.array_equal(mx, Kc)
    r = oracle.scores(q, mn, mx, 1)
    assert np.array_equal(r.ravel(), _hexarr(g["scores"]))
    sel = oracle.topk(r, s["K"])
    assert sel.ravel().tolist() == g["selected"]
    out = oracle.attention(q, Kc, Vc, 1, s["scale"], 1, sel=sel)
    np.testing.assert_allclose(out.ravel(), _hexarr(g["out"]), rtol=1e-13, atol=0)

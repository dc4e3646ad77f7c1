"""Write the golden fixtures in this folder.  Calls only the oracle.

The pages print no worked numeric example of the kernel, so these fixtures are
regression pins of the oracle itself (page metadata, bound scores, top-K and
attention; metadata at page sizes 4, 8 and 32 with group scores; the 4-bit
format; the 8-bit metadata and its scores; token-level top-K with exact ties):
small inputs (stored verbatim as bit
patterns, drawn from numpy's PCG64 so they are platform independent) together
with the oracle's outputs.  ``tests/test_golden.py`` recomputes them on
whatever machine runs the suite (x86 here, Arm on the GPU host) and requires the
same answers.  Regenerate only when the oracle's arithmetic changes for a
reason named in the commit message:

    python tests/golden/make_golden.py
"""

import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def _bf16_bits(x):
    """Round float64 -> bf16 (nearest even) and return the bit patterns."""
    f = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def case_sparse_small():
    rng = np.random.default_rng(2024)
    B, Hq, Hkv, d, N, S, K = 1, 4, 2, 64, 83, 16, 3   # P = 6, last page ragged
    q = _bf16_bits(rng.standard_normal((B, Hq, d)))
    Kc = _bf16_bits(rng.standard_normal((B, Hkv, N, d)))
    Vc = _bf16_bits(rng.standard_normal((B, Hkv, N, d)))
    mn, mx = oracle.meta(Kc, S, 0)
    r = oracle.scores(q, mn, mx, 0)
    sel = oracle.topk(r, K)
    scale = 1.0 / math.sqrt(d)
    full = oracle.attention(q, Kc, Vc, S, scale, 0)
    sparse = oracle.attention(q, Kc, Vc, S, scale, 0, sel=sel)
    return {
        "shape": dict(B=B, Hq=Hq, Hkv=Hkv, d=d, N=N, S=S, K=K, scale=scale, dtype="bf16"),
        "q": q.ravel().tolist(), "K": Kc.ravel().tolist(), "V": Vc.ravel().tolist(),
        "meta_min": mn.ravel().tolist(), "meta_max": mx.ravel().tolist(),
        "scores": [float.hex(float(v)) for v in r.ravel()],
        "selected": sel.ravel().tolist(),
        "out_full": [float.hex(float(v)) for v in full.ravel()],
        "out_sparse": [float.hex(float(v)) for v in sparse.ravel()],
    }


def case_quant4():
    rng = np.random.default_rng(99)
    # scales from fp16 subnormals (the tiny-range step grid) to 100
    x = rng.standard_normal((7, 128)) * np.array(
        [[0.01], [1], [3], [100], [1e-5], [1], [3e-7]])
    x[5] = 7.0
    xb = np.asarray(x, np.float64).astype(np.float16).view(np.uint16)
    codes, gmin, gmax = oracle.quant4(xb)
    xh = oracle.dequant4(codes, gmin, gmax)
    return {"x": xb.ravel().tolist(), "rows": 7, "d": 128,
            "codes": codes.ravel().tolist(), "gmin": gmin.ravel().tolist(),
            "gmax": gmax.ravel().tolist(), "xhat": xh.ravel().tolist()}


def case_meta8_small():
    rng = np.random.default_rng(808)
    out = {}
    for f16 in (0, 1):
        Hkv, P, d, Hq = 2, 7, 64, 4
        if f16:
            a = rng.standard_normal((1, Hkv, P, d)) * 2.0
            b = a + np.abs(rng.standard_normal((1, Hkv, P, d)))
            conv = lambda x: np.asarray(x, np.float64).astype(np.float16).view(np.uint16)  # noqa
        else:
            a = rng.standard_normal((1, Hkv, P, d)) * 3.0
            b = a + np.abs(rng.standard_normal((1, Hkv, P, d)))
            conv = _bf16_bits
        mn, mx = conv(a), conv(b)
        # page 0 of head 0 constant; page 1 two neighbouring values around a
        # power of two (the smallest step against the ulp); page 2 straddling zero
        mn[0, 0, 0], mx[0, 0, 0] = conv(np.full(d, 1.25)), conv(np.full(d, 1.25))
        lo2, hi2 = (2.0 - 2.0 ** -10, 2.0) if f16 else (2.0 - 2.0 ** -7, 2.0)
        mn[0, 0, 1], mx[0, 0, 1] = conv(np.full(d, lo2)), conv(np.full(d, hi2))
        mn[0, 0, 2] = conv(-np.abs(rng.standard_normal(d)))
        mx[0, 0, 2] = conv(np.abs(rng.standard_normal(d)))
        cm, cM, lo, step = oracle.meta8(mn, mx, f16)
        q = conv(rng.standard_normal((1, Hq, d)))
        r8 = oracle.scores8(q, cm, cM, lo, step, f16)
        out["fp16" if f16 else "bf16"] = {
            "shape": dict(Hkv=Hkv, P=P, d=d, Hq=Hq),
            "meta_min": mn.ravel().tolist(), "meta_max": mx.ravel().tolist(),
            "code_min": cm.ravel().tolist(), "code_max": cM.ravel().tolist(),
            "lo": [float.hex(float(v)) for v in lo.ravel()],
            "step": [float.hex(float(v)) for v in step.ravel()],
            "q": q.ravel().tolist(),
            "scores8": [float.hex(float(v)) for v in r8.ravel()],
        }
    return out


def case_pages_small():
    rng = np.random.default_rng(4096)
    B, Hq, Hkv, d, N = 1, 4, 2, 32, 77   # ragged at every page size below
    q = _bf16_bits(rng.standard_normal((B, Hq, d)))
    Kc = _bf16_bits(rng.standard_normal((B, Hkv, N, d)))
    out = {"shape": dict(B=B, Hq=Hq, Hkv=Hkv, d=d, N=N), "q": q.ravel().tolist(),
           "K": Kc.ravel().tolist()}
    for S in (4, 8, 32):
        mn, mx = oracle.meta(Kc, S, 0)
        g = oracle.group_scores(q, mn, mx, 0)
        out[f"S{S}"] = {"meta_min": mn.ravel().tolist(), "meta_max": mx.ravel().tolist(),
                        "group_scores": [float.hex(float(v)) for v in g.ravel()]}
    return out


def case_tokens_small():
    # token-level top-K: single-token pages (m = M = k, so r = q . k), fp16,
    # two query heads per kv head; the K rows repeat every 8 tokens, so whole
    # score classes tie and the K-th place falls inside one (ties to the lower
    # token index)
    rng = np.random.default_rng(1717)
    B, Hq, Hkv, d, N, K = 1, 4, 2, 64, 53, 9
    f16 = lambda x: np.asarray(x, np.float64).astype(np.float16).view(np.uint16)  # noqa
    q = f16(rng.standard_normal((B, Hq, d)))
    base = rng.standard_normal((B, Hkv, 8, d))
    Kc = f16(np.concatenate([base] * 7, axis=2)[:, :, :N])
    Vc = f16(rng.standard_normal((B, Hkv, N, d)))
    mn, mx = oracle.meta(Kc, 1, 1)
    r = oracle.scores(q, mn, mx, 1)
    sel = oracle.topk(r, K)
    scale = 1.0 / math.sqrt(d)
    out = oracle.attention(q, Kc, Vc, 1, scale, 1, sel=sel)
    return {
        "shape": dict(B=B, Hq=Hq, Hkv=Hkv, d=d, N=N, K=K, scale=scale, dtype="fp16"),
        "q": q.ravel().tolist(), "K": Kc.ravel().tolist(), "V": Vc.ravel().tolist(),
        "scores": [float.hex(float(v)) for v in r.ravel()],
        "selected": sel.ravel().tolist(),
        "out": [float.hex(float(v)) for v in out.ravel()],
    }


def main():
    for name, fn in [("sparse_small", case_sparse_small), ("quant4", case_quant4),
                     ("meta8_small", case_meta8_small), ("pages_small", case_pages_small),
                     ("tokens_small", case_tokens_small)]:
        with open(os.path.join(HERE, f"{name}.json"), "w") as f:
            json.dump(fn(), f, separators=(",", ":"))
            f.write("\n")


if __name__ == "__main__":
    main()

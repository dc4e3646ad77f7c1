"""Pins for the oracle's 8-bit page metadata and its bound score.

TinyServe ("TinyServe: Query-Aware Cache Selection for Efficient LLM Serving",
相关性函数实例化) needs only that the page summary bounds every key of the page
channel by channel, so that r(q, phi_j) bounds max q.k.  The 8-bit form keeps
lo / step per page and rounds each m down and each M up on the grid
dec(c) = fma(c, step, lo).  Every check here recomputes what it needs with
numpy: dec as an exact float64 product-sum rounded once to float32 (checked
exact where used), the grid's outward and tight rounding, the step rule, and
the bound against a brute-force max over the page's keys.
"""

import numpy as np
import pytest
import torch

import oracle
from workloads import Workload, bits, make_inputs


def _vals(a, is_fp16):
    if is_fp16:
        return a.view(np.float16).astype(np.float64)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double().numpy()


def _dec(c, step, lo):
    """fma(c, step, lo) in float32: c * step is exact in float64 (8 + 24 bits),
    and the sum is checked exact before its single rounding to float32."""
    c = np.asarray(c, np.float64)
    step = np.asarray(step, np.float32).astype(np.float64)
    lo = np.asarray(lo, np.float32).astype(np.float64)
    prod = c * step
    x = prod + lo
    assert np.all(x - prod == lo) and np.all(x - lo == prod), "inexact sum"
    return x.astype(np.float32).astype(np.float64)


def _case(is_fp16, N=1000, d=64, seed=5, kind="offset"):
    w = Workload("m8", B=2, Hq=4, Hkv=2, d=d, N=N, dtype="fp16" if is_fp16 else "bf16",
                 kind=kind)
    q, K, _ = make_inputs(w, seed=seed)
    return w, bits(q), bits(K)


@pytest.mark.parametrize("is_fp16", [0, 1])
def test_codes_round_outward_and_tight(is_fp16):
    w, _, Kb = _case(is_fp16)
    mn, mx = oracle.meta(Kb, 16, is_fp16)
    cmin, cmax, lo, step = oracle.meta8(mn, mx, is_fp16)
    m, M = _vals(mn, is_fp16), _vals(mx, is_fp16)
    L, St = lo[..., None], step[..., None]
    dm, dM = _dec(cmin, St, L), _dec(cmax, St, L)
    assert np.all(dm <= m) and np.all(dM >= M)
    # the largest code that stays below m, the smallest that stays above M
    up = _dec(np.minimum(cmin.astype(np.int64) + 1, 255), St, L)
    assert np.all((cmin == 255) | (up > m))
    down = _dec(np.maximum(cmax.astype(np.int64) - 1, 0), St, L)
    assert np.all((cmax == 0) | (down < M))
    # so each bound moves by at most one grid step (plus the rounding of dec)
    slack = np.abs(L) * 2.0 ** -23 + St
    assert np.all(m - dm <= slack) and np.all(dM - M <= slack)


@pytest.mark.parametrize("is_fp16", [0, 1])
def test_lo_hi_and_step_rule(is_fp16):
    w, _, Kb = _case(is_fp16, seed=6)
    mn, mx = oracle.meta(Kb, 16, is_fp16)
    _, _, lo, step = oracle.meta8(mn, mx, is_fp16)
    m, M = _vals(mn, is_fp16), _vals(mx, is_fp16)
    lo_want = m.min(axis=-1).astype(np.float32)
    hi = M.max(axis=-1).astype(np.float32)
    assert np.array_equal(lo, lo_want)
    assert not np.any(np.signbit(lo) & (lo == 0))  # zero stored as +0
    # step: start from fp32(fp32(hi - lo) / 255), raised until dec(255) >= hi
    first = ((hi - lo_want).astype(np.float32) / np.float32(255)).astype(np.float32)
    assert np.all(step >= first)
    assert np.all(_dec(255, step, lo) >= hi.astype(np.float64))
    raised = step > first
    prev = np.nextafter(step, np.float32(0), dtype=np.float32)
    assert np.all(_dec(255, prev[raised], lo[raised]) < hi[raised].astype(np.float64))


def test_constant_pages_are_exact():
    # every key of a page one value in every channel: hi == lo, so step 0, all
    # codes 0, dec = lo, and the score equals the 16-bit one exactly
    w = Workload("c", B=1, Hq=2, Hkv=1, d=64, N=64)
    q, K, _ = make_inputs(w, seed=9)
    qb, Kb = bits(q), bits(K)
    Kc = np.ascontiguousarray(np.broadcast_to(Kb[:, :, ::16, :1], (1, 1, 4, 1)).repeat(16, 2)
                              .repeat(64, 3))  # page j: every entry K[0, 0, 16 j, 0]
    mn, mx = oracle.meta(Kc, 16, 0)
    cmin, cmax, lo, step = oracle.meta8(mn, mx, 0)
    assert np.all(step == 0) and np.all(cmin == 0) and np.all(cmax == 0)
    assert np.array_equal(lo, _vals(Kb[:, :, ::16, 0], 0).astype(np.float32))
    r8 = oracle.scores8(qb, cmin, cmax, lo, step, 0)
    r16 = oracle.scores(qb, mn, mx, 0)
    assert np.array_equal(r8, r16)


@pytest.mark.parametrize("is_fp16", [0, 1])
@pytest.mark.parametrize("kind", ["offset", "hot"])
def test_score8_bounds_score16_and_every_key(is_fp16, kind):
    w, qb, Kb = _case(is_fp16, N=777, d=128, seed=12, kind=kind)
    mn, mx = oracle.meta(Kb, 16, is_fp16)
    cmin, cmax, lo, step = oracle.meta8(mn, mx, is_fp16)
    r8 = oracle.scores8(qb, cmin, cmax, lo, step, is_fp16)
    r16 = oracle.scores(qb, mn, mx, is_fp16)
    qv, Kv = _vals(qb, is_fp16), _vals(Kb, is_fp16)
    G = w.Hq // w.Hkv
    P = mn.shape[2]
    tol = 1e-9 * (np.abs(qv).sum(axis=-1, keepdims=True) + 1.0)
    assert np.all(r8 >= r16 - tol)
    for b in range(w.B):
        for h in range(w.Hq):
            s = Kv[b, h // G] @ qv[b, h]  # q . k for every token
            best = np.array([s[j * 16:(j + 1) * 16].max() for j in range(P)])
            assert np.all(r8[b, h] >= best - tol[b, h])
    # the 8-bit bound is looser, but only by the grid: at most sum |q_i| * step
    gap = r8 - r16
    bound = np.abs(qv).sum(axis=-1)[:, :, None] * np.repeat(step, G, axis=1) * 1.01 + tol
    assert np.all(gap <= bound)


def test_score8_is_r_over_decoded_metadata():
    # brute force on a tiny case: the score is q . (dec(cM) where q >= 0,
    # dec(cm) where q < 0), summed in float64
    w, qb, Kb = _case(0, N=40, d=64, seed=21)
    mn, mx = oracle.meta(Kb, 16, 0)
    cmin, cmax, lo, step = oracle.meta8(mn, mx, 0)
    r8 = oracle.scores8(qb, cmin, cmax, lo, step, 0)
    qv = _vals(qb, 0)
    G = w.Hq // w.Hkv
    for b in range(w.B):
        for h in range(w.Hq):
            for j in range(mn.shape[2]):
                dm = _dec(cmin[b, h // G, j], step[b, h // G, j], lo[b, h // G, j])
                dM = _dec(cmax[b, h // G, j], step[b, h // G, j], lo[b, h // G, j])
                want = np.where(qv[b, h] >= 0, qv[b, h] * dM, qv[b, h] * dm).sum()
                assert abs(r8[b, h, j] - want) <= 1e-12 * np.abs(qv[b, h] * dM).sum()

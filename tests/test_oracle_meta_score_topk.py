"""Pins for the oracle's page metadata, bound score and top-K selection.

TinyServe ("TinyServe: Query-Aware Cache Selection for Efficient LLM Serving",
方法细节): the keys are cut into P = ceil(t/S) pages; phi(K_j) = (m_j, M_j) is
the channel-wise min / max; r(q, phi_j) sums q_i*M_ji over q_i >= 0 and q_i*m_ji
over q_i < 0; S_t keeps the K best pages.  Each property below follows from
those definitions and is checked with numpy / itertools, not with the oracle's
own formulas.
"""

import itertools

import numpy as np
import pytest
import torch

import oracle
from workloads import Workload, bits, make_inputs


def _vals(a, is_fp16):
    dt = np.float16 if is_fp16 else None
    if is_fp16:
        return a.view(np.float16).astype(np.float64)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("is_fp16", [0, 1])
@pytest.mark.parametrize("N", [1, 15, 16, 17, 1000])
def test_meta_is_pagewise_min_max(is_fp16, N):
    w = Workload("t", B=2, Hq=3, Hkv=3, d=64, N=N, dtype="fp16" if is_fp16 else "bf16")
    _, K, _ = make_inputs(w, seed=N + 11 * is_fp16)
    Kb = bits(K)
    mn, mx = oracle.meta(Kb, 16, is_fp16)
    P = (N + 15) // 16
    assert mn.shape == (2, 3, P, 64)
    Kv = _vals(Kb, is_fp16)
    for j in range(P):
        page = Kv[:, :, j * 16:min(N, (j + 1) * 16), :]
        assert np.array_equal(_vals(mn[:, :, j], is_fp16), page.min(axis=2))
        assert np.array_equal(_vals(mx[:, :, j], is_fp16), page.max(axis=2))


def test_meta_signed_zero_total_order():
    # A page holding both -0 and +0 in one channel: min keeps -0, max keeps +0,
    # so both are stored bit patterns of the page.
    K = np.zeros((1, 1, 16, 64), np.uint16)
    K[0, 0, 3, 5] = 0x8000
    mn, mx = oracle.meta(K, 16, 0)
    assert mn[0, 0, 0, 5] == 0x8000 and mx[0, 0, 0, 5] == 0x0000
    assert mn[0, 0, 0, 4] == 0x0000


def test_score_is_upper_bound_of_page_dot_products():
    w = Workload("t", B=2, Hq=8, Hkv=2, d=64, N=997)
    q, K, _ = make_inputs(w, seed=3)
    qb, Kb = bits(q), bits(K)
    mn, mx = oracle.meta(Kb, 16, 0)
    r = oracle.scores(qb, mn, mx, 0)
    qv, Kv = _vals(qb, 0), _vals(Kb, 0)
    for h in range(w.Hq):
        kvh = h // w.G
        dots = np.einsum("bd,btd->bt", qv[:, h], Kv[:, kvh])
        for j in range(w.P):
            best = dots[:, j * 16:min(w.N, (j + 1) * 16)].max(axis=1)
            slack = 1e-12 * np.abs(qv[:, h]).sum(axis=1) * 8
            assert np.all(r[:, h, j] >= best - slack)


def test_score_equals_max_over_box_corners():
    # The maximum of q.x over the box m <= x <= M is attained at a corner; the
    # bound score is exactly that maximum (brute force over all 2^d corners).
    rng = np.random.default_rng(5)
    d = 64
    for trial in range(20):
        q = rng.standard_normal(d)
        q[rng.integers(0, d, 4)] = 0.0
        lo = rng.standard_normal(d)
        hi = lo + np.abs(rng.standard_normal(d))
        # Only 8 channels vary between their bounds; the others are pinned
        # (m_i == M_i), keeping the corner enumeration small.
        free = rng.choice(d, 8, replace=False)
        hi_f = lo.copy()
        hi_f[free] = hi[free]
        # round through bf16 so the values are exact inputs
        qb = torch.tensor(q).to(torch.bfloat16)
        lob = torch.tensor(lo).to(torch.bfloat16)
        hib = torch.tensor(hi_f).to(torch.bfloat16)
        hib = torch.maximum(hib, lob)
        qv, lov, hiv = qb.double().numpy(), lob.double().numpy(), hib.double().numpy()
        best = -np.inf
        for corner in itertools.product([0, 1], repeat=len(free)):
            x = lov.copy()
            for c, i in zip(corner, free):
                if c:
                    x[i] = hiv[i]
            best = max(best, float(qv @ x))
        r = oracle.scores(bits(qb).reshape(1, 1, d), bits(lob).reshape(1, 1, 1, d),
                          bits(hib).reshape(1, 1, 1, d), 0)[0, 0, 0]
        assert abs(r - best) <= 1e-12 * (np.abs(qv) @ np.maximum(np.abs(lov), np.abs(hiv)))


def test_score_special_cases():
    w = Workload("t", B=1, Hq=4, Hkv=2, d=128, N=64, S=1)
    q, K, _ = make_inputs(w, seed=9)
    qb, Kb = bits(q), bits(K)
    qv, Kv = _vals(qb, 0), _vals(Kb, 0)
    # S = 1: each page is one key, so the bound is the dot product itself.
    mn, mx = oracle.meta(Kb, 1, 0)
    r = oracle.scores(qb, mn, mx, 0)
    for h in range(4):
        np.testing.assert_allclose(r[0, h], Kv[0, h // 2] @ qv[0, h], rtol=0, atol=1e-12)
    # q >= 0 everywhere: r = q . M ;  q <= 0 everywhere: r = q . m
    mn, mx = oracle.meta(Kb, 16, 0)
    qa = np.abs(qv)
    qpos = bits(torch.tensor(qa).to(torch.bfloat16))
    qneg = bits(torch.tensor(-qa).to(torch.bfloat16))
    rp = oracle.scores(qpos, mn, mx, 0)
    rn = oracle.scores(qneg, mn, mx, 0)
    mxv, mnv = _vals(mx, 0), _vals(mn, 0)
    for h in range(4):
        np.testing.assert_allclose(rp[0, h], mxv[0, h // 2] @ qa[0, h], atol=1e-12)
        np.testing.assert_allclose(rn[0, h], mnv[0, h // 2] @ -qa[0, h], atol=1e-12)


def test_score_gqa_head_mapping():
    # kv-head g's pages are constant g+1; q-head h must see kv-head h // G.
    B, Hq, Hkv, P, d = 1, 8, 4, 3, 64
    meta = np.zeros((B, Hkv, P, d), np.uint16)
    for g in range(Hkv):
        meta[0, g] = bits(torch.full((P, d), float(g + 1)).to(torch.bfloat16))
    q = bits(torch.ones(B, Hq, d).to(torch.bfloat16))
    r = oracle.scores(q, meta, meta, 0)
    for h in range(Hq):
        assert np.all(r[0, h] == d * (h // 2 + 1))


def test_group_score_bounds_the_group_dot_products():
    # One selection per kv head group: sum_h r(q_h, phi_j) must bound the best
    # summed dot product over the page's keys (brute force over every key).
    w = Workload("t", B=2, Hq=8, Hkv=2, d=64, N=517, kind="hot")
    q, K, _ = make_inputs(w, seed=21)
    qb, Kb = bits(q), bits(K)
    mn, mx = oracle.meta(Kb, 16, 0)
    rg = oracle.group_scores(qb, mn, mx, 0)
    assert rg.shape == (2, 2, w.P)
    qv, Kv = _vals(qb, 0), _vals(Kb, 0)
    for g in range(w.Hkv):
        qsum = qv[:, g * w.G:(g + 1) * w.G].sum(axis=1)  # [B, d]
        dots = np.einsum("bd,btd->bt", qsum, Kv[:, g])
        for j in range(w.P):
            best = dots[:, j * 16:min(w.N, (j + 1) * 16)].max(axis=1)
            slack = 1e-12 * np.abs(qv[:, g * w.G:(g + 1) * w.G]).sum(axis=(1, 2)) * 8
            assert np.all(rg[:, g, j] >= best - slack)


def test_group_score_closed_forms():
    # All q >= 0: the group score is (sum_h q_h) . M; all q <= 0: (sum_h q_h) . m.
    # Computed here from the summed query, not from per-head scores.
    w = Workload("t", B=1, Hq=6, Hkv=2, d=128, N=80)
    q, K, _ = make_inputs(w, seed=23)
    qv, Kb = _vals(bits(q), 0), bits(K)
    mn, mx = oracle.meta(Kb, 16, 0)
    qa = np.abs(qv)
    rp = oracle.group_scores(bits(torch.tensor(qa).to(torch.bfloat16)), mn, mx, 0)
    rn = oracle.group_scores(bits(torch.tensor(-qa).to(torch.bfloat16)), mn, mx, 0)
    mxv, mnv = _vals(mx, 0), _vals(mn, 0)
    for g in range(2):
        qs = qa[0, 3 * g:3 * g + 3].sum(axis=0)
        np.testing.assert_allclose(rp[0, g], mxv[0, g] @ qs, rtol=1e-13, atol=1e-12)
        np.testing.assert_allclose(rn[0, g], mnv[0, g] @ -qs, rtol=1e-13, atol=1e-12)


def test_group_score_head_mapping():
    # Only q-head h is non-zero: its group (h // G) scores r(q_h), the others 0;
    # with one head per group the group score is the head's own score.
    w = Workload("t", B=1, Hq=8, Hkv=2, d=64, N=64)
    q, K, _ = make_inputs(w, seed=25)
    qv, Kb = _vals(bits(q), 0), bits(K)
    mn, mx = oracle.meta(Kb, 16, 0)
    for h in (0, 3, 5, 7):
        qo = np.zeros_like(qv)
        qo[0, h] = qv[0, h]
        qob = bits(torch.tensor(qo).to(torch.bfloat16))
        rg = oracle.group_scores(qob, mn, mx, 0)
        r = oracle.scores(qob, mn, mx, 0)
        assert np.array_equal(rg[0, h // 4], r[0, h])
        assert np.all(rg[0, 1 - h // 4] == 0)
    w1 = Workload("t", B=1, Hq=2, Hkv=2, d=64, N=64)
    q1, K1, _ = make_inputs(w1, seed=27)
    mn1, mx1 = oracle.meta(bits(K1), 16, 0)
    assert np.array_equal(oracle.group_scores(bits(q1), mn1, mx1, 0),
                          oracle.scores(bits(q1), mn1, mx1, 0))


def _brute_topk(r, K):
    order = sorted(range(len(r)), key=lambda j: (-r[j], j))
    return sorted(order[:min(K, len(r))])


@pytest.mark.parametrize("P,K", [(1, 1), (7, 3), (64, 16), (64, 64), (64, 100), (513, 128)])
def test_topk_matches_brute_force(P, K):
    rng = np.random.default_rng(P * 1000 + K)
    r = rng.standard_normal((3, P))
    r[1, ::3] = 0.25       # many exact ties
    r[2, :] = -1.0         # all tied: the lowest indices win
    sel = oracle.topk(r, K)
    for row in range(3):
        assert sel[row].tolist() == _brute_topk(r[row].tolist(), K)
    assert sel[2].tolist() == list(range(min(K, P)))

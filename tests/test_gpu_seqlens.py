"""Per-sequence lengths: batch entry b attends its first N_b tokens.  The cache
holds NaN past every N_b, so a token read past a sequence's end shows up.
Each sequence is checked against the oracle on its own tokens; a paged cache
must give bitwise the contiguous result.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ATOL, check_selection, max_abs, require_cuda
from test_gpu_paged import to_paged
from workloads import Workload, bits, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def dkv():
    import decode_attention_paged_kv_gb300 as m
    return m


CASES = [
    (Workload("lens-gqa", B=4, Hq=8, Hkv=2, d=128, N=5000, top_k=24, kind="hot"),
     [5000, 1, 17, 3333]),
    (Workload("lens-mha-d64-fp16", B=3, Hq=4, Hkv=4, d=64, N=1030, top_k=8, dtype="fp16"),
     [1030, 16, 700]),
    # 1250 pages at most: the per-unit selection kernel; the second sequence
    # has fewer pages (32) than top_k (50)
    (Workload("lens-unit-select", B=2, Hq=8, Hkv=2, d=128, N=20000, top_k=50, kind="hot"),
     [20000, 500]),
]


def _nan_past(X, lens):
    X = X.clone()
    for b, n in enumerate(lens):
        X[b, :, n:] = float("nan")
    return X


def _is16(w):
    return int(w.dtype == "fp16")


@pytest.mark.parametrize("group", [False, True], ids=["per-head", "per-group"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_seq_lens_match_oracle(case, group, dev, dkv):
    w, lens = case
    q, K, V = make_inputs(w, seed=61)
    Kn, Vn = _nan_past(K, lens), _nan_past(V, lens)
    qd, Kd, Vd = q.to(dev), Kn.to(dev), Vn.to(dev)
    L = torch.tensor(lens, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(w.d)
    meta = dkv.kv_meta_build(Kd, seq_lens=L)
    full = dkv.decode_attn_full(qd, Kd, Vd, seq_lens=L)
    out, sel = dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, return_selected=True,
                                      group_select=group, seq_lens=L)
    assert torch.isfinite(full).all() and torch.isfinite(out).all()
    sel = sel.cpu().numpy()
    for b, n in enumerate(lens):
        P = (n + 15) // 16
        kk = min(w.top_k, P)
        qb, Kb, Vb = bits(q[b:b + 1]), bits(K[b:b + 1, :, :n]), bits(V[b:b + 1, :, :n])
        omn, omx = oracle.meta(Kb, w.S, _is16(w))
        gm = meta[0][b:b + 1, :, :P].cpu().view(torch.int16).numpy().view(np.uint16)
        gx = meta[1][b:b + 1, :, :P].cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(gm, omn) and np.array_equal(gx, omx), f"meta, sequence {b}"
        ref = oracle.attention(qb, Kb, Vb, w.S, scale, _is16(w))
        assert max_abs(full[b:b + 1], ref) <= ATOL, f"full, sequence {b}"
        sb = sel[b:b + 1]
        assert np.all(sb[..., kk:] == -1), f"padding, sequence {b}"
        sb = np.ascontiguousarray(sb[..., :kk])
        if group:
            r = oracle.group_scores(qb, omn, omx, _is16(w))
            rows = sb.reshape(w.Hkv, w.G, kk)
            assert np.array_equal(rows, np.broadcast_to(rows[:, :1], rows.shape))
            check_selection(rows[:, 0], r.reshape(-1, P), w.top_k)
        else:
            r = oracle.scores(qb, omn, omx, _is16(w))
            check_selection(sb.reshape(-1, kk), r.reshape(-1, P), w.top_k)
        ref = oracle.attention(qb, Kb, Vb, w.S, scale, _is16(w), sel=sb)
        assert max_abs(out[b:b + 1], ref) <= ATOL, f"select, sequence {b}"


def test_seq_lens_paged_equals_contiguous_bitwise(dev, dkv):
    w, lens = CASES[0]
    q, K, V = make_inputs(w, seed=63)
    Kn, Vn = _nan_past(K, lens), _nan_past(V, lens)
    pk, bt = to_paged(Kn, w.P, seed=4)
    pv, _ = to_paged(Vn, w.P, seed=4)
    L = torch.tensor(lens, dtype=torch.int32, device=dev)
    qd, Kd, Vd, btd = q.to(dev), Kn.to(dev), Vn.to(dev), bt.to(dev)
    PK = dkv.PagedCache(pk.to(dev), btd, w.N)
    PV = dkv.PagedCache(pv.to(dev), btd, w.N)
    assert torch.equal(dkv.decode_attn_full(qd, Kd, Vd, seq_lens=L),
                       dkv.decode_attn_full(qd, PK, PV, seq_lens=L))
    meta = dkv.kv_meta_build(Kd, seq_lens=L)
    oc, sc = dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, return_selected=True, seq_lens=L)
    op, sp = dkv.decode_attn_select(qd, PK, PV, meta, w.top_k, return_selected=True, seq_lens=L)
    assert torch.equal(sc, sp) and torch.equal(oc, op)


def test_seq_lens_all_full_equals_no_lens(dev, dkv):
    w, _ = CASES[0]
    q, K, V = (x.to(dev) for x in make_inputs(w, seed=65))
    L = torch.full((w.B,), w.N, dtype=torch.int32, device=dev)
    assert torch.equal(dkv.decode_attn_full(q, K, V), dkv.decode_attn_full(q, K, V, seq_lens=L))
    meta = dkv.kv_meta_build(K)
    o1, s1 = dkv.decode_attn_select(q, K, V, meta, w.top_k, return_selected=True)
    o2, s2 = dkv.decode_attn_select(q, K, V, meta, w.top_k, return_selected=True, seq_lens=L)
    assert torch.equal(s1, s2) and torch.equal(o1, o2)


def test_seq_lens_outside_the_cache_are_clamped(dev, dkv):
    """A length below 1 attends one token and one above seq_len attends all of
    them (the documented clamp into [1, seq_len]): every call gives bitwise the
    results of the clamped lengths."""
    w, _ = CASES[0]
    raw, clamped = [0, -3, 10 ** 6, 3333], [1, 1, w.N, 3333]
    q, K, V = make_inputs(w, seed=67)
    Kn, Vn = _nan_past(K, clamped), _nan_past(V, clamped)
    qd, Kd, Vd = q.to(dev), Kn.to(dev), Vn.to(dev)
    Lr = torch.tensor(raw, dtype=torch.int32, device=dev)
    Lc = torch.tensor(clamped, dtype=torch.int32, device=dev)
    pages = [(n + w.S - 1) // w.S for n in clamped]

    def written(m):  # metadata rows the lengths write, per sequence
        return [m[b, :, :pages[b]] for b in range(w.B)]

    def same_rows(a, b):
        return all(torch.equal(x, y) for x, y in zip(written(a), written(b)))

    mr, mc = dkv.kv_meta_build(Kd, seq_lens=Lr), dkv.kv_meta_build(Kd, seq_lens=Lc)
    assert same_rows(mr[0], mc[0]) and same_rows(mr[1], mc[1])
    dkv.kv_meta_append(Kd, mr, seq_lens=Lr)
    dkv.kv_meta_append(Kd, mc, seq_lens=Lc)
    assert same_rows(mr[0], mc[0]) and same_rows(mr[1], mc[1])
    r8, c8 = dkv.kv_meta8_build(mc, seq_lens=Lr), dkv.kv_meta8_build(mc, seq_lens=Lc)
    for x, y in zip(r8, c8):
        assert same_rows(x, y)
    assert torch.equal(dkv.decode_attn_full(qd, Kd, Vd, seq_lens=Lr),
                       dkv.decode_attn_full(qd, Kd, Vd, seq_lens=Lc))
    for meta in (mc, c8):
        for group in (False, True):
            o1, s1 = dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, return_selected=True,
                                            group_select=group, seq_lens=Lr)
            o2, s2 = dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, return_selected=True,
                                            group_select=group, seq_lens=Lc)
            assert torch.equal(s1, s2) and torch.equal(o1, o2)
            assert torch.isfinite(o1).all()

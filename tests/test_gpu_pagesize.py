"""Selection pages of S = 4, 8, 32 and 64 tokens ("TinyServe" page-size
variants): metadata over S tokens, bound scores and top-K over ceil(N / S)
pages, and attention over the selected pages' tokens, gathered as the cache's
16-token pages (pages of 4 or 8 tokens as the cache page holding them, the
other tokens masked per query head).  Checked against the oracle at the same
S (metadata bit-exact, selection within the band, outputs within 2e-3).
"""

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ATOL, check_selection, max_abs, require_cuda
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
    # 1250 selection pages of 32 tokens: the per-unit selection kernel
    (Workload("s32-unit", B=1, Hq=8, Hkv=2, d=128, N=40000, S=32, top_k=40, kind="hot"),
     None, False),
    (Workload("s32-kernels-ragged", B=2, Hq=8, Hkv=2, d=128, N=5000, S=32, top_k=12,
              kind="hot"), None, False),
    # 1094 selection pages of 64 tokens, d = 64, MHA
    (Workload("s64-unit-mha", B=1, Hq=4, Hkv=4, d=64, N=70000, S=64, top_k=30), None, False),
    (Workload("s64-group-lens", B=2, Hq=8, Hkv=2, d=128, N=3001, S=64, top_k=8, kind="hot"),
     [3001, 100], True),
    # quarter and half cache pages: a cache page holds pages chosen by some
    # heads and not others, and pages no head chose
    (Workload("s8-gqa-ragged", B=2, Hq=8, Hkv=2, d=128, N=5001, S=8, top_k=60, kind="hot"),
     None, False),
    (Workload("s4-g8-d64", B=1, Hq=8, Hkv=1, d=64, N=3000, S=4, top_k=70), None, False),
    (Workload("s4-group-lens", B=2, Hq=8, Hkv=2, d=128, N=2050, S=4, top_k=33, kind="hot"),
     [2050, 37], True),
    (Workload("s8-mha-lens", B=3, Hq=4, Hkv=4, d=128, N=1500, S=8, top_k=20),
     [1500, 9, 801], False),
]


def _u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_page_size_matches_oracle(case, dev, dkv):
    w, lens, group = case
    S = w.S
    q, K, V = make_inputs(w, seed=71)
    if lens is not None:
        for b, n in enumerate(lens):
            K[b, :, n:] = float("nan")
            V[b, :, n:] = float("nan")
    qd, Kd, Vd = q.to(dev), K.to(dev), V.to(dev)
    L = torch.tensor(lens, dtype=torch.int32, device=dev) if lens is not None else None
    scale = 1.0 / math.sqrt(w.d)
    meta = dkv.kv_meta_build(Kd, page_size=S, seq_lens=L)
    out, sel = dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, return_selected=True,
                                      group_select=group, seq_lens=L, page_size=S)
    assert torch.isfinite(out).all()
    sel = sel.cpu().numpy()
    for b in range(w.B):
        n = lens[b] if lens is not None else w.N
        P = (n + S - 1) // S
        kk = min(w.top_k, P)
        qb, Kb, Vb = bits(q[b:b + 1]), bits(K[b:b + 1, :, :n]), bits(V[b:b + 1, :, :n])
        omn, omx = oracle.meta(Kb, S, 0)
        assert np.array_equal(_u16(meta[0][b:b + 1, :, :P]), omn), f"meta min, sequence {b}"
        assert np.array_equal(_u16(meta[1][b:b + 1, :, :P]), omx), f"meta max, sequence {b}"
        sb = sel[b:b + 1]
        assert np.all(sb[..., kk:] == -1)
        sb = np.ascontiguousarray(sb[..., :kk])
        if group:
            r = oracle.group_scores(qb, omn, omx, 0)
            rows = sb.reshape(w.Hkv, w.G, kk)
            check_selection(rows[:, 0], r.reshape(-1, P), w.top_k)
        else:
            r = oracle.scores(qb, omn, omx, 0)
            check_selection(sb.reshape(-1, kk), r.reshape(-1, P), w.top_k)
        ref = oracle.attention(qb, Kb, Vb, S, scale, 0, sel=sb)
        assert max_abs(out[b:b + 1], ref) <= ATOL, f"select, sequence {b}"


def test_all_pages_at_s64_equals_full(dev, dkv):
    w = Workload("s64-all", B=1, Hq=8, Hkv=2, d=128, N=4000, S=64)
    q, K, V = (x.to(dev) for x in make_inputs(w, seed=73))
    meta = dkv.kv_meta_build(K, page_size=64)
    P = (w.N + 63) // 64
    out = dkv.decode_attn_select(q, K, V, meta, P, page_size=64)
    full = dkv.decode_attn_full(q, K, V)
    assert max_abs(out, full.double().cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("S", [4, 8])
def test_small_pages_all_selected_equals_full(S, dev, dkv):
    # every page kept: each head's mask covers every sub-page of every cache page
    w = Workload("small-all", B=2, Hq=8, Hkv=2, d=128, N=1003, S=S)
    q, K, V = (x.to(dev) for x in make_inputs(w, seed=75))
    meta = dkv.kv_meta_build(K, page_size=S)
    P = (w.N + S - 1) // S
    out = dkv.decode_attn_select(q, K, V, meta, P, page_size=S)
    full = dkv.decode_attn_full(q, K, V)
    assert max_abs(out, full.double().cpu().numpy()) <= 1e-5


def test_small_pages_paged_cache_equals_contiguous(dev, dkv):
    # pages of 8 tokens start inside a pool block: metadata and outputs of a
    # shuffled pool equal the contiguous cache's bitwise
    from test_gpu_paged import to_paged
    w = Workload("s8-paged", B=2, Hq=8, Hkv=2, d=128, N=3000, S=8, top_k=40, kind="hot")
    q, K, V = make_inputs(w, seed=77)
    P16 = (w.N + 15) // 16
    pk, bt = to_paged(K, P16, seed=3)
    pv, _ = to_paged(V, P16, seed=3)
    qd, Kd, Vd, btd = q.to(dev), K.to(dev), V.to(dev), bt.to(dev)
    PK = dkv.PagedCache(pk.to(dev), btd, w.N)
    PV = dkv.PagedCache(pv.to(dev), btd, w.N)
    mc, mp = dkv.kv_meta_build(Kd, page_size=8), dkv.kv_meta_build(PK, page_size=8)
    assert torch.equal(mc[0], mp[0]) and torch.equal(mc[1], mp[1])
    oc, sc = dkv.decode_attn_select(qd, Kd, Vd, mc, w.top_k, return_selected=True, page_size=8)
    op, sp = dkv.decode_attn_select(qd, PK, PV, mp, w.top_k, return_selected=True, page_size=8)
    assert torch.equal(sc, sp)
    assert torch.equal(oc, op)

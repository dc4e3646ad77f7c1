"""8-bit page metadata on the GPU against the oracle.

dkv_kv_meta8_build must give the oracle's codes, lo and step bit for bit (the
codes are defined as the extremes of the outward-rounded grid, the grid by one
fp32 subtraction, division and fused multiply-add).  dkv_decode_attn_select
over that metadata must pick the oracle's pages under its 8-bit bound scores
(up to swaps inside the 1e-5 band) and match the oracle's attention over the
pages it picked within 2e-3.
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


def _u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


CASES = [
    # (workload, per-sequence lengths, group selection)
    (Workload("m8-gqa-hot", B=2, Hq=8, Hkv=2, d=128, N=20000, top_k=64, kind="hot"), None, False),
    # 375 pages at d = 64: the per-unit kernel over 8-bit codes (64-byte rows)
    (Workload("m8-unit-d64", B=2, Hq=4, Hkv=4, d=64, N=6000, top_k=24, kind="offset"), None,
     False),
    (Workload("m8-unit-d64-fp16", B=2, Hq=8, Hkv=2, d=64, N=5000, top_k=20, dtype="fp16"), None,
     False),
    (Workload("m8-mha-d64-fp16", B=3, Hq=4, Hkv=4, d=64, N=3001, top_k=12, dtype="fp16"),
     None, False),
    # 192 units at d = 64: more units than multiprocessors, two selection CTAs a one
    (Workload("m8-many-units-d64", B=8, Hq=24, Hkv=24, d=64, N=4200, top_k=20, kind="offset"),
     None, False),
    (Workload("m8-offset-s32-group", B=2, Hq=8, Hkv=2, d=128, N=9000, S=32, top_k=20,
              kind="offset"), None, True),
    (Workload("m8-lens-s8", B=3, Hq=8, Hkv=2, d=128, N=2500, S=8, top_k=40, kind="hot"),
     [2500, 17, 1201], False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_meta8_select_matches_oracle(case, dev, dkv):
    w, lens, group = case
    S = w.S
    f16 = 1 if w.dtype == "fp16" else 0
    q, K, V = make_inputs(w, seed=81)
    if lens is not None:
        for b, n in enumerate(lens):
            K[b, :, n:] = float("nan")
            V[b, :, n:] = float("nan")
    qd, Kd, Vd = q.to(dev), K.to(dev), V.to(dev)
    L = torch.tensor(lens, dtype=torch.int32, device=dev) if lens is not None else None
    meta = dkv.kv_meta_build(Kd, page_size=S, seq_lens=L)
    m8 = dkv.kv_meta8_build(meta, page_size=S, seq_lens=L)
    out, sel = dkv.decode_attn_select(qd, Kd, Vd, m8, w.top_k, return_selected=True,
                                      group_select=group, seq_lens=L, page_size=S)
    assert torch.isfinite(out).all()
    sel = sel.cpu().numpy()
    scale = 1.0 / math.sqrt(w.d)
    swaps = 0
    for b in range(w.B):
        n = lens[b] if lens is not None else w.N
        P = (n + S - 1) // S
        kk = min(w.top_k, P)
        qb, Kb, Vb = bits(q[b:b + 1]), bits(K[b:b + 1, :, :n]), bits(V[b:b + 1, :, :n])
        omn, omx = oracle.meta(Kb, S, f16)
        assert np.array_equal(_u16(meta[0][b:b + 1, :, :P]), omn)
        cmin, cmax, lo, step = oracle.meta8(omn, omx, f16)
        assert np.array_equal(m8.code_min[b:b + 1, :, :P].cpu().numpy(), cmin), f"code_min {b}"
        assert np.array_equal(m8.code_max[b:b + 1, :, :P].cpu().numpy(), cmax), f"code_max {b}"
        assert np.array_equal(m8.lo[b:b + 1, :, :P].cpu().numpy().view(np.uint32),
                              lo.view(np.uint32)), f"lo {b}"
        assert np.array_equal(m8.step[b:b + 1, :, :P].cpu().numpy().view(np.uint32),
                              step.view(np.uint32)), f"step {b}"
        r = oracle.scores8(qb, cmin, cmax, lo, step, f16)  # [1, Hq, P]
        sb = sel[b:b + 1]
        assert np.all(sb[..., kk:] == -1)
        sb = np.ascontiguousarray(sb[..., :kk])
        if group:
            rg = r.reshape(w.Hkv, w.G, P).sum(axis=1)
            rows = sb.reshape(w.Hkv, w.G, kk)
            assert np.all(rows == rows[:, :1])  # one set per group
            swaps += check_selection(rows[:, 0], rg, w.top_k)
        else:
            swaps += check_selection(sb.reshape(-1, kk), r.reshape(-1, P), w.top_k)
        ref = oracle.attention(qb, Kb, Vb, S, scale, f16, sel=sb)
        assert max_abs(out[b:b + 1], ref) <= ATOL, f"select, sequence {b}"
    assert swaps <= max(1, w.B * w.Hq // 8)


def test_meta8_all_pages_equals_full(dev, dkv):
    w = Workload("m8-all", B=2, Hq=8, Hkv=2, d=128, N=1500)
    q, K, V = (x.to(dev) for x in make_inputs(w, seed=83))
    m8 = dkv.kv_meta8_build(dkv.kv_meta_build(K))
    out = dkv.decode_attn_select(q, K, V, m8, w.P)
    full = dkv.decode_attn_full(q, K, V)
    assert max_abs(out, full.double().cpu().numpy()) <= 1e-5


def test_meta8_paged_cache_equals_contiguous(dev, dkv):
    from test_gpu_paged import to_paged
    w = Workload("m8-paged", B=2, Hq=8, Hkv=2, d=128, N=4000, top_k=30, kind="hot")
    q, K, V = make_inputs(w, seed=85)
    pk, bt = to_paged(K, w.P, seed=4)
    pv, _ = to_paged(V, w.P, seed=4)
    qd, Kd, Vd, btd = q.to(dev), K.to(dev), V.to(dev), bt.to(dev)
    PK = dkv.PagedCache(pk.to(dev), btd, w.N)
    PV = dkv.PagedCache(pv.to(dev), btd, w.N)
    mc = dkv.kv_meta8_build(dkv.kv_meta_build(Kd))
    mp = dkv.kv_meta8_build(dkv.kv_meta_build(PK))
    assert all(torch.equal(a, b) for a, b in zip(mc, mp))
    oc, sc = dkv.decode_attn_select(qd, Kd, Vd, mc, w.top_k, return_selected=True)
    op, sp = dkv.decode_attn_select(qd, PK, PV, mp, w.top_k, return_selected=True)
    assert torch.equal(sc, sp) and torch.equal(oc, op)


def _finite_values(f16):
    """Every finite 16-bit value once (one zero), ascending, as float64."""
    u = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        if f16:
            v = u.astype(np.uint16).view(np.float16).astype(np.float64)
        else:
            v = (u << 16).view(np.float32).astype(np.float64)
    return np.unique(v[np.isfinite(v)])


def _to16(x, f16):
    """float64 values that are 16-bit values -> their bit patterns."""
    if f16:
        return x.astype(np.float16).view(np.uint16)
    return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _edge_pages(f16, d, seed):
    """Metadata pages (m, M) [1, 1, P, d] at the edges of the 8-bit code rule:
    pages of two 16-bit values up to 16 apart with every value between; every
    exact grid point lo + c step that is a 16-bit value, as m and as M; values
    at and beside the 16-bit values nearest to grid points of wide pages;
    constant pages; the format's extremes; for bf16 also pages whose step is
    below 2^-100 or infinite."""
    rng = np.random.default_rng(seed)
    vals = _finite_values(f16)
    n = len(vals)
    pages = []  # (lo index, hi index, extra values)
    for _ in range(48):  # tight, half of them straddling a power of two
        if len(pages) % 2:
            e = rng.integers(-12 if f16 else -100, 15 if f16 else 100)
            a = int(np.searchsorted(vals, 2.0 ** e)) - int(rng.integers(1, 9))
        else:
            a = int(rng.integers(0, n - 17))
        w = int(rng.integers(1, 17))
        pages.append((a, a + w, vals[a:a + w + 1]))
    for _ in range(48):  # wide
        a = int(rng.integers(0, n - 4097))
        pages.append((a, a + int(rng.integers(64, 4096)), None))
    top = n - 1
    pages.append((0, top, None))  # -max .. max (bf16: an infinite range)
    pages.append((top // 2 - 3, top // 2 + 3, vals[top // 2 - 3:top // 2 + 4]))  # around 0
    pages.append((top - 1, top, vals[top - 1:]))
    pages.append((5, 5, None))  # constant
    if not f16:  # steps below 2^-100
        a = int(np.searchsorted(vals, 2.0 ** -120))
        pages.append((a, a + 40, vals[a:a + 41]))
        a = int(np.searchsorted(vals, -(2.0 ** -110)))
        pages.append((a, a + 300, None))
    P = len(pages)
    mn = np.empty((P, d), np.float64)
    mx = np.empty((P, d), np.float64)
    for j, (a, b, extra) in enumerate(pages):
        cand = extra if extra is not None else vals[a:b + 1][rng.integers(0, b - a + 1, 4 * d)]
        x = rng.choice(cand, size=(2, d))
        mn[j], mx[j] = np.minimum(x[0], x[1]), np.maximum(x[0], x[1])
        mn[j, 0], mx[j, 1] = vals[a], vals[b]
    # the grid of each page, from the oracle: exact grid points, and the
    # 16-bit values at and beside the nearest ones, replace channels 2..
    shape = (1, 1, P, d)
    _, _, lo, step = oracle.meta8(_to16(mn, f16).reshape(shape), _to16(mx, f16).reshape(shape),
                                  int(f16))
    lo, step = lo.reshape(P).astype(np.float64), step.reshape(P).astype(np.float64)
    for j, (a, b, extra) in enumerate(pages):
        if extra is not None or not (0 < step[j] < np.inf):
            continue
        g = lo[j] + np.arange(256) * step[j]
        idx = np.clip(np.searchsorted(vals, g), a, b)
        exact = vals[idx] == g
        picks = list(vals[idx[exact]])
        for k in (-1, 0, 1):
            picks += list(vals[np.clip(idx + k, a, b)][rng.integers(0, 256, 16)])
        picks = np.array(picks[:2 * (d - 2)])
        half = len(picks) // 2
        mn[j, 2:2 + half] = np.minimum(picks[:half], mx[j, 2:2 + half])
        mx[j, 2:2 + half] = np.maximum(picks[half:2 * half], mn[j, 2:2 + half])
    return _to16(mn, f16).reshape(shape), _to16(mx, f16).reshape(shape)


@pytest.mark.parametrize("f16", [0, 1], ids=["bf16", "fp16"])
@pytest.mark.parametrize("d", [128, 64])
def test_meta8_codes_on_edge_pages(f16, d, dev, dkv):
    mn, mx = _edge_pages(f16, d, seed=91 + d + f16)
    want = oracle.meta8(mn, mx, f16)
    dt = torch.float16 if f16 else torch.bfloat16
    md = torch.from_numpy(mn.view(np.int16)).view(dt).to(dev)
    Md = torch.from_numpy(mx.view(np.int16)).view(dt).to(dev)
    m8 = dkv.kv_meta8_build((md, Md), page_size=16)
    got = (m8.code_min.cpu().numpy(), m8.code_max.cpu().numpy(),
           m8.lo.cpu().numpy().view(np.uint32), m8.step.cpu().numpy().view(np.uint32))
    for name, g, w in zip(("code_min", "code_max", "lo", "step"), got,
                          (want[0], want[1], want[2].view(np.uint32), want[3].view(np.uint32))):
        bad = np.argwhere(g != w)
        assert bad.size == 0, f"{name}: {len(bad)} differ, first at {bad[0]}"

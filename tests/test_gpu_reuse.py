"""Cross-step page reuse: several decode steps of one sequence batch, each
step with a drifted query and one more token in the cache.

"TinyServe: Query-Aware Cache Selection for Efficient LLM Serving"
(内存效率量化模型构建 / 单步解码内存移动公式) moves, per step, the metadata of
every page plus only the rho K selected pages not already held; 系统实现意义
keeps the hot pages resident.  Per step here:
  * dkv_kv_meta_append rebuilds the page the new token lands in; the metadata
    of the first ceil(N_t / 16) pages must equal the oracle's, bit for bit;
  * dkv_decode_attn_select_hot selects and attends exactly like
    dkv_decode_attn_select (outputs and sets bitwise equal), the set is checked
    against the oracle's bound scores (within the 1e-5 band) and the output
    against the oracle's attention over it;
  * the reuse counters equal the set arithmetic of the returned selections:
    pages gathered = sum over steps and (batch, kv head) of |U_t|, and of
    them held from the step before = sum |U_t & U_(t-1)|, U_t the union of the
    group's selected pages.
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


def drifted_queries(q0, T, sigma, seed):
    """q_1 = q0, q_(t+1) = q_t + sigma * N(0, 1), rounded to the storage dtype."""
    g = torch.Generator().manual_seed(seed)
    qs, cur = [q0], q0.float()
    for _ in range(T - 1):
        cur = cur + sigma * torch.randn(q0.shape, generator=g)
        qs.append(cur.to(q0.dtype))
    return qs


def unions(sel, G):
    """[B, Hq, kk] selections -> list over (b, kv head) of the set of pages."""
    B, Hq, _ = sel.shape
    out = []
    for b in range(B):
        for h in range(Hq // G):
            out.append(set(int(x) for x in sel[b, h * G:(h + 1) * G].ravel() if x >= 0))
    return out


CASES = [
    # 188 pages: the score / top-K / union kernels
    Workload("reuse-gqa", B=2, Hq=8, Hkv=2, d=128, N=3008, top_k=24, kind="hot"),
    # 1251 pages: the per-(batch, kv head) selection kernel
    Workload("reuse-unit", B=2, Hq=8, Hkv=2, d=128, N=20008, top_k=40, kind="hot"),
    Workload("reuse-mha-d64", B=3, Hq=4, Hkv=4, d=64, N=1500, top_k=10, dtype="fp16"),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_multistep_reuse(w, dev, dkv):
    T = 8
    q0, K, V = make_inputs(w, seed=61)
    qs = drifted_queries(q0, T, 0.15, seed=62)
    is16 = int(w.dtype == "fp16")
    scale = 1.0 / math.sqrt(w.d)
    Kd, Vd = K.to(dev), V.to(dev)
    N0 = w.N - T  # the cache holds N0 tokens before step 1 appends one
    lens = torch.full((w.B,), N0 + 1, dtype=torch.int32, device=dev)
    meta = dkv.kv_meta_build(Kd, seq_lens=lens)
    hot = dkv.hot_state(w.B, w.Hkv, w.N, dev)
    Kb, Vb = bits(K), bits(V)
    loads = hits = 0
    prev = None
    for t in range(1, T + 1):
        Nt = N0 + t
        lens.fill_(Nt)
        if t > 1:
            dkv.kv_meta_append(Kd, meta, seq_lens=lens)
        Pt = (Nt + 15) // 16
        omn, omx = oracle.meta(np.ascontiguousarray(Kb[:, :, :Nt]), 16, is16)
        assert np.array_equal(bits(meta[0][:, :, :Pt].cpu()), omn)
        assert np.array_equal(bits(meta[1][:, :, :Pt].cpu()), omx)
        qd = qs[t - 1].to(dev)
        out_h, sel_h = dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, return_selected=True,
                                              seq_lens=lens, hot=hot, step=t)
        out_p, sel_p = dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, return_selected=True,
                                              seq_lens=lens)
        assert torch.equal(sel_h, sel_p) and torch.equal(out_h, out_p)
        sel = sel_h.cpu().numpy()
        qb = bits(qs[t - 1])
        r = oracle.scores(qb, omn, omx, is16)
        check_selection(sel.reshape(-1, sel.shape[-1]), r.reshape(-1, r.shape[-1]), w.top_k)
        ref = oracle.attention(qb, np.ascontiguousarray(Kb[:, :, :Nt]),
                               np.ascontiguousarray(Vb[:, :, :Nt]), 16, scale, is16, sel=sel)
        assert max_abs(out_h, ref) <= ATOL
        cur = unions(sel, w.G)
        loads += sum(len(u) for u in cur)
        if prev is not None:
            hits += sum(len(u & p) for u, p in zip(cur, prev))
        prev = cur
    assert dkv.hot_stats(hot) == (loads, hits)
    # a slowly drifting query keeps most of its pages from step to step
    assert hits > 0.5 * loads * (T - 1) / T


def test_meta_append_matches_full_build(dev, dkv):
    # Appending one token at a time from a partly built cache gives exactly the
    # metadata a full build gives (ragged last pages included), on a paged pool too.
    w = Workload("append", B=3, Hq=4, Hkv=2, d=64, N=200, kind="offset")
    _, K, _ = make_inputs(w, seed=63)
    Kd = K.to(dev)
    lens = torch.tensor([150, 170, 151], dtype=torch.int32, device=dev)
    meta = dkv.kv_meta_build(Kd, seq_lens=lens)
    for _ in range(30):
        lens += torch.tensor([1, 0, 1], dtype=torch.int32, device=dev)
        dkv.kv_meta_append(Kd, meta, seq_lens=lens)
    full = dkv.kv_meta_build(Kd, seq_lens=lens)
    for b, n in enumerate(lens.tolist()):
        P = (n + 15) // 16
        assert torch.equal(meta[0][b, :, :P], full[0][b, :, :P])
        assert torch.equal(meta[1][b, :, :P], full[1][b, :, :P])


def test_hot_state_rejects_bad_use(dev, dkv):
    w = Workload("bad", B=1, Hq=4, Hkv=2, d=64, N=300, top_k=4)
    q, K, V = (t.to(dev) for t in make_inputs(w, seed=64))
    meta = dkv.kv_meta_build(K)
    hot = dkv.hot_state(w.B, w.Hkv, w.N, dev)
    with pytest.raises(dkv.DkvError) as e:
        dkv.decode_attn_select(q, K, V, meta, w.top_k, hot=hot, step=0)  # steps start at 1
    assert e.value.status == 2
    with pytest.raises(dkv.DkvError) as e:
        dkv.decode_attn_select(q, K, V, meta, w.top_k, hot=hot[:64], step=1)  # too small
    assert e.value.status == 6
    with pytest.raises(ValueError, match="16-bit metadata"):
        dkv.decode_attn_select(q, K, V, dkv.kv_meta8_build(meta), w.top_k, hot=hot, step=1)

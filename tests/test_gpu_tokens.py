"""Token-level sparse attention (each query head's top-K tokens by the exact
score q . k, attention over them only), against the oracle: the exact scores
are the bound score over single-token pages (m = M = k), the selection is
checked within the band, and the output against the oracle's attention over
the tokens the GPU chose."""

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
    Workload("tok-gqa", B=2, Hq=8, Hkv=2, d=128, N=5000, top_k=500),
    Workload("tok-mha-d64-fp16", B=2, Hq=4, Hkv=4, d=64, N=3001, top_k=300, dtype="fp16"),
    # 45000 keys per row: more than the top-K keeps in shared memory
    Workload("tok-long", B=1, Hq=4, Hkv=1, d=128, N=45000, top_k=4500, kind="offset"),
    # 192 rows of 5000 keys: the top-K reads its keys from the score rows
    Workload("tok-many-rows", B=4, Hq=48, Hkv=8, d=64, N=5000, top_k=500),
]


def _is16(w):
    return int(w.dtype == "fp16")


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_token_topk_matches_oracle(w, dev, dkv):
    q, K, V = make_inputs(w, seed=81)
    scale = 1.0 / math.sqrt(w.d)
    out, sel = dkv.decode_attn_topk_tokens(q.to(dev), K.to(dev), V.to(dev), w.top_k,
                                           return_selected=True)
    sel = sel.cpu().numpy()
    qb, Kb, Vb = bits(q), bits(K), bits(V)
    km, kx = oracle.meta(Kb, 1, _is16(w))
    assert np.array_equal(km, kx)  # single-token pages: m = M = k
    r = oracle.scores(qb, km, kx, _is16(w))  # exactly q . k_t
    check_selection(sel.reshape(-1, sel.shape[-1]), r.reshape(-1, w.N), w.top_k)
    ref = oracle.attention(qb, Kb, Vb, 1, scale, _is16(w), sel=sel)
    assert max_abs(out, ref) <= ATOL


def test_token_topk_all_tokens_equals_full(dev, dkv):
    w = CASES[0]
    q, K, V = (x.to(dev) for x in make_inputs(w, seed=83))
    out = dkv.decode_attn_topk_tokens(q, K, V, w.N + 7)
    full = dkv.decode_attn_full(q, K, V)
    assert max_abs(out, full.double().cpu().numpy()) <= 1e-5


@pytest.mark.parametrize("shape", [(1, 4, 1), (4, 48, 8)], ids=["4-rows", "192-rows"])
def test_token_topk_exact_ties_take_lower_tokens(shape, dev, dkv):
    """K repeats with period 8, so the scores fall into 8 exactly tied classes
    (identical rows give identical scores on both sides): the top-K is the
    best classes whole and the lowest-index tokens of the class at the K-th
    place, the same set as the oracle's (rows staged in shared memory, and
    rows read from the score rows)."""
    B, Hq, Hkv = shape
    w = Workload("tok-ties", B=B, Hq=Hq, Hkv=Hkv, d=128, N=6000, top_k=1000)
    q, K, V = make_inputs(w, seed=85)
    K = K[:, :, :8].repeat(1, 1, w.N // 8, 1).contiguous()
    out, sel = dkv.decode_attn_topk_tokens(q.to(dev), K.to(dev), V.to(dev), w.top_k,
                                           return_selected=True)
    sel = sel.cpu().numpy()
    qb, Kb, Vb = bits(q), bits(K), bits(V)
    km, kx = oracle.meta(Kb, 1, 0)
    r = oracle.scores(qb, km, kx, 0).reshape(-1, w.N)
    rows = sel.reshape(-1, sel.shape[-1])
    for i in range(r.shape[0]):
        order = sorted(range(w.N), key=lambda j: (-r[i, j], j))
        assert rows[i].tolist() == sorted(order[:w.top_k]), f"row {i}"
    ref = oracle.attention(qb, Kb, Vb, 1, 1.0 / math.sqrt(w.d), 0, sel=sel)
    assert max_abs(out, ref) <= ATOL

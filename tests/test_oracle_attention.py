"""Pins for the oracle's decode attention (exact and page-sparse).

Definitions: HeadInfer ("论文阅读：HeadInfer", 核心 idea) -- per-head
Softmax(q K^T / sqrt(d_k)) V, heads independent, head-by-head identical to all
heads; TinyServe ("TinyServe: ...", 问题公式化定义 / Algorithm 1) -- the same
softmax-weighted sum restricted to the tokens of the selected pages.
Checks: an fp64 library routine (torch scaled_dot_product_attention on CPU),
closed forms, invariances and bounds.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from workloads import Workload, bits, from_bits, make_inputs


def _sdpa(q, K, V, scale):
    """fp64 torch SDPA with the kv heads repeated for GQA."""
    B, Hq, d = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    Kx = K.double().repeat_interleave(G, dim=1)
    Vx = V.double().repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(
        q.double().unsqueeze(2), Kx, Vx, scale=scale)
    return o.squeeze(2).numpy()


@pytest.mark.parametrize("w", [
    Workload("t", B=1, Hq=16, Hkv=16, d=64, N=1024),
    Workload("t", B=2, Hq=8, Hkv=2, d=128, N=1000),
    Workload("t", B=3, Hq=4, Hkv=1, d=64, N=1),
    Workload("t", B=2, Hq=6, Hkv=3, d=128, N=257, dtype="fp16"),
])
def test_full_matches_torch_sdpa_fp64(w):
    q, K, V = make_inputs(w, seed=w.N)
    is16 = int(w.dtype == "fp16")
    scale = 1.0 / math.sqrt(w.d)
    got = oracle.attention(bits(q), bits(K), bits(V), 16, scale, is16)
    ref = _sdpa(q, K, V, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    # another softmax scale (TinyServe prints softmax(q^T k) without 1/sqrt(d))
    got1 = oracle.attention(bits(q), bits(K), bits(V), 16, 1.0, is16)
    np.testing.assert_allclose(got1, _sdpa(q, K, V, 1.0), rtol=0, atol=1e-11)


def test_single_token_returns_its_value():
    w = Workload("t", B=2, Hq=4, Hkv=2, d=64, N=1)
    q, K, V = make_inputs(w, seed=1)
    got = oracle.attention(bits(q), bits(K), bits(V), 16, 0.125, 0)
    for h in range(4):
        assert np.array_equal(got[:, h], V[:, h // 2, 0].double().numpy())


def test_equal_keys_give_mean_value():
    w = Workload("t", B=1, Hq=2, Hkv=1, d=64, N=100)
    q, K, V = make_inputs(w, seed=2)
    K[:] = K[:, :, :1, :]
    got = oracle.attention(bits(q), bits(K), bits(V), 16, 0.125, 0)
    np.testing.assert_allclose(got[0, 0], V[0, 0].double().mean(0).numpy(), atol=1e-14)
    # q = 0 also gives the mean, whatever the keys
    q0 = torch.zeros_like(q)
    _, K2, _ = make_inputs(w, seed=3)
    got0 = oracle.attention(bits(q0), bits(K2), bits(V), 16, 0.125, 0)
    np.testing.assert_allclose(got0[0, 1], V[0, 0].double().mean(0).numpy(), atol=1e-14)


def test_dominant_key_selects_its_value():
    w = Workload("t", B=1, Hq=1, Hkv=1, d=64, N=50)
    q, K, V = make_inputs(w, seed=4)
    q[:] = 1.0
    K[0, 0, 17] = 4.0  # q.k_17 = 256 dominates every other score by far
    got = oracle.attention(bits(q), bits(K), bits(V), 16, 1.0, 0)
    np.testing.assert_allclose(got[0, 0], V[0, 0, 17].double().numpy(), atol=1e-12)


def test_shift_invariance():
    # Adding one vector c to every key shifts all scores by q.c: softmax and
    # output are unchanged.  Integer-valued keys keep K + c exact in bf16.
    g = torch.Generator().manual_seed(5)
    q = torch.randint(-3, 4, (1, 2, 64), generator=g).to(torch.bfloat16)
    K = torch.randint(-3, 4, (1, 1, 40, 64), generator=g).to(torch.bfloat16)
    V = torch.randn(1, 1, 40, 64, generator=g).to(torch.bfloat16)
    c = torch.randint(-5, 6, (64,), generator=g).to(torch.bfloat16)
    o1 = oracle.attention(bits(q), bits(K), bits(V), 16, 0.1, 0)
    o2 = oracle.attention(bits(q), bits(K + c), bits(V), 16, 0.1, 0)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_output_is_convex_combination():
    w = Workload("t", B=2, Hq=4, Hkv=4, d=64, N=333)
    q, K, V = make_inputs(w, seed=6)
    o = oracle.attention(bits(q), bits(K), bits(V), 16, 0.125, 0)
    Vd = V.double().numpy()
    assert np.all(o <= Vd.max(axis=2) + 1e-12)
    assert np.all(o >= Vd.min(axis=2) - 1e-12)


def test_headwise_equals_all_heads_bitwise():
    # HeadInfer: evaluating one kv head (and its q-head group) at a time gives
    # exactly the all-heads result.
    w = Workload("t", B=2, Hq=8, Hkv=4, d=128, N=300)
    q, K, V = make_inputs(w, seed=7)
    full = oracle.attention(bits(q), bits(K), bits(V), 16, 1 / math.sqrt(128), 0)
    for h in range(w.Hkv):
        part = oracle.attention(bits(q[:, 2 * h:2 * h + 2]), bits(K[:, h:h + 1]),
                                bits(V[:, h:h + 1]), 16, 1 / math.sqrt(128), 0)
        assert np.array_equal(part, full[:, 2 * h:2 * h + 2])


def test_select_all_pages_equals_full_bitwise():
    w = Workload("t", B=1, Hq=16, Hkv=16, d=64, N=1024)
    q, K, V = make_inputs(w, seed=42)
    qb, Kb, Vb = bits(q), bits(K), bits(V)
    full = oracle.attention(qb, Kb, Vb, 16, 0.125, 0)
    mn, mx = oracle.meta(Kb, 16, 0)
    sel = oracle.topk(oracle.scores(qb, mn, mx, 0), 64)
    assert np.array_equal(sel[0, 0], np.arange(64))
    sp = oracle.attention(qb, Kb, Vb, 16, 0.125, 0, sel=sel)
    assert np.array_equal(sp, full)


def test_select_equals_full_attention_over_gathered_tokens():
    # Sparse attention over S_t is ordinary attention over the concatenated
    # tokens of the selected pages (softmax normalised over those tokens).
    w = Workload("t", B=1, Hq=2, Hkv=1, d=64, N=200)
    q, K, V = make_inputs(w, seed=8)
    sel = np.array([[[1, 4, 12], [0, 5, 12]]], np.int32)  # page 12 is ragged (8 tokens)
    sp = oracle.attention(bits(q), bits(K), bits(V), 16, 0.125, 0, sel=sel)
    for h in range(2):
        toks = [t for j in sel[0, h] for t in range(16 * j, min(200, 16 * j + 16))]
        Kg, Vg = K[:, :, toks], V[:, :, toks]
        ref = oracle.attention(bits(q[:, h:h + 1]), bits(Kg), bits(Vg), 16, 0.125, 0)
        assert np.array_equal(sp[:, h], ref[:, 0])
        np.testing.assert_allclose(sp[:, h], _sdpa(q[:, h:h + 1], Kg, Vg, 0.125)[:, 0],
                                   atol=1e-12)

"""Paged caches: K and V held as a pool of 16-token pages (blocks) addressed
through a block table.  Every call must give bitwise the result of the
contiguous cache holding the same tokens (the same per-page arithmetic in the
same order), and match the oracle.  The pool's blocks are shuffled, the pool
has spare blocks, the table has spare columns, and every token slot past N is
NaN, so a read of the wrong block or of an unused slot shows up.
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


def to_paged(X, P, seed, spare_blocks=7, spare_cols=5):
    """[B, Hkv, N, d] -> (pool [nb, Hkv, 16, d], block table [B, P + spare_cols])."""
    B, H, N, d = X.shape
    nb = B * P + spare_blocks
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(nb, generator=g)[:B * P]
    bt = torch.full((B, P + spare_cols), -1, dtype=torch.int32)
    bt[:, :P] = order.view(B, P).to(torch.int32)
    pool = torch.full((nb, H, 16, d), float("nan"), dtype=X.dtype)
    Xp = torch.full((B, H, P * 16, d), float("nan"), dtype=X.dtype)
    Xp[:, :, :N] = X
    pool[order] = Xp.view(B, H, P, 16, d).permute(0, 2, 1, 3, 4).reshape(B * P, H, 16, d)
    return pool, bt


CASES = [
    Workload("paged-gqa-ragged", B=2, Hq=8, Hkv=2, d=128, N=5000, top_k=24, kind="hot"),
    Workload("paged-mha-d64-fp16", B=3, Hq=4, Hkv=4, d=64, N=1030, top_k=8, dtype="fp16"),
    # 1250 pages: the per-unit selection kernel
    Workload("paged-unit-select", B=1, Hq=8, Hkv=2, d=128, N=20000, top_k=50, kind="hot"),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_paged_equals_contiguous_bitwise(w, dev, dkv):
    q, K, V = make_inputs(w, seed=51)
    pk, bt = to_paged(K, w.P, seed=1)
    pv, _ = to_paged(V, w.P, seed=1)
    qd, Kd, Vd = q.to(dev), K.to(dev), V.to(dev)
    btd = bt.to(dev)
    PK = dkv.PagedCache(pk.to(dev), btd, w.N)
    PV = dkv.PagedCache(pv.to(dev), btd, w.N)
    mc, mp = dkv.kv_meta_build(Kd), dkv.kv_meta_build(PK)
    assert torch.equal(mc[0], mp[0]) and torch.equal(mc[1], mp[1])
    oc = dkv.decode_attn_full(qd, Kd, Vd)
    op = dkv.decode_attn_full(qd, PK, PV)
    assert torch.isfinite(op).all()
    assert torch.equal(oc, op)
    sc_out, sc_sel = dkv.decode_attn_select(qd, Kd, Vd, mc, w.top_k, return_selected=True)
    sp_out, sp_sel = dkv.decode_attn_select(qd, PK, PV, mp, w.top_k, return_selected=True)
    assert torch.equal(sc_sel, sp_sel)
    assert torch.equal(sc_out, sp_out)


def test_paged_matches_oracle(dev, dkv):
    w = CASES[0]
    q, K, V = make_inputs(w, seed=53)
    pk, bt = to_paged(K, w.P, seed=2)
    pv, _ = to_paged(V, w.P, seed=2)
    btd = bt.to(dev)
    PK = dkv.PagedCache(pk.to(dev), btd, w.N)
    PV = dkv.PagedCache(pv.to(dev), btd, w.N)
    qd = q.to(dev)
    scale = 1.0 / math.sqrt(w.d)
    out = dkv.decode_attn_full(qd, PK, PV)
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, scale, 0)
    assert max_abs(out, ref) <= ATOL
    meta = dkv.kv_meta_build(PK)
    omn, omx = oracle.meta(bits(K), w.S, 0)
    assert np.array_equal(meta[0].cpu().view(torch.int16).numpy().view(np.uint16), omn)
    assert np.array_equal(meta[1].cpu().view(torch.int16).numpy().view(np.uint16), omx)
    out, sel = dkv.decode_attn_select(qd, PK, PV, meta, w.top_k, return_selected=True)
    sel = sel.cpu().numpy()
    r = oracle.scores(bits(q), omn, omx, 0)
    check_selection(sel.reshape(-1, sel.shape[-1]), r.reshape(-1, r.shape[-1]), w.top_k)
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, scale, 0, sel=sel)
    assert max_abs(out, ref) <= ATOL


@pytest.mark.parametrize("bad", [-5, 10 ** 6])
def test_out_of_range_block_entry_is_reported(bad, dev, dkv):
    # A block-table entry outside [0, num_blocks) is clamped into the pool
    # before any copy is issued (nothing outside the pool is read) and
    # reported as DKV_ERR_DEVICE_CHECK in the workspace status word; the
    # sequences whose tables are valid are unaffected.
    w = Workload("paged-bad", B=2, Hq=8, Hkv=2, d=128, N=700, top_k=44)  # 44 pages: all
    q, K, V = make_inputs(w, seed=57)
    pk, bt = to_paged(K, w.P, seed=3)
    pv, _ = to_paged(V, w.P, seed=3)
    btd = bt.to(dev)  # K and V share one table
    PK = dkv.PagedCache(pk.to(dev), btd, w.N)
    PV = dkv.PagedCache(pv.to(dev), btd, w.N)
    qd = q.to(dev)
    scale = 1.0 / math.sqrt(w.d)
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, scale, 0)
    ws = torch.zeros(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k), dtype=torch.uint8,
                     device=dev)
    meta = dkv.kv_meta_build(PK)
    dkv.decode_attn_full(qd, PK, PV, workspace=ws)
    assert dkv.read_device_status(ws) == dkv.DKV_OK  # a valid table
    bt_bad = bt.clone()
    bt_bad[1, 5] = bad
    btb = bt_bad.to(dev)
    PKb = dkv.PagedCache(PK.pool, btb, w.N)
    PVb = dkv.PagedCache(PV.pool, btb, w.N)
    out = dkv.decode_attn_full(qd, PKb, PVb, workspace=ws)
    assert dkv.read_device_status(ws) == dkv.DKV_ERR_DEVICE_CHECK
    assert max_abs(out[:1], ref[:1]) <= ATOL
    out_s = dkv.decode_attn_select(qd, PKb, PVb, meta, w.top_k, workspace=ws)
    assert dkv.read_device_status(ws) == dkv.DKV_ERR_DEVICE_CHECK
    assert max_abs(out_s[:1], ref[:1]) <= ATOL
    dkv.decode_attn_select(qd, PK, PV, meta, w.top_k, workspace=ws)
    assert dkv.read_device_status(ws) == dkv.DKV_OK

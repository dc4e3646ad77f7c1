"""Parity at the five workloads' full sizes, in the launch configuration the
benchmark times (inputs drawn on the GPU with the benchmark's seeds, the same
calls and default workspaces), checked on sampled (batch, kv head) units that
the oracle computes one by one: metadata and 4-bit codes bit-exact, selections
within the 1e-5 band, outputs within 2e-3.  The 1M-token workload also checks
that one kv head per call gives bitwise the all-heads output, and the 32K
GQA workload is checked once more over 8-bit page metadata.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ATOL, check_selection, max_abs, require_cuda
from workloads import WORKLOADS, bits, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


def _units(w, n):
    """About n (batch, kv head) units spread over the workload, first and last included."""
    total = w.B * w.Hkv
    picks = sorted({0, total - 1, *np.linspace(0, total - 1, n).astype(int).tolist()})
    return [(u // w.Hkv, u % w.Hkv) for u in picks]


def _head_slice(t, b, h, G):
    return t[b:b + 1, h * G:(h + 1) * G]


def _check_unit(w, b, h, q, Kb, Vb, is16, out_full=None, meta=None, out_sel=None, sel=None):
    """Kb, Vb: uint16 bits [1, 1, N, d] of unit (b, h) as the kernels read it."""
    G = w.G
    qs = bits(_head_slice(q, b, h, G).cpu())
    scale = 1.0 / math.sqrt(w.d)
    if out_full is not None:
        ref = oracle.attention(qs, Kb, Vb, w.S, scale, is16)
        err = max_abs(_head_slice(out_full, b, h, G), ref)
        assert err <= ATOL, (b, h, err)
    if out_sel is not None:
        mn, mx = oracle.meta(Kb, w.S, is16)
        assert np.array_equal(bits(meta[0][b:b + 1, h:h + 1].cpu()), mn)
        assert np.array_equal(bits(meta[1][b:b + 1, h:h + 1].cpu()), mx)
        r = oracle.scores(qs, mn, mx, is16)
        s = _head_slice(sel, b, h, G).cpu().numpy()
        check_selection(s.reshape(G, -1), r.reshape(G, -1), w.top_k)
        ref = oracle.attention(qs, Kb, Vb, w.S, scale, is16, sel=s)
        err = max_abs(_head_slice(out_sel, b, h, G), ref)
        assert err <= ATOL, (b, h, err)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_dense_workloads_full_size(idx, dev):
    import decode_attention_paged_kv_gb300 as dkv
    w = WORKLOADS[idx]
    q, K, V = make_inputs(w, seed=42 + idx, device=dev)
    meta = dkv.kv_meta_build(K)
    out_full = dkv.decode_attn_full(q, K, V)
    out_sel, sel = dkv.decode_attn_select(q, K, V, meta, w.top_k, return_selected=True)
    torch.cuda.synchronize()
    for b, h in _units(w, 4 if idx else w.B * w.Hkv):
        Kb = bits(K[b:b + 1, h:h + 1].cpu())
        Vb = bits(V[b:b + 1, h:h + 1].cpu())
        _check_unit(w, b, h, q, Kb, Vb, 0, out_full, meta, out_sel, sel)


def test_headwise_1m_full_size(dev):
    import decode_attention_paged_kv_gb300 as dkv
    w = WORKLOADS[3]
    q, K, V = make_inputs(w, seed=45, device=dev)
    out = dkv.decode_attn_full(q, K, V)
    out_hw = torch.empty_like(out)
    for h in range(w.Hkv):
        dkv.decode_attn_full(q[:, h * w.G:(h + 1) * w.G], K[:, h:h + 1], V[:, h:h + 1],
                             out=out_hw[:, h * w.G:(h + 1) * w.G])
    torch.cuda.synchronize()
    assert torch.equal(out, out_hw)
    for b, h in [(0, 0), (0, w.Hkv - 1)]:
        Kb = bits(K[b:b + 1, h:h + 1].cpu())
        Vb = bits(V[b:b + 1, h:h + 1].cpu())
        _check_unit(w, b, h, q, Kb, Vb, 0, out_full=out)


def test_q4_workload_full_size(dev):
    import decode_attention_paged_kv_gb300 as dkv
    w = WORKLOADS[4]
    q, K, V = make_inputs(w, seed=46, device=dev)
    K4, V4 = dkv.kv_quant4(K), dkv.kv_quant4(V)
    meta = dkv.kv_meta_build(K4)
    out_full = dkv.decode_attn_full(q, K4, V4)
    out_sel, sel = dkv.decode_attn_select(q, K4, V4, meta, w.top_k, return_selected=True)
    torch.cuda.synchronize()
    for b, h in _units(w, 4):
        # The oracle quantises the unit's fp16 rows itself; the GPU's codes and
        # group bounds must match bit for bit, and attention runs on the
        # oracle's dequantised values.
        planes = []
        for x, x4 in ((K, K4), (V, V4)):
            codes, gmin, gmax = oracle.quant4(bits(x[b:b + 1, h:h + 1].cpu()))
            assert np.array_equal(x4.codes[b:b + 1, h:h + 1].cpu().numpy(), codes)
            assert np.array_equal(bits(x4.gmin[b:b + 1, h:h + 1].cpu()), gmin)
            assert np.array_equal(bits(x4.gmax[b:b + 1, h:h + 1].cpu()), gmax)
            planes.append(oracle.dequant4(codes, gmin, gmax))
        _check_unit(w, b, h, q, planes[0], planes[1], 1, out_full, meta, out_sel, sel)


def test_meta8_select_full_size(dev):
    # the 32K-token GQA workload with 8-bit page metadata, as the benchmark's
    # meta8 leg runs it: codes, lo and step bit-exact on sampled units, the
    # selection within the band of the oracle's 8-bit scores, outputs vs the
    # oracle over the GPU's pages
    import decode_attention_paged_kv_gb300 as dkv
    w = WORKLOADS[2]
    q, K, V = make_inputs(w, seed=44, device=dev)
    m8 = dkv.kv_meta8_build(dkv.kv_meta_build(K))
    out, sel = dkv.decode_attn_select(q, K, V, m8, w.top_k, return_selected=True)
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(w.d)
    for b, h in _units(w, 4):
        Kb = bits(K[b:b + 1, h:h + 1].cpu())
        Vb = bits(V[b:b + 1, h:h + 1].cpu())
        qs = bits(_head_slice(q, b, h, w.G).cpu())
        mn, mx = oracle.meta(Kb, w.S, 0)
        cmin, cmax, lo, step = oracle.meta8(mn, mx, 0)
        assert np.array_equal(m8.code_min[b:b + 1, h:h + 1].cpu().numpy(), cmin)
        assert np.array_equal(m8.code_max[b:b + 1, h:h + 1].cpu().numpy(), cmax)
        assert np.array_equal(m8.lo[b:b + 1, h:h + 1].cpu().numpy().view(np.uint32),
                              lo.view(np.uint32))
        assert np.array_equal(m8.step[b:b + 1, h:h + 1].cpu().numpy().view(np.uint32),
                              step.view(np.uint32))
        r = oracle.scores8(qs, cmin, cmax, lo, step, 0)
        s = _head_slice(sel, b, h, w.G).cpu().numpy()
        check_selection(s.reshape(w.G, -1), r.reshape(w.G, -1), w.top_k)
        ref = oracle.attention(qs, Kb, Vb, w.S, scale, 0, sel=s)
        assert max_abs(_head_slice(out, b, h, w.G), ref) <= ATOL, (b, h)

"""GPU parity at sizes the oracle finishes in seconds: several tiles per call,
ragged tails, GQA and MHA, bf16 and fp16, strided views.

Bars: metadata and 4-bit codes / group min / max / dequantised values
bit-exact; attention outputs within 2e-3 max-abs (fp32 output); selections
identical to the oracle's top-K except inside the 1e-5 relative band around
the K-th score, and the sparse output compared with the oracle's attention
over the pages the GPU selected.
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
    Workload("c0", B=1, Hq=16, Hkv=16, d=64, N=1024, top_k=16),
    Workload("mha-ragged", B=2, Hq=4, Hkv=4, d=64, N=3001, top_k=40, kind="offset"),
    Workload("gqa-hot", B=2, Hq=8, Hkv=2, d=128, N=5000, top_k=24, kind="hot"),
    Workload("gqa8", B=1, Hq=16, Hkv=2, d=128, N=2100, top_k=10),
    Workload("gqa2-fp16", B=3, Hq=4, Hkv=2, d=64, N=777, top_k=7, dtype="fp16"),
    Workload("fp16-d128", B=1, Hq=8, Hkv=8, d=128, N=4096, top_k=33, dtype="fp16", kind="offset"),
    Workload("one-token", B=2, Hq=4, Hkv=1, d=128, N=1, top_k=3),
    Workload("one-page", B=1, Hq=2, Hkv=1, d=64, N=16, top_k=1),
    Workload("page+1", B=1, Hq=2, Hkv=2, d=128, N=17, top_k=1),
    Workload("long-chunks", B=1, Hq=4, Hkv=1, d=128, N=70000, top_k=64),
    # the largest context the per-unit selection kernel takes (2048 pages), and
    # one page more, where the separate selection kernels run
    Workload("unit-select-max-pages", B=1, Hq=4, Hkv=1, d=64, N=32768, top_k=100, kind="hot"),
    Workload("unit-select-max-pages+1", B=1, Hq=8, Hkv=2, d=128, N=32769, top_k=100, kind="hot"),
    # the per-unit selection kernel: 8 heads per group with a ragged last page;
    # one head per group in fp16; exact score ties at the threshold
    Workload("unit-select-gqa8", B=2, Hq=16, Hkv=2, d=128, N=20000, top_k=50, kind="hot"),
    Workload("unit-select-mha-fp16", B=3, Hq=3, Hkv=3, d=64, N=16400, top_k=200, dtype="fp16"),
    Workload("unit-select-ties", B=2, Hq=8, Hkv=2, d=64, N=16384, top_k=77, kind="coarse"),
    # exact score ties in the separate selection kernels (500 pages)
    Workload("kernels-ties", B=2, Hq=8, Hkv=2, d=64, N=8000, top_k=77, kind="coarse"),
    # more work items than persistent CTAs (2 per SM): every CTA streams
    # several items back to back, exact and sparse
    Workload("multi-item-gqa", B=16, Hq=16, Hkv=8, d=128, N=8192, top_k=48, kind="hot"),
    Workload("multi-item-mha", B=16, Hq=32, Hkv=32, d=64, N=4100, top_k=64, kind="offset"),
    # a union of 2400 pages (75 chunks per unit) chosen by the separate
    # selection kernels
    Workload("select-merge-kernel", B=1, Hq=4, Hkv=1, d=128, N=40000, top_k=600, kind="hot"),
    # one head per kv head past the per-unit kernel's 2048 pages: the block
    # top-K writes the union lists itself (as the warp top-K does for the
    # shorter one-head cases above)
    Workload("block-topk-mha", B=2, Hq=2, Hkv=2, d=64, N=40000, top_k=100, kind="offset"),
]


def _is16(w):
    return int(w.dtype == "fp16")


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_meta_bit_exact(w, dev, dkv):
    _, K, _ = make_inputs(w, seed=11)
    mn, mx = dkv.kv_meta_build(K.to(dev))
    omn, omx = oracle.meta(bits(K), w.S, _is16(w))
    assert np.array_equal(bits(mn.cpu()), omn)
    assert np.array_equal(bits(mx.cpu()), omx)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_full_matches_oracle(w, dev, dkv):
    q, K, V = make_inputs(w, seed=21)
    scale = 1.0 / math.sqrt(w.d)
    out = dkv.decode_attn_full(q.to(dev), K.to(dev), V.to(dev))
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, scale, _is16(w))
    assert max_abs(out, ref) <= ATOL


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_select_matches_oracle(w, dev, dkv):
    q, K, V = make_inputs(w, seed=31)
    scale = 1.0 / math.sqrt(w.d)
    qd, Kd, Vd = q.to(dev), K.to(dev), V.to(dev)
    meta = dkv.kv_meta_build(Kd)
    out, sel = dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, return_selected=True)
    sel = sel.cpu().numpy()
    omn, omx = oracle.meta(bits(K), w.S, _is16(w))
    r = oracle.scores(bits(q), omn, omx, _is16(w))
    check_selection(sel.reshape(-1, sel.shape[-1]), r.reshape(-1, r.shape[-1]), w.top_k)
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, scale, _is16(w), sel=sel)
    assert max_abs(out, ref) <= ATOL


# One selection per kv head group (summed bound scores): the per-unit selection
# kernel (1024-2048 pages) and the separate selection kernels (shorter and
# longer contexts), GQA 4 and 8, bf16 and fp16, ragged last pages.
GROUP_CASES = [
    Workload("group-unit-gqa4", B=2, Hq=8, Hkv=2, d=128, N=20000, top_k=50, kind="hot"),
    Workload("group-unit-gqa8-d64", B=1, Hq=16, Hkv=2, d=64, N=32768, top_k=100, kind="hot"),
    Workload("group-kernels-short", B=2, Hq=8, Hkv=2, d=128, N=5000, top_k=24, kind="hot"),
    Workload("group-kernels-long", B=1, Hq=4, Hkv=1, d=128, N=40000, top_k=300, kind="hot"),
    Workload("group-unit-fp16", B=3, Hq=4, Hkv=2, d=64, N=16400, top_k=40, dtype="fp16"),
]


@pytest.mark.parametrize("w", GROUP_CASES, ids=lambda w: w.name)
def test_group_select_matches_oracle(w, dev, dkv):
    q, K, V = make_inputs(w, seed=41)
    scale = 1.0 / math.sqrt(w.d)
    qd, Kd, Vd = q.to(dev), K.to(dev), V.to(dev)
    meta = dkv.kv_meta_build(Kd)
    out, sel = dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, return_selected=True,
                                      group_select=True)
    sel = sel.cpu().numpy()
    kk = sel.shape[-1]
    per_group = sel.reshape(w.B, w.Hkv, w.G, kk)
    assert np.array_equal(per_group, np.broadcast_to(per_group[:, :, :1], per_group.shape))
    omn, omx = oracle.meta(bits(K), w.S, _is16(w))
    rg = oracle.group_scores(bits(q), omn, omx, _is16(w))
    check_selection(per_group[:, :, 0].reshape(-1, kk), rg.reshape(-1, rg.shape[-1]), w.top_k)
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, scale, _is16(w), sel=sel)
    assert max_abs(out, ref) <= ATOL


def test_group_select_with_one_head_per_group_is_per_head_select(dev, dkv):
    w = Workload("mha", B=2, Hq=4, Hkv=4, d=128, N=20000, top_k=64, kind="offset")
    q, K, V = (x.to(dev) for x in make_inputs(w, seed=43))
    meta = dkv.kv_meta_build(K)
    o1, s1 = dkv.decode_attn_select(q, K, V, meta, w.top_k, return_selected=True)
    o2, s2 = dkv.decode_attn_select(q, K, V, meta, w.top_k, return_selected=True,
                                    group_select=True)
    assert torch.equal(s1, s2)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("w", CASES[:4], ids=lambda w: w.name)
def test_select_all_pages_equals_full(w, dev, dkv):
    q, K, V = make_inputs(w, seed=41)
    qd, Kd, Vd = q.to(dev), K.to(dev), V.to(dev)
    meta = dkv.kv_meta_build(Kd)
    out, sel = dkv.decode_attn_select(qd, Kd, Vd, meta, w.P + 5, return_selected=True)
    assert sel.shape[-1] == w.P
    assert torch.equal(sel.cpu(), torch.arange(w.P, dtype=torch.int32).expand_as(sel.cpu()))
    full = dkv.decode_attn_full(qd, Kd, Vd)
    assert max_abs(out, full) <= ATOL
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, 1 / math.sqrt(w.d), _is16(w))
    assert max_abs(out, ref) <= ATOL


def test_headwise_equals_all_heads_bitwise(dev, dkv):
    # One kv head at a time (HeadInfer) through strided views == the all-heads call.
    w = Workload("hw", B=2, Hq=8, Hkv=4, d=128, N=9000)
    q, K, V = (t.to(dev) for t in make_inputs(w, seed=51))
    full = dkv.decode_attn_full(q, K, V)
    for h in range(w.Hkv):
        part = dkv.decode_attn_full(q[:, 2 * h:2 * h + 2], K[:, h:h + 1], V[:, h:h + 1])
        assert torch.equal(part, full[:, 2 * h:2 * h + 2])


def test_workspace_reuse_across_calls(dev, dkv):
    # One zero-filled workspace serves calls of different shapes in a row: the
    # work counter returns to zero after every call.
    wa = Workload("wa", B=2, Hq=8, Hkv=2, d=128, N=40000, top_k=20, kind="hot")
    wb = Workload("wb", B=3, Hq=4, Hkv=4, d=64, N=3000, top_k=9)
    qa, Ka, Va = (t.to(dev) for t in make_inputs(wa, seed=3))
    qb, Kb, Vb = (t.to(dev) for t in make_inputs(wb, seed=4))
    n = max(dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, k)
            for w in (wa, wb) for k in (0, w.top_k))
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    ref_a = dkv.decode_attn_full(qa, Ka, Va)
    ma, mb = dkv.kv_meta_build(Ka), dkv.kv_meta_build(Kb)
    ref_sa = dkv.decode_attn_select(qa, Ka, Va, ma, wa.top_k)
    ref_sb = dkv.decode_attn_select(qb, Kb, Vb, mb, wb.top_k)
    for _ in range(2):
        assert torch.equal(dkv.decode_attn_full(qa, Ka, Va, workspace=ws), ref_a)
        assert torch.equal(dkv.decode_attn_select(qb, Kb, Vb, mb, wb.top_k, workspace=ws), ref_sb)
        assert torch.equal(dkv.decode_attn_select(qa, Ka, Va, ma, wa.top_k, workspace=ws), ref_sa)
    # the status word and the work and exit counters are back at zero
    assert int(ws[:256].sum().item()) == 0


def test_strided_query_and_output(dev, dkv):
    w = Workload("st", B=2, Hq=4, Hkv=2, d=64, N=600)
    q, K, V = make_inputs(w, seed=61)
    big_q = torch.zeros(2, 6, 64, dtype=q.dtype)
    big_q[:, 1:5] = q
    qd = big_q.to(dev)[:, 1:5]
    out_big = torch.full((2, 7, 64), float("nan"), device=dev)
    dkv.decode_attn_full(qd, K.to(dev), V.to(dev), out=out_big[:, 2:6])
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, 1 / 8, 0)
    assert max_abs(out_big[:, 2:6], ref) <= ATOL
    assert torch.isnan(out_big[:, :2]).all() and torch.isnan(out_big[:, 6:]).all()


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_half_outputs(out_dtype, dev, dkv):
    w = Workload("ho", B=2, Hq=8, Hkv=2, d=128, N=2000)
    q, K, V = make_inputs(w, seed=71)
    out = dkv.decode_attn_full(q.to(dev), K.to(dev), V.to(dev), out_dtype=out_dtype)
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, 1 / math.sqrt(128), 0)
    got = out.float().cpu().double().numpy()
    eps = 2.0 ** -9 if out_dtype == torch.bfloat16 else 2.0 ** -12
    assert np.all(np.abs(got - ref) <= ATOL + eps * np.abs(ref))


def test_custom_scale(dev, dkv):
    w = Workload("sc", B=1, Hq=4, Hkv=4, d=64, N=500)
    q, K, V = make_inputs(w, seed=81)
    out = dkv.decode_attn_full(q.to(dev), K.to(dev), V.to(dev), scale=0.02)
    ref = oracle.attention(bits(q), bits(K), bits(V), w.S, 0.02, 0)
    assert max_abs(out, ref) <= ATOL


def test_quant4_dequant4_bit_exact(dev, dkv):
    rng = np.random.default_rng(5)
    rows, d = 3000, 128
    x = rng.standard_normal((rows, d)) * np.exp2(rng.integers(-20, 12, (rows, 1)))
    x[0] = 0.0
    x[1] = -0.0
    x[1, 7] = 0.0
    x[2] = 1.5
    x[3, :64] = np.arange(64)
    x[4] = np.clip(rng.standard_normal(d) * 4e4, -65504, 65504)  # finite, near the fp16 max
    # exact half-way quotients: step = 1 (min 0, max 15), values k + 1/2 round
    # to even; and steps that are fp16 subnormals
    x[5, :64] = np.concatenate([[0.0, 15.0], np.arange(31) * 0.5, np.arange(31) * 0.5 + 0.25])
    x[5, 64:] = np.concatenate([[-3.0, 12.0], np.arange(62) * 0.5 - 3.0])
    x[6] = rng.integers(0, 16, d) * 2.0 ** -24  # a subnormal grid
    x[7] = rng.standard_normal(d) * 2.0 ** -20
    # narrow groups (range below 451 * 2^-24: the fp32 step grid), from the
    # subnormals up to where fp16 spacing passes the threshold, and around it
    u = 2.0 ** -24
    r = 8
    for base in [0.0, 2.0 ** -14, 2.0 ** -13 - 100 * u, 2.0 ** -10, -2.0 ** -7, 2.0 ** -6]:
        for k in [1, 2, 7, 14, 15, 16, 29, 31, 100, 255, 300, 449, 450, 451, 452, 600, 2000]:
            for sign in (1.0, -1.0):
                x[r] = sign * (base + rng.integers(0, k + 1, d) * u)
                r += 1
    for k in range(1, 200):  # straddling zero
        x[r] = (rng.integers(0, k + 1, d) - k // 2) * u
        r += 1
    assert r < rows
    xb = np.asarray(x, np.float64).astype(np.float16).view(np.uint16)
    xt = torch.from_numpy(xb.view(np.int16)).view(torch.float16)
    q4 = dkv.kv_quant4(xt.to(dev))
    codes, gmin, gmax = oracle.quant4(xb)
    assert np.array_equal(q4.codes.cpu().numpy(), codes)
    assert np.array_equal(bits(q4.gmin.cpu()), gmin)
    assert np.array_equal(bits(q4.gmax.cpu()), gmax)
    xh = dkv.kv_dequant4(q4)
    assert np.array_equal(bits(xh.cpu()), oracle.dequant4(codes, gmin, gmax))


def test_q4_meta_bit_exact(dev, dkv):
    w = Workload("q4m", B=2, Hq=3, Hkv=3, d=128, N=1000, dtype="fp16")
    _, K, _ = make_inputs(w, seed=91)
    q4 = dkv.kv_quant4(K.to(dev).contiguous())
    mn, mx = dkv.kv_meta_build(q4)
    codes, gmin, gmax = oracle.quant4(bits(K))
    kh = oracle.dequant4(codes, gmin, gmax)
    omn, omx = oracle.meta(kh, w.S, 1)
    assert np.array_equal(bits(mn.cpu()), omn)
    assert np.array_equal(bits(mx.cpu()), omx)


@pytest.mark.parametrize("S", [4, 8, 16, 32, 64])
@pytest.mark.parametrize("d", [64, 128])
def test_q4_meta_page_sizes_lengths_and_append(S, d, dev, dkv):
    # Metadata of a 4-bit cache for every page size, sequences of different
    # lengths (ragged last pages, one shorter than a page) and rows of narrow
    # groups (the fp32 step, some straddling zero) in two of the sequences, so
    # that pages take both the fp16 min / max and the key path; then each
    # sequence's last page rebuilt alone (kv_meta_append) over a spoiled copy.
    w = Workload(f"q4m-s{S}", B=3, Hq=2, Hkv=2, d=d, N=1000, dtype="fp16")
    _, K, _ = make_inputs(w, seed=97 + S + d)
    g = torch.Generator().manual_seed(S + d)
    u = 2.0 ** -24
    for b in (0, 2):
        for h in range(w.Hkv):
            rows = torch.randint(0, w.N, (12,), generator=g)
            span = torch.randint(1, 400, (12, 1), generator=g).float()
            base = torch.randint(-300, 300, (12, 1), generator=g).float()
            K[b, h, rows] = ((base + torch.floor(torch.rand(12, w.d, generator=g) * span)) * u).to(K.dtype)
    lens = [1000, 3, 517]
    L = torch.tensor(lens, dtype=torch.int32, device=dev)
    q4 = dkv.kv_quant4(K.to(dev).contiguous())
    meta = dkv.kv_meta_build(q4, page_size=S, seq_lens=L)
    kh = oracle.dequant4(*oracle.quant4(bits(K)))
    want = []
    for b, n in enumerate(lens):
        P = (n + S - 1) // S
        omn, omx = oracle.meta(kh[b:b + 1, :, :n], S, 1)
        assert np.array_equal(bits(meta[0][b:b + 1, :, :P].cpu()), omn), f"min, sequence {b}"
        assert np.array_equal(bits(meta[1][b:b + 1, :, :P].cpu()), omx), f"max, sequence {b}"
        want.append((P, omn, omx))
    spoiled = tuple(m.clone() for m in meta)
    for b, n in enumerate(lens):
        last = (n - 1) // S
        for m in spoiled:
            m[b, :, last] = 7.0
    dkv.kv_meta_append(q4, spoiled, page_size=S, seq_lens=L)
    for b, (P, omn, omx) in enumerate(want):
        assert np.array_equal(bits(spoiled[0][b:b + 1, :, :P].cpu()), omn), f"append min {b}"
        assert np.array_equal(bits(spoiled[1][b:b + 1, :, :P].cpu()), omx), f"append max {b}"


# 4-bit caches: contiguous group bounds need N * d / 64 to be a multiple of 8
# (16-byte head strides); every case still ends in a ragged page.
Q4_CASES = [
    Workload("q4-mha", B=3, Hq=8, Hkv=8, d=128, N=2000, top_k=20, dtype="fp16"),
    Workload("q4-gqa-d64", B=2, Hq=8, Hkv=2, d=64, N=1000, top_k=9, dtype="fp16", kind="offset"),
    Workload("q4-ragged", B=1, Hq=4, Hkv=1, d=128, N=36, top_k=2, dtype="fp16"),
    Workload("q4-multi-item", B=16, Hq=16, Hkv=16, d=128, N=2052, top_k=32, dtype="fp16"),
    Workload("q4-long-gqa", B=2, Hq=8, Hkv=2, d=128, N=16400, top_k=64, dtype="fp16"),
]


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("w", [Q4_CASES[0], Q4_CASES[1], Q4_CASES[4]],
                         ids=["one-chunk-mha", "one-chunk-gqa-d64", "merged-chunks"])
def test_q4_select_half_outputs_are_the_rounded_fp32_outputs(w, out_dtype, dev, dkv):
    # A unit whose union fits one work item writes out from the attention
    # kernel itself; longer unions go through the merge.  Either way a 16-bit
    # output is the fp32 result rounded to nearest.
    q, K, V = make_inputs(w, seed=203)
    K4, V4 = dkv.kv_quant4(K.to(dev)), dkv.kv_quant4(V.to(dev))
    qd = q.to(dev)
    meta = dkv.kv_meta_build(K4)
    o32 = dkv.decode_attn_select(qd, K4, V4, meta, w.top_k)
    o16 = dkv.decode_attn_select(qd, K4, V4, meta, w.top_k, out_dtype=out_dtype)
    assert o16.dtype == out_dtype and torch.equal(o16, o32.to(out_dtype))


@pytest.mark.parametrize("w", Q4_CASES, ids=lambda w: w.name)
def test_q4_attention_matches_oracle(w, dev, dkv):
    # Attention over 4-bit caches: the kernels dequantise in registers to the
    # same fp16 values as kv_dequant4; the oracle attends over its own
    # dequantised cache.
    q, K, V = make_inputs(w, seed=201)
    scale = 1.0 / math.sqrt(w.d)
    K4, V4 = dkv.kv_quant4(K.to(dev)), dkv.kv_quant4(V.to(dev))
    kh = oracle.dequant4(*oracle.quant4(bits(K)))
    vh = oracle.dequant4(*oracle.quant4(bits(V)))
    qd = q.to(dev)
    out = dkv.decode_attn_full(qd, K4, V4)
    ref = oracle.attention(bits(q), kh, vh, w.S, scale, 1)
    assert max_abs(out, ref) <= ATOL
    meta = dkv.kv_meta_build(K4)
    out_s, sel = dkv.decode_attn_select(qd, K4, V4, meta, w.top_k, return_selected=True)
    sel = sel.cpu().numpy()
    omn, omx = oracle.meta(kh, w.S, 1)
    r = oracle.scores(bits(q), omn, omx, 1)
    check_selection(sel.reshape(-1, sel.shape[-1]), r.reshape(-1, r.shape[-1]), w.top_k)
    ref_s = oracle.attention(bits(q), kh, vh, w.S, scale, 1, sel=sel)
    assert max_abs(out_s, ref_s) <= ATOL


def test_q4_attention_with_narrow_groups(dev, dkv):
    # Tokens whose groups are narrower than 451 * 2^-24 dequantise through the
    # fp32 step (the kernels' slower per-page path); the rest of each page stays
    # on the fp16 step.  The ragged last page (zeroed bounds) takes it too.
    w = Workload("q4-narrow", B=2, Hq=8, Hkv=4, d=128, N=520, top_k=12, dtype="fp16")
    q, K, V = make_inputs(w, seed=303)
    g = torch.Generator().manual_seed(9)
    for T in (K, V):
        rows = torch.randint(0, w.N, (w.B, w.Hkv, 60), generator=g)
        for b in range(w.B):
            for h in range(w.Hkv):
                scale = torch.exp2(-torch.randint(14, 26, (60, 1), generator=g).float())
                T[b, h, rows[b, h]] = (torch.randn(60, w.d, generator=g) * scale).to(T.dtype)
    scale = 1.0 / math.sqrt(w.d)
    K4, V4 = dkv.kv_quant4(K.to(dev)), dkv.kv_quant4(V.to(dev))
    codes, gmin, gmax = oracle.quant4(bits(K))
    assert np.array_equal(K4.codes.cpu().numpy(), codes)
    kh = oracle.dequant4(codes, gmin, gmax)
    vh = oracle.dequant4(*oracle.quant4(bits(V)))
    assert np.array_equal(bits(dkv.kv_dequant4(K4).cpu()), kh)
    qd = q.to(dev)
    out = dkv.decode_attn_full(qd, K4, V4)
    assert max_abs(out, oracle.attention(bits(q), kh, vh, w.S, scale, 1)) <= ATOL
    meta = dkv.kv_meta_build(K4)
    omn, omx = oracle.meta(kh, w.S, 1)
    assert np.array_equal(bits(meta[0].cpu()), omn) and np.array_equal(bits(meta[1].cpu()), omx)
    out_s, sel = dkv.decode_attn_select(qd, K4, V4, meta, w.top_k, return_selected=True)
    sel = sel.cpu().numpy()
    r = oracle.scores(bits(q), omn, omx, 1)
    check_selection(sel.reshape(-1, sel.shape[-1]), r.reshape(-1, r.shape[-1]), w.top_k)
    ref_s = oracle.attention(bits(q), kh, vh, w.S, scale, 1, sel=sel)
    assert max_abs(out_s, ref_s) <= ATOL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kind", ["bf16", "fp16", "q4"])
@pytest.mark.parametrize("sparse", [False, True])
def test_attention_kernels_keep_two_ctas_per_sm(d, kind, sparse):
    """The persistent attention grid is built for two resident CTAs per SM;
    a register count above 168 silently halves the bytes in flight."""
    require_cuda()
    import decode_attention_paged_kv_gb300 as dkv
    dt = torch.float16 if kind != "bf16" else torch.bfloat16
    assert dkv.attn_ctas_per_sm(d, dt, q4=kind == "q4", sparse=sparse) == 2

"""The C-ABI library loads, exports every symbol include/dkv.h declares, and
rejects bad arguments on the host -- before any CUDA call, so this runs
without a GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from decode_attention_paged_kv_gb300 import build as b
    b.build()
    import decode_attention_paged_kv_gb300 as dkv
    return dkv.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "dkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dkv_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "dkv_decode_attn_select" in names and len(names) >= 8
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    assert L.dkv_status_string(0) == b"ok"
    assert b"timeout" not in L.dkv_status_string(1)
    assert L.dkv_status_string(8).startswith(b"device")
    assert L.dkv_status_string(12345) == b"unknown status"


def _params(**kw):
    import decode_attention_paged_kv_gb300 as dkv
    p = dkv._Params()
    p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim, p.seq_len, p.page_size = 2, 8, 2, 128, 1000, 16
    p.q_stride_b, p.q_stride_h, p.o_stride_b, p.o_stride_h = 8 * 128, 128, 8 * 128, 128
    p.scale = 0.088
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_workspace_bytes_layout(L):
    p = _params()
    full = L.dkv_workspace_bytes(ctypes.byref(p), 0)
    sel = L.dkv_workspace_bytes(ctypes.byref(p), 8)
    # the header (status word, work counters), then
    # (m, l) and o for one chunk per row (ceil(63 / 64) = 1 chunk; 16 rows,
    # d = 128), each region 256-aligned
    header = 256
    assert full == header + 256 + 16 * 128 * 4
    assert sel > full
    assert L.dkv_workspace_bytes(ctypes.byref(_params(head_dim=96)), 0) == 0
    assert L.dkv_workspace_bytes(ctypes.byref(_params(num_q_heads=7)), 0) == 0
    assert L.dkv_workspace_bytes(ctypes.byref(_params(page_size=12)), 0) == 0
    assert L.dkv_workspace_bytes(ctypes.byref(_params(page_size=48)), 0) == 0
    # selection pages of 4, 8, 32 or 64 tokens: the exact path is unchanged
    for S in (4, 8, 32):
        assert L.dkv_workspace_bytes(ctypes.byref(_params(page_size=S)), 0) == full
    assert L.dkv_workspace_bytes(ctypes.byref(_params(page_size=64)), 8) > 0
    assert L.dkv_workspace_bytes(ctypes.byref(_params(page_size=4)), 8) > 0
    assert L.dkv_workspace_bytes(None, 0) == 0


def test_hot_state_bytes(L):
    # a 256-byte header (two u64 counters) and one u32 stamp per 16-token cache
    # page of every (batch entry, kv head), rounded up to 256 bytes
    p = _params()
    pages = -(-p.seq_len // 16)
    want = 256 + -(-(4 * p.batch * p.num_kv_heads * pages) // 256) * 256
    assert L.dkv_hot_state_bytes(ctypes.byref(p)) == want
    assert L.dkv_hot_state_bytes(ctypes.byref(_params(head_dim=96))) == 0


def test_host_validation_before_launch(L):
    import decode_attention_paged_kv_gb300 as dkv
    kv = dkv._KV()
    kv.format, kv.dtype, kv.data = 0, 0, 4096
    kv.stride_b, kv.stride_h = 2 * 1000 * 128, 1000 * 128
    p = _params()
    ws = ctypes.c_void_p(1 << 20)
    q = out = ctypes.c_void_p(1 << 16)
    f = L.dkv_decode_attn_full
    assert f(None, q, ctypes.byref(kv), ctypes.byref(kv), out, 2, ws, 1 << 20, None) == 1
    assert f(ctypes.byref(p), None, ctypes.byref(kv), ctypes.byref(kv), out, 2, ws, 1 << 20, None) == 1
    assert f(ctypes.byref(_params(head_dim=80)), q, ctypes.byref(kv), ctypes.byref(kv), out, 2,
             ws, 1 << 20, None) == 5
    assert f(ctypes.byref(_params(num_kv_heads=3)), q, ctypes.byref(kv), ctypes.byref(kv), out,
             2, ws, 1 << 20, None) == 2
    assert f(ctypes.byref(_params(num_q_heads=32, num_kv_heads=2)), q, ctypes.byref(kv),
             ctypes.byref(kv), out, 2, ws, 1 << 20, None) == 5
    assert f(ctypes.byref(p), ctypes.c_void_p((1 << 16) + 2), ctypes.byref(kv), ctypes.byref(kv),
             out, 2, ws, 1 << 20, None) == 3
    assert f(ctypes.byref(_params(q_stride_h=100)), q, ctypes.byref(kv), ctypes.byref(kv), out,
             2, ws, 1 << 20, None) == 3
    assert f(ctypes.byref(p), q, ctypes.byref(kv), ctypes.byref(kv), out, 2, ws, 16, None) == 6
    assert f(ctypes.byref(p), q, ctypes.byref(kv), ctypes.byref(kv), out, 2, None, 1 << 20, None) == 6
    assert f(ctypes.byref(p), q, ctypes.byref(kv), ctypes.byref(kv), out, 7, ws, 1 << 20, None) == 4
    bad = dkv._KV()
    bad.format, bad.dtype, bad.data = 0, 2, 4096  # fp32 cache
    assert f(ctypes.byref(p), q, ctypes.byref(bad), ctypes.byref(kv), out, 2, ws, 1 << 20, None) == 4
    assert f(ctypes.byref(_params(scale=0.0)), q, ctypes.byref(kv), ctypes.byref(kv), out, 2, ws,
             1 << 20, None) == 2
    s = L.dkv_decode_attn_select
    assert s(ctypes.byref(p), q, ctypes.byref(kv), ctypes.byref(kv), None, None, 0, out, 2, None,
             ws, 1 << 24, None) == 2
    assert s(ctypes.byref(p), q, ctypes.byref(kv), ctypes.byref(kv), None, None, 4, out, 2, None,
             ws, 1 << 24, None) == 1
    assert L.dkv_kv_quant4(10, 100, q, q, q, q, None) == 2
    assert L.dkv_kv_quant4(10, 128, None, q, q, q, None) == 1
    assert L.dkv_kv_dequant4(10, 128, ctypes.c_void_p(3), q, q, q, None) == 3
    assert L.dkv_kv_meta_build(ctypes.byref(p), ctypes.byref(kv), None, q, None) == 1
    assert L.dkv_read_device_status(None, None) == 1
    n = ctypes.c_int32(0)
    assert L.dkv_attn_ctas_per_sm(128, 0, 0, 0, None) == 1
    assert L.dkv_attn_ctas_per_sm(96, 0, 0, 0, ctypes.byref(n)) == 5
    assert L.dkv_attn_ctas_per_sm(128, 2, 0, 0, ctypes.byref(n)) == 5   # fp32 cache
    assert L.dkv_attn_ctas_per_sm(128, 0, 1, 0, ctypes.byref(n)) == 5   # bf16 4-bit cache


def test_struct_layout_matches_header(tmp_path):
    # The ctypes structs the binding marshals must have the header's offsets.
    import subprocess
    import decode_attention_paged_kv_gb300 as dkv
    fields = {"dkv_kv": [f for f, _ in dkv._KV._fields_],
              "dkv_params": [f for f, _ in dkv._Params._fields_]}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "dkv.h"', "int main(void) {"]
    for st, fs in fields.items():
        lines.append(f'  printf("{st} %zu\\n", sizeof({st}));')
        for f in fs:
            lines.append(f'  printf("{st}.{f} %zu\\n", offsetof({st}, {f}));')
    lines.append("  return 0;\n}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True)
    out = dict(l.split() for l in subprocess.run([str(exe)], check=True, capture_output=True,
                                                 text=True).stdout.splitlines())
    for st, cls in (("dkv_kv", dkv._KV), ("dkv_params", dkv._Params)):
        assert int(out[st]) == ctypes.sizeof(cls), st
        for f in fields[st]:
            assert int(out[f"{st}.{f}"]) == getattr(cls, f).offset, f"{st}.{f}"


def test_paged_cache_validation(L):
    import decode_attention_paged_kv_gb300 as dkv
    bt = (ctypes.c_int32 * 256)()

    def paged(**kw):
        kv = dkv._KV()
        kv.format, kv.dtype, kv.data = dkv.DKV_KV_PAGED, 0, 4096
        kv.stride_b, kv.stride_h = 2 * 16 * 128, 16 * 128
        kv.block_table, kv.block_table_stride, kv.num_blocks = ctypes.addressof(bt), 63, 200
        for k, v in kw.items():
            setattr(kv, k, v)
        return kv

    p = _params()
    ws = ctypes.c_void_p(1 << 20)
    q = out = ctypes.c_void_p(1 << 16)
    f = L.dkv_decode_attn_full
    mb = L.dkv_kv_meta_build
    k, v = paged(), paged()
    assert mb(ctypes.byref(p), ctypes.byref(paged(block_table=None)), q, q, None) == 1
    assert mb(ctypes.byref(p), ctypes.byref(paged(block_table=ctypes.addressof(bt) + 2)), q, q,
              None) == 3
    assert mb(ctypes.byref(p), ctypes.byref(paged(num_blocks=0)), q, q, None) == 2
    assert mb(ctypes.byref(p), ctypes.byref(paged(stride_h=16 * 128 + 4)), q, q, None) == 3
    assert mb(ctypes.byref(p), ctypes.byref(paged(dtype=2)), q, q, None) == 4
    # rows of the [B, P] block table may not overlap (P = 63 cache pages here)
    assert mb(ctypes.byref(p), ctypes.byref(paged(block_table_stride=62)), q, q, None) == 2
    # K and V must share one block table
    assert f(ctypes.byref(p), q, ctypes.byref(k), ctypes.byref(paged(block_table_stride=64)), out,
             2, ws, 1 << 20, None) == 2
    assert f(ctypes.byref(p), q, ctypes.byref(k), ctypes.byref(paged(num_blocks=199)), out, 2, ws,
             1 << 20, None) == 2
    dense = dkv._KV()
    dense.format, dense.dtype, dense.data = 0, 0, 4096
    dense.stride_b, dense.stride_h = 2 * 1000 * 128, 1000 * 128
    assert f(ctypes.byref(p), q, ctypes.byref(k), ctypes.byref(dense), out, 2, ws, 1 << 20,
             None) == 4


def test_token_topk_validation(L):
    import decode_attention_paged_kv_gb300 as dkv
    p = _params()
    ws = ctypes.c_void_p(1 << 20)
    q = out = ctypes.c_void_p(1 << 16)
    kv = dkv._KV()
    kv.format, kv.dtype, kv.data = 0, 0, 4096
    kv.stride_b, kv.stride_h = 2 * 1000 * 128, 1000 * 128  # contiguous [2, 2, 1000, 128]
    t = L.dkv_decode_attn_topk_tokens
    args = lambda k, v, top_k=100, size=1 << 30, pp=p: (
        ctypes.byref(pp), q, ctypes.byref(k), ctypes.byref(v), top_k, out, 2, None, ws, size, None)
    need = L.dkv_workspace_bytes_tokens(ctypes.byref(p), 100)
    assert need >= 256 + 16 * 1000 * 4 + 16 * 100 * 4
    assert L.dkv_workspace_bytes_tokens(ctypes.byref(p), 0) == 0
    assert t(*args(kv, kv, top_k=0)) == 2
    assert t(*args(kv, kv, size=need - 1)) == 6
    strided = dkv._KV()
    strided.format, strided.dtype, strided.data = 0, 0, 4096
    strided.stride_b, strided.stride_h = 2 * 1024 * 128, 1024 * 128  # not contiguous in N
    assert t(*args(strided, kv)) == 5
    q4 = dkv._KV()
    q4.format, q4.dtype, q4.data, q4.gmin, q4.gmax = 1, 1, 4096, 4096, 4096
    assert t(*args(q4, q4)) == 4
    lens = (ctypes.c_int32 * 2)(1000, 500)
    pl = _params(seq_lens=ctypes.addressof(lens))
    assert t(*args(kv, kv, pp=pl)) == 5

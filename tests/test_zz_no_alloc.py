"""dkv_decode_attn_full_noalloc: exact decode attention for callers that
cannot allocate device memory for the library (their allocator owns the whole
device budget, or their loop must never reach cudaMalloc).  It runs the same
kernels as dkv_decode_attn_full with a fixed scratch array inside the library
instead of a caller workspace.

Called here through the C ABI directly, twice in a row on different shapes
(the second call finds the first one's scratch contents).  Both entry points
run the same kernels with the same fixed chunking, so the results must be
bitwise equal; each is also checked against the CPU oracle within the parity
tolerance.  A call whose bounded waits are forced to expire must show it as
NaN in its output, and the call after it must be correct again.  This file is
collected last so that a stop at the first failure has run every other test
first; it also passes on its own in a fresh process.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ATOL, max_abs, require_cuda
from workloads import Workload, bits, make_inputs

pytestmark = pytest.mark.gpu


def _call_noalloc(dkv, q, K, V, out, flags=0):
    ks, B, H, N, d = dkv._kv_struct(K)
    vs = dkv._kv_struct(V)[0]
    p = dkv._params(q, B, H, N, d, out, 1.0 / math.sqrt(d))
    p.flags = flags
    fn = dkv.lib().dkv_decode_attn_full_noalloc
    fn.argtypes = [ctypes.POINTER(dkv._Params), ctypes.c_void_p, ctypes.POINTER(dkv._KV),
                   ctypes.POINTER(dkv._KV), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn(ctypes.byref(p), q.data_ptr(), ctypes.byref(ks), ctypes.byref(vs), out.data_ptr(),
              dkv.DKV_FP32, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice():
    dev = require_cuda()
    import decode_attention_paged_kv_gb300 as dkv
    shapes = [Workload("na1", B=4, Hq=32, Hkv=8, d=128, N=20000, kind="hot"),
              Workload("na2", B=3, Hq=8, Hkv=8, d=64, N=3001, kind="offset")]
    for i, w in enumerate(shapes):
        qc, Kc, Vc = make_inputs(w, seed=100 + i)
        q, K, V = qc.to(dev), Kc.to(dev), Vc.to(dev)
        ref = dkv.decode_attn_full(q, K, V)
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(dkv, q, K, V, out) == dkv.DKV_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        want = oracle.attention(bits(qc), bits(Kc), bits(Vc), w.S, 1.0 / math.sqrt(w.d),
                                0 if w.dtype == "bf16" else 1)
        assert max_abs(out, want) <= ATOL


def test_noalloc_device_error_shows_as_nan_then_recovers():
    dev = require_cuda()
    import decode_attention_paged_kv_gb300 as dkv
    w = Workload("na3", B=2, Hq=8, Hkv=2, d=128, N=4000)
    q, K, V = (t.to(dev) for t in make_inputs(w, seed=7))
    out = torch.zeros(w.B, w.Hq, w.d, device=dev)
    # every bounded wait gives up at once (no hang): the call still returns
    # DKV_OK, its output is all NaN
    assert _call_noalloc(dkv, q, K, V, out, flags=dkv.DKV_FLAG_FORCE_TIMEOUT) == dkv.DKV_OK
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    ref = dkv.decode_attn_full(q, K, V)
    out2 = torch.full_like(ref, float("nan"))
    assert _call_noalloc(dkv, q, K, V, out2) == dkv.DKV_OK
    torch.cuda.synchronize()
    assert torch.equal(out2, ref)


def test_noalloc_rejects_problems_beyond_its_scratch():
    dev = require_cuda()
    import decode_attention_paged_kv_gb300 as dkv
    # 64 x 32 query heads x 256 chunks of partials is far beyond 16 MiB; the
    # call must refuse before launching anything.
    w = Workload("big", B=64, Hq=32, Hkv=8, d=128, N=1 << 20)
    q = torch.zeros(w.B, w.Hq, w.d, dtype=torch.bfloat16, device=dev)
    out = torch.empty(w.B, w.Hq, w.d, device=dev)
    need = dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, 0)
    assert need > (16 << 20)
    ks = dkv._KV()  # never read: the size check comes first
    ks.format, ks.dtype, ks.data = 0, 0, q.data_ptr()
    ks.stride_b, ks.stride_h = w.Hkv * w.N * w.d, w.N * w.d
    p = dkv._params(q, w.B, w.Hkv, w.N, w.d, out, None)
    fn = dkv.lib().dkv_decode_attn_full_noalloc
    fn.argtypes = [ctypes.POINTER(dkv._Params), ctypes.c_void_p, ctypes.POINTER(dkv._KV),
                   ctypes.POINTER(dkv._KV), ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    st = fn(ctypes.byref(p), q.data_ptr(), ctypes.byref(ks), ctypes.byref(ks), out.data_ptr(),
            dkv.DKV_FP32, None)
    assert st == 6  # DKV_ERR_WORKSPACE: beyond the fixed scratch

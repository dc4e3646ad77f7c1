"""Failure paths on the GPU without faulting it: the forced-timeout hook makes
every bounded device wait give up at once, so the kernel records a timeout in
the workspace status word, drains the copies it issued and exits; the context
stays usable and the next call is correct.  Argument errors raise before any
launch."""

import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import ATOL, max_abs, require_cuda
from workloads import Workload, bits, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


def test_forced_timeout_reports_and_recovers(dev):
    import decode_attention_paged_kv_gb300 as dkv
    w = Workload("to", B=2, Hq=8, Hkv=2, d=128, N=40000, top_k=16)
    q, K, V = make_inputs(w, seed=7)
    qd, Kd, Vd = q.to(dev), K.to(dev), V.to(dev)
    n = dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, 0)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    dkv.decode_attn_full(qd, Kd, Vd, workspace=ws, flags=dkv.DKV_FLAG_FORCE_TIMEOUT)
    assert dkv.read_device_status(ws) == dkv.DKV_ERR_DEVICE_TIMEOUT
    assert dkv.read_device_status(ws) == dkv.DKV_OK  # reading clears it
    out = dkv.decode_attn_full(qd, Kd, Vd, workspace=ws)
    assert dkv.read_device_status(ws) == dkv.DKV_OK
    ref = oracle.attention(bits(q), bits(K), bits(V), 16, 1 / math.sqrt(128), 0)
    assert max_abs(out, ref) <= ATOL

    meta = dkv.kv_meta_build(Kd)
    n = dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, workspace=ws,
                           flags=dkv.DKV_FLAG_FORCE_TIMEOUT)
    assert dkv.read_device_status(ws) == dkv.DKV_ERR_DEVICE_TIMEOUT
    dkv.decode_attn_select(qd, Kd, Vd, meta, w.top_k, workspace=ws)
    assert dkv.read_device_status(ws) == dkv.DKV_OK


@pytest.mark.parametrize("N", [20000, 2000])
def test_forced_timeout_select_paths(N, dev):
    # 1250 pages: the per-(batch, kv head) selection kernel; 125 pages: the
    # score / top-K / union kernels.  Both report the timeout and recover.
    import decode_attention_paged_kv_gb300 as dkv
    w = Workload("to2", B=2, Hq=8, Hkv=2, d=128, N=N, top_k=16, kind="hot")
    q, K, V = (t.to(dev) for t in make_inputs(w, seed=8))
    meta = dkv.kv_meta_build(K)
    n = dkv.workspace_bytes(w.B, w.Hq, w.Hkv, w.d, w.N, w.top_k)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    dkv.decode_attn_select(q, K, V, meta, w.top_k, workspace=ws, flags=dkv.DKV_FLAG_FORCE_TIMEOUT)
    assert dkv.read_device_status(ws) == dkv.DKV_ERR_DEVICE_TIMEOUT
    good = dkv.decode_attn_select(q, K, V, meta, w.top_k, workspace=ws)
    assert dkv.read_device_status(ws) == dkv.DKV_OK
    ref = dkv.decode_attn_select(q, K, V, meta, w.top_k)
    assert torch.equal(good, ref)


def test_argument_errors_raise(dev):
    import decode_attention_paged_kv_gb300 as dkv
    q = torch.zeros(1, 4, 96, dtype=torch.bfloat16, device=dev)
    K = torch.zeros(1, 4, 32, 96, dtype=torch.bfloat16, device=dev)
    with pytest.raises(dkv.DkvError) as e:
        dkv.decode_attn_full(q, K, K)
    assert e.value.status == 5  # head_dim 96 unsupported
    q = torch.zeros(1, 6, 64, dtype=torch.bfloat16, device=dev)
    K = torch.zeros(1, 4, 32, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(dkv.DkvError) as e:
        dkv.decode_attn_full(q, K, K)
    assert e.value.status == 2  # 6 % 4 != 0
    with pytest.raises(dkv.DkvError):
        dkv.decode_attn_full(q[:, :4].float(), K.float(), K.float())

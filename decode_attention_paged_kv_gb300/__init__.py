"""Python binding of libdkv: GB300 decode attention over a paged KV cache.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/dkv.h``.  PyTorch provides the
device memory (outputs and workspace are allocated with torch) and the current
stream.  There is no fallback: if ``libdkv.so`` has not been built, or a call
returns an error status, the call raises.

Public calls (same names as the C ABI, without the ``dkv_`` prefix):
  kv_meta_build(K)                      -> (meta_min, meta_max)
  decode_attn_full(q, K, V)             -> out
  decode_attn_select(q, K, V, meta, k)  -> out (, selected)
  kv_quant4(x) / kv_dequant4(q4)
  workspace_bytes(...), read_device_status(workspace)
K and V are dense tensors [B, Hkv, N, d] (bf16 / fp16; any batch / head
strides, token stride d) or ``Q4Cache`` tuples in the 4-bit format.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import NamedTuple, Optional

import torch

from . import build as _build_mod

__all__ = [
    "Q4Cache", "PagedCache", "Meta8", "DkvError", "lib", "kv_meta_build", "kv_meta8_build",
    "kv_meta_append", "hot_state", "hot_stats", "decode_attn_full",
    "decode_attn_select", "decode_attn_topk_tokens", "kv_quant4", "kv_dequant4",
    "workspace_bytes", "workspace_bytes_tokens", "read_device_status", "status_string",
    "PAGE_SIZE", "DKV_FLAG_GROUP_SELECT",
]

PAGE_SIZE = 16

# enums of include/dkv.h
DKV_OK = 0
DKV_ERR_DEVICE_TIMEOUT = 8
DKV_ERR_DEVICE_CHECK = 9
DKV_BF16, DKV_FP16, DKV_FP32 = 0, 1, 2
DKV_KV_DENSE, DKV_KV_Q4G64, DKV_KV_PAGED = 0, 1, 2
DKV_FLAG_FORCE_TIMEOUT = 0x1
DKV_FLAG_GROUP_SELECT = 0x2


class DkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: dkv status {status} ({status_string(status)})")


class Q4Cache(NamedTuple):
    """A K or V cache in the 4-bit group-of-64 format.

    codes [B, Hkv, N, d/2] uint8 (channel 2i in the low nibble of byte i);
    gmin, gmax [B, Hkv, N, d/64] fp16 (per-group min / max).
    """
    codes: torch.Tensor
    gmin: torch.Tensor
    gmax: torch.Tensor


class Meta8(NamedTuple):
    """8-bit page metadata (kv_meta8_build): per page a grid
    dec(c) = fmaf(c, step, lo), and per channel the codes of m rounded down
    and of M rounded up on it.  code_min / code_max uint8 [B, Hkv, P, d];
    lo / step float32 [B, Hkv, P]."""
    code_min: torch.Tensor
    code_max: torch.Tensor
    lo: torch.Tensor
    step: torch.Tensor


class PagedCache(NamedTuple):
    """A K or V cache held as a pool of 16-token pages (blocks).

    pool [num_blocks, Hkv, 16, d] bf16 / fp16 (token and channel strides d, 1);
    block_table [B, P] int32: page j of batch entry b is pool block
    block_table[b, j]; seq_len: the N tokens every sequence attends.
    K and V passed to one call must share the block table.
    """
    pool: torch.Tensor
    block_table: torch.Tensor
    seq_len: int


class _Params(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("seq_len", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("q_stride_b", ctypes.c_int64), ("q_stride_h", ctypes.c_int64),
                ("o_stride_b", ctypes.c_int64), ("o_stride_h", ctypes.c_int64),
                ("scale", ctypes.c_float), ("flags", ctypes.c_uint32),
                ("seq_lens", ctypes.c_void_p)]


class _KV(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("data", ctypes.c_void_p), ("gmin", ctypes.c_void_p), ("gmax", ctypes.c_void_p),
                ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64),
                ("gstride_b", ctypes.c_int64), ("gstride_h", ctypes.c_int64),
                ("block_table", ctypes.c_void_p), ("block_table_stride", ctypes.c_int64),
                ("num_blocks", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded libdkv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build_mod.LIB
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libdkv.so not found at {path}; build it with "
                    "`python -m decode_attention_paged_kv_gb300.build`")
            L = ctypes.CDLL(path)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            P, KVp = ctypes.POINTER(_Params), ctypes.POINTER(_KV)
            L.dkv_workspace_bytes.argtypes = [P, i32]
            L.dkv_workspace_bytes.restype = sz
            L.dkv_kv_meta_build.argtypes = [P, KVp, vp, vp, vp]
            L.dkv_decode_attn_full.argtypes = [P, vp, KVp, KVp, vp, i32, vp, sz, vp]
            L.dkv_decode_attn_select.argtypes = [P, vp, KVp, KVp, vp, vp, i32, vp, i32, vp, vp,
                                                 sz, vp]
            L.dkv_decode_attn_topk_tokens.argtypes = [P, vp, KVp, KVp, i32, vp, i32, vp, vp,
                                                      sz, vp]
            L.dkv_kv_meta8_build.argtypes = [P, vp, vp, i32, vp, vp, vp, vp, vp]
            L.dkv_decode_attn_select_meta8.argtypes = [P, vp, KVp, KVp, vp, vp, vp, vp, i32,
                                                       vp, i32, vp, vp, sz, vp]
            L.dkv_workspace_bytes_tokens.argtypes = [P, i32]
            L.dkv_workspace_bytes_tokens.restype = sz
            L.dkv_kv_meta_append.argtypes = [P, KVp, vp, vp, vp]
            L.dkv_hot_state_bytes.argtypes = [P]
            L.dkv_hot_state_bytes.restype = sz
            L.dkv_decode_attn_select_hot.argtypes = [P, vp, KVp, KVp, vp, vp, i32, vp, i32, vp,
                                                     vp, sz, i32, vp, sz, vp]
            L.dkv_kv_quant4.argtypes = [i64, i32, vp, vp, vp, vp, vp]
            L.dkv_kv_dequant4.argtypes = [i64, i32, vp, vp, vp, vp, vp]
            L.dkv_read_device_status.argtypes = [vp, vp]
            L.dkv_attn_ctas_per_sm.argtypes = [i32, i32, i32, i32, ctypes.POINTER(i32)]
            L.dkv_status_string.argtypes = [i32]
            L.dkv_status_string.restype = ctypes.c_char_p
            for name in ("dkv_kv_meta_build", "dkv_decode_attn_full", "dkv_decode_attn_select",
                         "dkv_decode_attn_topk_tokens", "dkv_kv_meta8_build",
                         "dkv_decode_attn_select_meta8", "dkv_kv_meta_append",
                         "dkv_decode_attn_select_hot",
                         "dkv_kv_quant4", "dkv_kv_dequant4", "dkv_read_device_status",
                         "dkv_attn_ctas_per_sm"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().dkv_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != DKV_OK:
        raise DkvError(status, where)


def _stream(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return DKV_BF16
    if dt == torch.float16:
        return DKV_FP16
    if dt == torch.float32:
        return DKV_FP32
    raise TypeError(f"unsupported dtype {dt}")


def _kv_struct(kv) -> tuple[_KV, int, int, int, int]:
    """(struct, B, Hkv, N, d) for a dense tensor, a Q4Cache or a PagedCache."""
    s = _KV()
    if isinstance(kv, PagedCache):
        pool, bt, N = kv
        nb, H, S, d = pool.shape
        if S != PAGE_SIZE or pool.stride(3) != 1 or pool.stride(2) != d:
            raise ValueError("pool must be [num_blocks, Hkv, 16, d] with token stride d")
        if bt.dtype != torch.int32 or bt.dim() != 2 or bt.stride(1) != 1:
            raise ValueError("block_table must be int32 [B, P] with unit column stride")
        P = (int(N) + PAGE_SIZE - 1) // PAGE_SIZE
        if bt.shape[1] < P:
            raise ValueError("block_table has fewer than ceil(seq_len / 16) columns")
        s.format, s.dtype = DKV_KV_PAGED, _dtype_code(pool.dtype)
        s.data = pool.data_ptr()
        s.stride_b, s.stride_h = pool.stride(0), pool.stride(1)
        s.block_table, s.block_table_stride, s.num_blocks = bt.data_ptr(), bt.stride(0), nb
        return s, bt.shape[0], H, int(N), d
    if isinstance(kv, Q4Cache):
        c, gmn, gmx = kv
        B, H, N, half = c.shape
        d = half * 2
        if c.dtype != torch.uint8 or gmn.dtype != torch.float16 or gmx.dtype != torch.float16:
            raise TypeError("Q4Cache wants uint8 codes and fp16 gmin/gmax")
        if c.stride(3) != 1 or c.stride(2) != half:
            raise ValueError("codes must have token stride d/2 and channel stride 1")
        if gmn.stride() != gmx.stride() or gmn.stride(3) != 1 or gmn.stride(2) != d // 64:
            raise ValueError("gmin / gmax must share strides with token stride d/64")
        s.format, s.dtype = DKV_KV_Q4G64, DKV_FP16
        s.data, s.gmin, s.gmax = c.data_ptr(), gmn.data_ptr(), gmx.data_ptr()
        s.stride_b, s.stride_h = c.stride(0), c.stride(1)
        s.gstride_b, s.gstride_h = gmn.stride(0), gmn.stride(1)
        return s, B, H, N, d
    B, H, N, d = kv.shape
    if kv.stride(3) != 1 or kv.stride(2) != d:
        raise ValueError("K/V must have token stride d and channel stride 1")
    s.format, s.dtype = DKV_KV_DENSE, _dtype_code(kv.dtype)
    s.data = kv.data_ptr()
    s.stride_b, s.stride_h = kv.stride(0), kv.stride(1)
    return s, B, H, N, d


def _device_of(kv) -> torch.device:
    if isinstance(kv, Q4Cache):
        return kv.codes.device
    return kv.pool.device if isinstance(kv, PagedCache) else kv.device


def _params(q: Optional[torch.Tensor], B, Hkv, N, d, out: Optional[torch.Tensor],
            scale: Optional[float], flags: int = 0,
            seq_lens: Optional[torch.Tensor] = None) -> _Params:
    p = _Params()
    if seq_lens is not None:
        if (seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,) or not seq_lens.is_cuda
                or not seq_lens.is_contiguous()):
            raise ValueError("seq_lens must be a contiguous int32 CUDA tensor [B]")
        p.seq_lens = seq_lens.data_ptr()
    p.batch, p.num_kv_heads, p.head_dim, p.seq_len, p.page_size = B, Hkv, d, N, PAGE_SIZE
    p.num_q_heads = q.shape[1] if q is not None else Hkv
    if q is not None:
        if q.shape[0] != B or q.shape[2] != d or q.stride(2) != 1:
            raise ValueError(f"q shape {tuple(q.shape)} does not match the cache")
        p.q_stride_b, p.q_stride_h = q.stride(0), q.stride(1)
    if out is not None:
        p.o_stride_b, p.o_stride_h = out.stride(0), out.stride(1)
    p.scale = float(scale) if scale is not None else 1.0 / math.sqrt(d)
    p.flags = flags
    return p


def workspace_bytes(B: int, Hq: int, Hkv: int, d: int, N: int, top_k: int = 0,
                    page_size: int = PAGE_SIZE) -> int:
    """Workspace bytes dkv_decode_attn_full (top_k = 0) or _select needs."""
    p = _Params()
    p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim, p.seq_len = B, Hq, Hkv, d, N
    p.page_size, p.scale = page_size, 1.0
    n = lib().dkv_workspace_bytes(ctypes.byref(p), int(top_k))
    if n == 0:
        raise DkvError(2, "dkv_workspace_bytes")
    return int(n)


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def kv_meta_build(K, page_size: int = PAGE_SIZE, seq_lens: Optional[torch.Tensor] = None):
    """Page metadata (meta_min, meta_max), each [B, Hkv, P, d]."""
    ks, B, H, N, d = _kv_struct(K)
    dev = _device_of(K)
    dt = (torch.float16 if isinstance(K, Q4Cache)
          else K.pool.dtype if isinstance(K, PagedCache) else K.dtype)
    P = (N + page_size - 1) // page_size
    mn = torch.empty(B, H, P, d, dtype=dt, device=dev)
    mx = torch.empty(B, H, P, d, dtype=dt, device=dev)
    p = _params(None, B, H, N, d, None, None, seq_lens=seq_lens)
    p.page_size = page_size
    _check(lib().dkv_kv_meta_build(ctypes.byref(p), ctypes.byref(ks), mn.data_ptr(),
                                   mx.data_ptr(), _stream(mn)), "dkv_kv_meta_build")
    return mn, mx


def kv_meta_append(K, meta, page_size: int = PAGE_SIZE,
                   seq_lens: Optional[torch.Tensor] = None):
    """After a decode step appended tokens: rebuild, in place, only the page
    of `meta` (from kv_meta_build) holding each sequence's last token (N_b - 1,
    N_b from seq_lens, else the cache length)."""
    ks, B, H, N, d = _kv_struct(K)
    mn, mx = meta
    P = (N + page_size - 1) // page_size
    if tuple(mn.shape) != (B, H, P, d) or not mn.is_contiguous() or not mx.is_contiguous():
        raise ValueError("meta must be contiguous [B, Hkv, P, d]")
    p = _params(None, B, H, N, d, None, None, seq_lens=seq_lens)
    p.page_size = page_size
    _check(lib().dkv_kv_meta_append(ctypes.byref(p), ctypes.byref(ks), mn.data_ptr(),
                                    mx.data_ptr(), _stream(mn)), "dkv_kv_meta_append")
    return mn, mx


def hot_state(B: int, Hkv: int, N: int, device) -> torch.Tensor:
    """A zeroed cross-step reuse state for decode_attn_select(hot=..., step=...)
    on caches of B sequences, Hkv kv heads and N tokens."""
    p = _params(None, B, Hkv, N, 64, None, None)
    n = int(lib().dkv_hot_state_bytes(ctypes.byref(p)))
    if n == 0:
        raise ValueError("invalid shape for a reuse state")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def hot_stats(state: torch.Tensor) -> tuple[int, int]:
    """(cache pages gathered, of them gathered at the previous step too), summed
    over the calls since the state was zeroed."""
    h = state[:16].cpu().view(torch.int64)
    return int(h[0]), int(h[1])


def kv_meta8_build(meta, page_size: int = PAGE_SIZE,
                   seq_lens: Optional[torch.Tensor] = None) -> Meta8:
    """8-bit page metadata from (meta_min, meta_max) [B, Hkv, P, d] (bf16 or
    fp16, as kv_meta_build returns it)."""
    mn, mx = meta
    if mn.dtype not in (torch.bfloat16, torch.float16) or mx.dtype != mn.dtype:
        raise ValueError("meta must be bf16 or fp16")
    if not mn.is_contiguous() or not mx.is_contiguous() or mn.shape != mx.shape:
        raise ValueError("meta must be two contiguous [B, Hkv, P, d] tensors")
    B, H, P, d = mn.shape
    m8 = Meta8(torch.empty(B, H, P, d, dtype=torch.uint8, device=mn.device),
               torch.empty(B, H, P, d, dtype=torch.uint8, device=mn.device),
               torch.empty(B, H, P, dtype=torch.float32, device=mn.device),
               torch.empty(B, H, P, dtype=torch.float32, device=mn.device))
    # N only sets P here: the largest N with ceil(N / S) = P
    p = _params(None, B, H, P * page_size, d, None, None, seq_lens=seq_lens)
    p.page_size = page_size
    _check(lib().dkv_kv_meta8_build(ctypes.byref(p), mn.data_ptr(), mx.data_ptr(),
                                    _dtype_code(mn.dtype), m8.code_min.data_ptr(),
                                    m8.code_max.data_ptr(), m8.lo.data_ptr(),
                                    m8.step.data_ptr(), _stream(mn)), "dkv_kv_meta8_build")
    return m8


def decode_attn_full(q, K, V, scale: Optional[float] = None,
                     out_dtype: torch.dtype = torch.float32,
                     out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, flags: int = 0,
                     seq_lens: Optional[torch.Tensor] = None):
    """Exact decode attention; returns out [B, Hq, d] (seq_lens: int32 [B] on the
    device, tokens each sequence attends; None: all N)."""
    ks, B, H, N, d = _kv_struct(K)
    vs, B2, H2, N2, d2 = _kv_struct(V)
    if (B, H, N, d) != (B2, H2, N2, d2):
        raise ValueError("K and V shapes differ")
    if out is None:
        out = torch.empty(B, q.shape[1], d, dtype=out_dtype, device=q.device)
    p = _params(q, B, H, N, d, out, scale, flags, seq_lens)
    nbytes = lib().dkv_workspace_bytes(ctypes.byref(p), 0)
    ws = _workspace(nbytes, q.device, workspace)
    _check(lib().dkv_decode_attn_full(ctypes.byref(p), q.data_ptr(), ctypes.byref(ks),
                                      ctypes.byref(vs), out.data_ptr(), _dtype_code(out.dtype),
                                      ws.data_ptr(), nbytes, _stream(q)), "dkv_decode_attn_full")
    return out


def decode_attn_select(q, K, V, meta, top_k: int, scale: Optional[float] = None,
                       out_dtype: torch.dtype = torch.float32,
                       out: Optional[torch.Tensor] = None, return_selected: bool = False,
                       selected: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, flags: int = 0,
                       group_select: bool = False, seq_lens: Optional[torch.Tensor] = None,
                       page_size: int = PAGE_SIZE, hot: Optional[torch.Tensor] = None,
                       step: int = 0):
    """Query-aware page-sparse decode attention over the top_k pages per q-head
    (group_select: one selection per kv head group, by the summed bound scores;
    page_size: tokens per metadata / selection page, as meta was built with;
    meta: (meta_min, meta_max), or a Meta8 from kv_meta8_build; hot, step: one
    step (1, 2, ...) of a decode loop keeping hot pages in L2, with a state
    from hot_state())."""
    if group_select:
        flags |= DKV_FLAG_GROUP_SELECT
    ks, B, H, N, d = _kv_struct(K)
    vs, B2, H2, N2, d2 = _kv_struct(V)
    if (B, H, N, d) != (B2, H2, N2, d2):
        raise ValueError("K and V shapes differ")
    P = (N + page_size - 1) // page_size
    m8 = meta if isinstance(meta, Meta8) else None
    if m8 is not None and hot is not None:
        raise ValueError("cross-step reuse takes 16-bit metadata")
    if m8 is not None:
        if (tuple(m8.code_min.shape) != (B, H, P, d) or tuple(m8.lo.shape) != (B, H, P)
                or not all(t.is_contiguous() for t in m8)):
            raise ValueError("Meta8 must hold contiguous [B, Hkv, P, d] codes, [B, Hkv, P] grid")
    else:
        mn, mx = meta
        if tuple(mn.shape) != (B, H, P, d) or not mn.is_contiguous() or not mx.is_contiguous():
            raise ValueError("meta must be contiguous [B, Hkv, P, d]")
    if out is None:
        out = torch.empty(B, q.shape[1], d, dtype=out_dtype, device=q.device)
    kk = min(int(top_k), P)
    if return_selected and selected is None:
        selected = torch.empty(B, q.shape[1], kk, dtype=torch.int32, device=q.device)
    p = _params(q, B, H, N, d, out, scale, flags, seq_lens)
    p.page_size = page_size
    nbytes = lib().dkv_workspace_bytes(ctypes.byref(p), int(top_k))
    ws = _workspace(nbytes, q.device, workspace)
    sel_ptr = selected.data_ptr() if selected is not None else None
    if m8 is not None:
        _check(lib().dkv_decode_attn_select_meta8(
            ctypes.byref(p), q.data_ptr(), ctypes.byref(ks), ctypes.byref(vs),
            m8.code_min.data_ptr(), m8.code_max.data_ptr(), m8.lo.data_ptr(),
            m8.step.data_ptr(), int(top_k), out.data_ptr(), _dtype_code(out.dtype), sel_ptr,
            ws.data_ptr(), nbytes, _stream(q)), "dkv_decode_attn_select_meta8")
    elif hot is not None:
        _check(lib().dkv_decode_attn_select_hot(
            ctypes.byref(p), q.data_ptr(), ctypes.byref(ks), ctypes.byref(vs), mn.data_ptr(),
            mx.data_ptr(), int(top_k), out.data_ptr(), _dtype_code(out.dtype), sel_ptr,
            hot.data_ptr(), hot.numel(), int(step), ws.data_ptr(), nbytes, _stream(q)),
            "dkv_decode_attn_select_hot")
    else:
        _check(lib().dkv_decode_attn_select(ctypes.byref(p), q.data_ptr(), ctypes.byref(ks),
                                            ctypes.byref(vs), mn.data_ptr(), mx.data_ptr(),
                                            int(top_k), out.data_ptr(), _dtype_code(out.dtype),
                                            sel_ptr, ws.data_ptr(), nbytes, _stream(q)),
               "dkv_decode_attn_select")
    return (out, selected) if return_selected else out


def decode_attn_topk_tokens(q, K, V, top_k: int, scale: Optional[float] = None,
                            out_dtype: torch.dtype = torch.float32,
                            out: Optional[torch.Tensor] = None, return_selected: bool = False,
                            selected: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None):
    """Token-level sparse decode attention: per q-head, the top_k tokens by the
    exact score q . k and attention over them only (K contiguous [B, Hkv, N, d])."""
    ks, B, H, N, d = _kv_struct(K)
    vs, B2, H2, N2, d2 = _kv_struct(V)
    if (B, H, N, d) != (B2, H2, N2, d2):
        raise ValueError("K and V shapes differ")
    if out is None:
        out = torch.empty(B, q.shape[1], d, dtype=out_dtype, device=q.device)
    kk = min(int(top_k), N)
    if return_selected and selected is None:
        selected = torch.empty(B, q.shape[1], kk, dtype=torch.int32, device=q.device)
    p = _params(q, B, H, N, d, out, scale)
    nbytes = lib().dkv_workspace_bytes_tokens(ctypes.byref(p), int(top_k))
    ws = _workspace(nbytes, q.device, workspace)
    sel_ptr = selected.data_ptr() if selected is not None else None
    _check(lib().dkv_decode_attn_topk_tokens(ctypes.byref(p), q.data_ptr(), ctypes.byref(ks),
                                             ctypes.byref(vs), int(top_k), out.data_ptr(),
                                             _dtype_code(out.dtype), sel_ptr, ws.data_ptr(),
                                             nbytes, _stream(q)),
           "dkv_decode_attn_topk_tokens")
    return (out, selected) if return_selected else out


def workspace_bytes_tokens(B: int, Hq: int, Hkv: int, d: int, N: int, top_k: int) -> int:
    """Workspace bytes dkv_decode_attn_topk_tokens needs."""
    p = _Params()
    p.batch, p.num_q_heads, p.num_kv_heads, p.head_dim, p.seq_len = B, Hq, Hkv, d, N
    p.page_size, p.scale = PAGE_SIZE, 1.0
    n = lib().dkv_workspace_bytes_tokens(ctypes.byref(p), int(top_k))
    if n == 0:
        raise DkvError(2, "dkv_workspace_bytes_tokens")
    return int(n)


def kv_quant4(x: torch.Tensor) -> Q4Cache:
    """4-bit group-of-64 quantisation of an fp16 tensor [..., d] (contiguous)."""
    if x.dtype != torch.float16 or not x.is_contiguous():
        raise ValueError("kv_quant4 wants a contiguous fp16 tensor")
    d = x.shape[-1]
    rows = x.numel() // d
    codes = torch.empty(*x.shape[:-1], d // 2, dtype=torch.uint8, device=x.device)
    gmin = torch.empty(*x.shape[:-1], d // 64, dtype=torch.float16, device=x.device)
    gmax = torch.empty_like(gmin)
    _check(lib().dkv_kv_quant4(rows, d, x.data_ptr(), codes.data_ptr(), gmin.data_ptr(),
                               gmax.data_ptr(), _stream(x)), "dkv_kv_quant4")
    return Q4Cache(codes, gmin, gmax)


def kv_dequant4(q4: Q4Cache) -> torch.Tensor:
    codes, gmin, gmax = q4
    d = codes.shape[-1] * 2
    rows = codes.numel() // (d // 2)
    x = torch.empty(*codes.shape[:-1], d, dtype=torch.float16, device=codes.device)
    _check(lib().dkv_kv_dequant4(rows, d, codes.data_ptr(), gmin.data_ptr(), gmax.data_ptr(),
                                 x.data_ptr(), _stream(x)), "dkv_kv_dequant4")
    return x


def attn_ctas_per_sm(head_dim: int, dtype: torch.dtype = torch.bfloat16, q4: bool = False,
                     sparse: bool = False) -> int:
    """Resident CTAs per SM of the persistent attention kernel (a diagnostic)."""
    n = ctypes.c_int32(0)
    _check(lib().dkv_attn_ctas_per_sm(int(head_dim), _dtype_code(dtype),
                                      DKV_KV_Q4G64 if q4 else DKV_KV_DENSE, int(sparse),
                                      ctypes.byref(n)), "dkv_attn_ctas_per_sm")
    return int(n.value)


def read_device_status(workspace: torch.Tensor) -> int:
    """Synchronise and return (then clear) the device status word of a workspace.

    After a device error the workspace's merge counters may be left mid-count,
    so the whole workspace is zero-filled again, ready for the next call.
    """
    st = int(lib().dkv_read_device_status(workspace.data_ptr(), _stream(workspace)))
    if st != DKV_OK:
        workspace.zero_()
    return st

"""Algorithmic byte counts of each step of the decode path (host-side logic).

These are the bytes a step must move at minimum -- every input read once and
every output written once -- and are the numerators of the roofline figures.

TinyServe ("TinyServe: Query-Aware Cache Selection for Efficient LLM Serving",
内存效率量化模型构建 / 与全缓存注意力的归一化对比) models one sparse decode
step as moving 2M(L/S + rho K S) bytes (per-page min/max metadata plus the K
selected pages' K and V; M = bytes per token of one cache tensor) against 2ML
for full attention, i.e. a fraction 1/S + rho K S / L.  With rho = 1 (no reuse
across steps: every call here is one step) select_bytes / full_bytes reduces
to that fraction for MHA when q and out are left out.
"""

from __future__ import annotations


def _el(dtype_bytes: int) -> int:
    return int(dtype_bytes)


def full_bytes(B, Hq, Hkv, d, N, elt=2, out_elt=4, q4=False) -> int:
    """q + K + V (+ the 4-bit format's group min / max) + out."""
    q = B * Hq * d * elt
    out = B * Hq * d * out_elt
    if q4:
        kv = 2 * B * Hkv * N * (d // 2 + 2 * (d // 64) * 2)
    else:
        kv = 2 * B * Hkv * N * d * elt
    return q + kv + out


def meta_bytes(B, Hkv, d, N, S=16, elt=2, q4=False) -> int:
    """K read + (m_j, M_j) written."""
    P = (N + S - 1) // S
    k = B * Hkv * N * ((d // 2 + 2 * (d // 64) * 2) if q4 else d * elt)
    return k + 2 * B * Hkv * P * d * elt


def select_bytes(B, Hq, Hkv, d, N, gathered_tokens, S=16, elt=2, out_elt=4, q4=False) -> int:
    """q + metadata of every page + K and V of the gathered tokens + out.

    gathered_tokens: total valid tokens of the unique pages gathered over all
    (batch, kv head) -- the union of the group's selections, each page once.
    """
    P = (N + S - 1) // S
    q = B * Hq * d * elt
    out = B * Hq * d * out_elt
    meta = 2 * B * Hkv * P * d * elt
    per_tok = (d // 2 + 2 * (d // 64) * 2) if q4 else d * elt
    return q + meta + 2 * gathered_tokens * per_tok + out


def meta8_bytes(B, Hkv, d, N, S=16, elt=2) -> int:
    """16-bit page metadata read; 8-bit codes and the per-page grid written."""
    P = (N + S - 1) // S
    return 2 * B * Hkv * P * d * elt + 2 * B * Hkv * P * d + 2 * B * Hkv * P * 4


def select8_bytes(B, Hq, Hkv, d, N, gathered_tokens, S=16, elt=2, out_elt=4,
                  q4=False) -> int:
    """q + 8-bit metadata of every page (two code bytes per channel, lo and
    step) + K and V of the gathered tokens + out."""
    P = (N + S - 1) // S
    q = B * Hq * d * elt
    out = B * Hq * d * out_elt
    meta = 2 * B * Hkv * P * d + 2 * B * Hkv * P * 4
    per_tok = (d // 2 + 2 * (d // 64) * 2) if q4 else d * elt
    return q + meta + 2 * gathered_tokens * per_tok + out


def quant4_bytes(rows, d) -> int:
    """fp16 rows read + 4-bit codes and group min / max written."""
    return rows * d * 2 + rows * (d // 2 + 2 * (d // 64) * 2)


def memory_fraction(S: int, K: int, L: int, rho: float = 1.0) -> float:
    """TinyServe's sparse-over-full memory fraction 1/S + rho K S / L."""
    return 1.0 / S + rho * K * S / L


def token_bytes(B, Hq, Hkv, d, N, kk, elt=2, out_elt=4) -> int:
    """Token-level top-K attention: q + all of K (every token is scored) + the
    V rows of each q-head's kk selected tokens + out.  The score workspace is
    overhead, as for the page-sparse path."""
    return B * Hq * d * elt + B * Hkv * N * d * elt + B * Hq * kk * d * elt + B * Hq * d * out_elt

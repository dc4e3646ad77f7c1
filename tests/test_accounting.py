"""The bench's byte accounting reproduces TinyServe's memory-fraction model
("TinyServe: ...", 与全缓存注意力的归一化对比: 1/S + rho K S / L, rho = 1)."""

import pytest

from decode_attention_paged_kv_gb300 import accounting as acc


@pytest.mark.parametrize("N,K,S,d", [(8192, 128, 16, 64), (32768, 128, 16, 128),
                                     (32768, 614, 16, 128), (2048, 32, 16, 128)])
def test_select_over_full_is_memory_fraction(N, K, S, d):
    B, H = 3, 5  # MHA: each head gathers exactly its own K pages
    gathered = B * H * K * S
    q_out = B * H * d * 2 + B * H * d * 4
    sel = acc.select_bytes(B, H, H, d, N, gathered, S=S) - q_out
    full = acc.full_bytes(B, H, H, d, N) - q_out
    assert sel / full == pytest.approx(acc.memory_fraction(S, K, N), rel=1e-12)


def test_fraction_values():
    # K = 0.3 P at L = 32K, S = 16: 1/16 + 0.3 = 0.3625 (about 2.8x less traffic)
    P = 32768 // 16
    assert acc.memory_fraction(16, int(0.3 * P), 32768) == pytest.approx(1 / 16 + 614 * 16 / 32768)
    assert acc.memory_fraction(16, 128, 8192) == pytest.approx(0.3125)


def test_full_bytes_workloads():
    # Llama-3-8B GQA, B=16, N=32K: 2 GiB of K+V
    kv = acc.full_bytes(16, 32, 8, 128, 32768) - 16 * 32 * 128 * 6
    assert kv == 2 * 2 ** 30
    # 1M tokens x 8 kv heads x d=128: 4 GiB
    assert acc.full_bytes(1, 32, 8, 128, 1 << 20) - 32 * 128 * 6 == 4 * 2 ** 30
    # 4-bit OPT-30B shape: codes + group min/max
    b = acc.full_bytes(64, 56, 56, 128, 2048, q4=True) - 64 * 56 * 128 * 6
    assert b == 2 * 64 * 56 * 2048 * (64 + 8)


def test_quant4_bytes():
    # 2 bytes in per value; 4 bits + 4 bytes of bounds per 64 values out
    assert acc.quant4_bytes(10, 128) == 10 * 256 + 10 * (64 + 8)


def test_token_bytes():
    # keeping every token with one head per group reads what the exact path reads
    assert acc.token_bytes(2, 8, 8, 128, 1000, 1000) == acc.full_bytes(2, 8, 8, 128, 1000)
    # GQA: K once per kv head, V rows once per q head
    assert (acc.token_bytes(1, 32, 8, 128, 32768, 3276) ==
            32 * 128 * 2 + 8 * 32768 * 128 * 2 + 32 * 3276 * 128 * 2 + 32 * 128 * 4)


def test_meta8_byte_counts():
    # 32K GQA shape: 16-bit metadata 128 MiB read, codes 64 MiB + grid 1 MiB written
    B, Hkv, d, N = 16, 8, 128, 32768
    P = N // 16
    assert acc.meta8_bytes(B, Hkv, d, N) == 2 * B * Hkv * P * d * 2 + 2 * B * Hkv * P * d + 8 * B * Hkv * P
    full16 = acc.select_bytes(B, 32, Hkv, d, N, 1000)
    full8 = acc.select8_bytes(B, 32, Hkv, d, N, 1000)
    # the 8-bit metadata scan is half the 16-bit one plus 8 bytes a page
    assert full16 - full8 == 2 * B * Hkv * P * d - 8 * B * Hkv * P

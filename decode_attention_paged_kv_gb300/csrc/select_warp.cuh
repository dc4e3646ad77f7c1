// select_warp.cuh -- one warp selects one query head's pages: the top-K of the
// head's P bound scores, as a bitmap, an ascending row, and (for the group)
// the union list.
//
// Per query head ("TinyServe: Query-Aware Cache Selection for Efficient LLM
// Serving", 问题公式化定义: S_t = TopK_j r(q_t, phi_j), |S_t| = K; Algorithm 1
// step 2): the K largest of the head's P scores, ties taken by the lower page
// index.  Scores become order-preserving 32-bit keys held in registers (lane l
// owns pages 32 i + l).  The keys' minimum and maximum give the leading bits
// they all share; below those, the K-th largest key T is found bit by bit
// (keep bit b when at least K keys are >= T | 2^b), stopping as soon as
// exactly K keys are >= T.  Then those K keys are the selection; if instead
// several keys equal T (a tie at the K-th place), the keys above T and the
// first K - #(> T) keys equal to T in page order are.  This is radix selection
// with 1-bit digits; the counts are warp reductions of eight independent
// partial sums each.
// The selection is a bitmap over pages in shared memory; the ascending row is
// written from it.  The union of the group's bitmaps, ascending, each page
// with a bit per query head that chose it, is the list the sparse attention
// gathers.
#pragma once

#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {

constexpr int kSelKeys = kUnitMaxP / 32;  // keys a lane holds
// Bitmap words of one query head.
constexpr int kSelBitmapWords = kUnitMaxP / 32;

// -1 when a < b, else 0: the borrow of a - b (no predicate register per compare).
__device__ __forceinline__ int minus_borrow(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("{\n\t.reg .u32 t;\n\tsub.cc.u32 t, %1, %2;\n\tsubc.u32 %0, 0, 0;\n\t}"
      : "=r"(d)
      : "r"(a), "r"(b));
  return static_cast<int>(d);
}

// Keys >= x among the warp's keys k (slots past the head's P hold 0, and
// x >= 1, so they never count).  Every slot is counted: a per-group bound
// check costs more than the compares it saves.  Eight partial sums keep the
// compares from forming one dependent chain.
template <int NK>
__device__ __forceinline__ int warp_count_ge(const uint32_t (&k)[NK], uint32_t x) {
  int c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < NK; ++i) c[i & 7] += minus_borrow(k[i], x);
  const int below = -(((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7])));
  return 32 * NK - __reduce_add_sync(0xffffffffu, below);
}

// The largest T such that at least lo of the warp's keys are >= T, found bit by
// bit from bit `top` down, starting from T0 (every key at hand is >= T0 and
// agrees with it above bit `top`); stops early (with a smaller T) once the
// count of keys >= T lies in [lo, hi].  ge = keys >= T.  lo >= 1.
template <int NK>
__device__ uint32_t warp_threshold(const uint32_t (&k)[NK], int lo, int hi, int& ge,
                                   uint32_t T0 = 0u, int top = 31) {
  uint32_t T = T0;
  ge = -1;  // not counted: every key at hand is >= T0
  for (int bit = top; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    const int c = warp_count_ge(k, cand);
    if (c >= lo) {
      T = cand;
      ge = c;
      if (c <= hi) break;
    }
  }
  return T;
}

// Top-kk of one head's P keys (key_at(j): the order-preserving key of page j;
// 1 <= kk <= P <= 32 NK) by one warp, NK key slots a lane: writes the
// selection bitmap words bm[0 .. ceil(P / 32)).  kmax / kmin: the largest and
// smallest of the keys.
template <int NK, class KeyAt>
__device__ void warp_topk_head_n(const KeyAt& key_at, int P, int kk, uint32_t* bm, uint32_t kmax,
                                 uint32_t kmin) {
  static_assert(NK % 8 == 0 && NK <= kSelKeys, "eight ballots at a time");
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const int nr = static_cast<int>(ceil_div(P, 32));         // key rows
  const int nv = static_cast<int>(ceil_div(P - lane, 32));  // this lane's valid rows
  uint32_t key[NK];
#pragma unroll
  for (int i = 0; i < NK; ++i) key[i] = i < nv ? key_at(32 * i + lane) : 0u;
  // The kk-th largest key T, bit by bit below the common prefix (keys past P
  // read as 0 and stay below every candidate when the prefix is not 0).
  int ge = -1;
  uint32_t T;
  if (kmax == kmin) {
    T = kmax;  // all equal: a tie at T
  } else {
    const int top = 31 - __clz(kmax ^ kmin);
    const uint32_t prefix = top == 31 ? 0u : (kmax >> (top + 1)) << (top + 1);
    T = warp_threshold(key, kk, kk, ge, prefix, top);
  }
  if (ge == kk) {
    // No tie at T: the selection is every key >= T (eight ballots at a time).
#pragma unroll
    for (int g = 0; g < NK / 8; ++g) {
      if (8 * g < nr) {
        uint32_t m8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) m8[u] = __ballot_sync(0xffffffffu, 8 * g + u < nv && key[8 * g + u] >= T);
        if (lane < 8 && 8 * g + lane < nr) {
          uint32_t v = m8[0];
#pragma unroll
          for (int u = 1; u < 8; ++u) v = lane == u ? m8[u] : v;
          bm[8 * g + lane] = v;
        }
      }
    }
    return;
  }
  // Ties at T (or keys past P that compare as 0 with a zero prefix): T exactly,
  // then keys > T and the first kk - #(> T) keys equal to T in page order.
  T = warp_threshold(key, kk, kk, ge);
  int gt = 0;
#pragma unroll
  for (int i = 0; i < NK; ++i)
    if (i < nr) gt += __popc(__ballot_sync(0xffffffffu, i < nv && key[i] > T));
  const int need = kk - gt;  // keys equal to T to take, lowest pages first
  int eq_before = 0;
#pragma unroll
  for (int i = 0; i < NK; ++i) {
    if (i < nr) {
      const bool is_gt = i < nv && key[i] > T, is_eq = i < nv && key[i] == T;
      const uint32_t eqm = __ballot_sync(0xffffffffu, is_eq);
      const int eq_rank = eq_before + __popc(eqm & lt);
      const uint32_t selm = __ballot_sync(0xffffffffu, is_gt || (is_eq && eq_rank < need));
      if (lane == 0) bm[i] = selm;
      eq_before += __popc(eqm);
    }
  }
}

// The same with as few key slots a lane as P needs (every count touches every
// slot, so short heads run on 16 or 32).  SHORT = false keeps one copy (64
// slots), for kernels whose heads are long and whose code size matters.
template <bool SHORT = true, class KeyAt>
__device__ void warp_topk_head(const KeyAt& key_at, int P, int kk, uint32_t* bm, uint32_t kmax,
                               uint32_t kmin) {
  if constexpr (SHORT) {
    if (P <= 16 * 32) {
      warp_topk_head_n<16>(key_at, P, kk, bm, kmax, kmin);
      return;
    }
    if (P <= 32 * 32) {
      warp_topk_head_n<32>(key_at, P, kk, bm, kmax, kmin);
      return;
    }
  }
  warp_topk_head_n<kSelKeys>(key_at, P, kk, bm, kmax, kmin);
}

// Ascending page rows from a head's selection bitmap (words [0, W)); the words
// also go to bm_out when it is not null.
__device__ inline void warp_emit_row(const uint32_t* bm, int W, int32_t* out, uint32_t* bm_out) {
  const int lane = threadIdx.x & 31;
  int pos = 0;
  for (int base = 0; base < W; base += 32) {
    const int w = base + lane;
    uint32_t x = w < W ? bm[w] : 0u;
    if (bm_out != nullptr && w < W) bm_out[w] = x;
    const int c = __popc(x);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    int at = pos + incl - c;
    while (x) {
      const int bit = __ffs(x) - 1;
      x &= x - 1;
      out[at++] = w * 32 + bit;
    }
    pos += __shfl_sync(0xffffffffu, incl, 31);
  }
}

}  // namespace dkv

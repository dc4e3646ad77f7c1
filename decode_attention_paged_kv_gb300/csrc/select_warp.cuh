// select_warp.cuh -- one warp selects one query head's pages: the top-K of the
// head's P bound scores, as a bitmap, an ascending row, and (for the group)
// the union list.
//
// Per query head ("TinyServe: Query-Aware Cache Selection for Efficient LLM
// Serving", 问题公式化定义: S_t = TopK_j r(q_t, phi_j), |S_t| = K; Algorithm 1
// step 2): the K largest of the head's P scores, ties taken by the lower page
// index.  Scores become order-preserving 32-bit keys held in registers (lane l
// owns pages 32 i + l).
//   1. A threshold estimate T' from every 4th page's key: a rank in that
//      sample a little above the one that scales to K, found bit by bit from
//      the top (keep bit b of the result when enough sampled keys are
//      >= result | 2^b), stopping once the count falls in a window.
//   2. One pass counts the keys >= T'.  If that is at least K and at most
//      kCandCap, the candidates are compacted into shared memory and the exact
//      K-th largest key T among them is found the same way.  If exactly K
//      candidates are >= T, they are the selection.
//   3. Otherwise (a poor estimate, or ties at T to break by page order) the
//      same exact search runs over all keys, and the first K - #(> T) keys
//      equal to T in page order complete the selection.
// The selection is a bitmap over pages in shared memory; the ascending row is
// written from it.  The union of the group's bitmaps, ascending, each page
// with a bit per query head that chose it, is the list the sparse attention
// gathers.
#pragma once

#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {

constexpr int kSelKeys = kUnitMaxP / 32;  // keys a lane holds
constexpr int kSampleStride = 4;           // the estimate reads every 4th page
constexpr int kSampleKeys = kSelKeys / kSampleStride;
constexpr int kCandCap = 512;              // candidates the exact search takes
constexpr int kCandKeys = kCandCap / 32;
// Bitmap words of one query head.
constexpr int kSelBitmapWords = kUnitMaxP / 32;
// A selecting warp's scratch: the head's bitmap, then kCandCap candidate keys
// and kCandCap 16-bit page indices.
constexpr int kSelCandOffset = kSelBitmapWords * 4;
constexpr int kSelScratchBytes = kSelCandOffset + kCandCap * (4 + 2);
static_assert(kUnitMaxP <= 65536, "16-bit candidate page indices");
static_assert(kSelKeys % kSampleStride == 0, "whole sample rows");

// -1 when a < b, else 0: the borrow of a - b (no predicate register per compare).
__device__ __forceinline__ int minus_borrow(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("{\n\t.reg .u32 t;\n\tsub.cc.u32 t, %1, %2;\n\tsubc.u32 %0, 0, 0;\n\t}"
      : "=r"(d)
      : "r"(a), "r"(b));
  return static_cast<int>(d);
}

// Keys >= x among the warp's k[0 .. 8 ceil(used / 8)) (unused slots must hold
// 0 and x >= 1).  Eight partial sums keep the compares from forming one
// dependent chain.
template <int NK>
__device__ __forceinline__ int warp_count_ge(const uint32_t (&k)[NK], int used, uint32_t x) {
  int c[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  int slots = 0;
#pragma unroll
  for (int g = 0; g < (NK + 7) / 8; ++g) {
    if (8 * g < used) {
#pragma unroll
      for (int u = 0; u < 8 && 8 * g + u < NK; ++u) c[u] += minus_borrow(k[8 * g + u], x);
      slots += (8 * g + 8 <= NK) ? 8 : NK - 8 * g;
    }
  }
  const int below = -(((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7])));
  return 32 * slots - __reduce_add_sync(0xffffffffu, below);
}

// The largest T such that at least lo of the warp's keys are >= T, found bit by
// bit from the top; stops early (with a smaller T) once the count of keys >= T
// lies in [lo, hi].  ge = keys >= T.  lo >= 1.
template <int NK>
__device__ uint32_t warp_threshold(const uint32_t (&k)[NK], int used, int lo, int hi, int& ge) {
  uint32_t T = 0;
  ge = -1;  // unknown: every key is >= 0
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t cand = T | (1u << bit);
    const int c = warp_count_ge(k, used, cand);
    if (c >= lo) {
      T = cand;
      ge = c;
      if (c <= hi) break;
    }
  }
  return T;
}

// Top-kk of one head's P keys (key_at(j): the order-preserving key of page j;
// 1 <= kk <= P <= kUnitMaxP) by one warp: sets the selected pages' bits in
// bm[0 .. ceil(P / 32)), which the caller has zeroed.  cand_key / cand_page:
// kCandCap-entry buffers.
template <class KeyAt>
__device__ void warp_topk_head(const KeyAt& key_at, int P, int kk, uint32_t* bm,
                               uint32_t* cand_key, uint16_t* cand_page) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const int nr = static_cast<int>(ceil_div(P, 32));         // key rows
  const int nv = static_cast<int>(ceil_div(P - lane, 32));  // this lane's valid rows
  uint32_t key[kSelKeys];
#pragma unroll
  for (int i = 0; i < kSelKeys; ++i) key[i] = i < nv ? key_at(32 * i + lane) : 0u;
  // Sample: pages 0, 4, 8, ...; page 32 i + 4 q (q = 0..7) goes to lane
  // 8 (i % 4) + q, slot i / 4.
  uint32_t smp[kSampleKeys];
#pragma unroll
  for (int m = 0; m < kSampleKeys; ++m) smp[m] = 0u;
#pragma unroll
  for (int i = 0; i < kSelKeys; ++i) {
    if (i < nr) {
      const uint32_t v = __shfl_sync(0xffffffffu, key[i], 4 * (lane & 7));
      if ((lane >> 3) == (i & 3)) smp[i >> 2] = v;
    }
  }
  const int S = static_cast<int>(ceil_div(P, kSampleStride));
  const int ns = static_cast<int>(ceil_div(nr, kSampleStride));  // sample slots in use
  bool done = false;
  // 1. The estimate: a sample rank window a little above kk * S / P.
  const float want = static_cast<float>(kk) * static_cast<float>(S) / static_cast<float>(P);
  const int lo = static_cast<int>(want + 2.f * sqrtf(want) + 3.f);
  const int hi = static_cast<int>(want + 3.f * sqrtf(want) + 5.f);
  if (lo < S) {
    int ge_s;
    const uint32_t Te = warp_threshold(smp, ns, lo, hi, ge_s);
    // 2. Keys >= T' (T' >= 1 unless scores were NaN; then the full search).
    const int C = Te >= 1 ? warp_count_ge(key, nr, Te) : P + 1;
    if (C >= kk && C <= kCandCap) {
      int mine = 0;
#pragma unroll
      for (int i = 0; i < kSelKeys; ++i) mine += (i < nr && key[i] >= Te) ? 1 : 0;
      int incl = mine;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
      }
      int at = incl - mine;
#pragma unroll
      for (int i = 0; i < kSelKeys; ++i) {
        if (i < nr && key[i] >= Te) {  // keys past P are 0 < T'
          cand_key[at] = key[i];
          cand_page[at] = static_cast<uint16_t>(32 * i + lane);
          ++at;
        }
      }
      __syncwarp();
      // 3. Exact kk-th largest key among the C candidates.
      uint32_t ck[kCandKeys];
#pragma unroll
      for (int m = 0; m < kCandKeys; ++m) {
        const int c = lane + 32 * m;
        ck[m] = c < C ? cand_key[c] : 0u;
      }
      int ge;
      const uint32_t T = warp_threshold(ck, static_cast<int>(ceil_div(C, 32)), kk, kk, ge);
      if (ge == kk) {  // no tie at T to break
#pragma unroll
        for (int m = 0; m < kCandKeys; ++m) {
          const int c = lane + 32 * m;
          if (c < C && ck[m] >= T) {
            const int pg = cand_page[c];
            atomicOr(bm + (pg >> 5), 1u << (pg & 31));
          }
        }
        done = true;
      }
      __syncwarp();  // the candidate buffers are free again
    }
  }
  if (done) return;
  // Full search over all keys: T = the kk-th largest key.
  int ge_T;
  const uint32_t T = warp_threshold(key, nr, kk, kk, ge_T);
  int gt = 0;
#pragma unroll
  for (int i = 0; i < kSelKeys; ++i)
    if (i < nr) gt += __popc(__ballot_sync(0xffffffffu, i < nv && key[i] > T));
  const int need = kk - gt;  // keys equal to T to take, lowest pages first
  int eq_before = 0;
#pragma unroll
  for (int i = 0; i < kSelKeys; ++i) {
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

// Union of G heads' selection bitmaps (bm + h * stride, words [0, W); in
// global memory, or shared when global is false), ascending, with a bit per
// head: out[0 .. count) = (page, mask); returns count to every lane.
__device__ inline int warp_union(const uint32_t* bm, int64_t stride, int G, int W, int2* out,
                          bool global = true) {
  const int lane = threadIdx.x & 31;
  int pos = 0;
  for (int base = 0; base < W; base += 32) {
    const int w = base + lane;
    uint32_t hw[8];
    uint32_t u = 0;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      hw[h] = (h < G && w < W) ? (global ? __ldcg(bm + h * stride + w) : bm[h * stride + w]) : 0u;
      u |= hw[h];
    }
    const int c = __popc(u);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    int at = pos + incl - c;
    while (u) {
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      uint32_t m = 0;
#pragma unroll
      for (int h = 0; h < 8; ++h) m |= ((hw[h] >> bit) & 1u) << h;
      out[at++] = make_int2(w * 32 + bit, static_cast<int>(m));
    }
    pos += __shfl_sync(0xffffffffu, incl, 31);
  }
  return pos;
}

}  // namespace dkv

// select.cu -- query-aware page selection: bound scores and top-K.
//
// Bound score ("TinyServe: Query-Aware Cache Selection for Efficient LLM
// Serving", 相关性函数实例化; Algorithm 1 step 1):
//   r(q, phi_j) = sum_i (q_i >= 0 ? q_i M_ji : q_i m_ji)
// Because the two cases are exclusive it equals  q+ . M_j + q- . m_j  with
// q+ = max(q, 0), q- = min(q, 0): one dot product of length 2d between the
// page's concatenated metadata [M_j | m_j] and [q+ | q-].  score_kernel runs it
// for 16 pages x (up to 8) query heads per mma.sync m16n8k16 step: pages on the
// M side straight from global memory (16-byte loads, coalesced rows), the G
// query heads of the group on the N side.  bf16 x bf16 products are exact in
// the fp32 accumulator.
//
// Top-K (问题公式化定义: S_t = TopK_j r, |S_t| = K; Algorithm 1 step 2, "radix
// select"): topk_kernel radix-selects the K largest scores of one (b, h) row on
// order-preserving 32-bit keys (8-bit digits, most significant first), then
// writes the selected pages in ascending order; among equal scores the lower
// page index is taken first.  It also writes a bitmap of the selection, which
// the sparse attention kernel merges across the heads of a group.

#include <math.h>

#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {
namespace {

constexpr int kScoreWarps = 4;
constexpr int kScorePagesPerCta = 16 * kScoreWarps;

// Split 8 packed 16-bit q values (one 16-byte chunk) into q+ or q-.
__device__ __forceinline__ uint32_t keep_sign(uint32_t w, bool negative_part) {
  uint32_t out = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t v = (w >> (16 * h)) & 0xffffu;
    const bool neg = (v & 0x8000u) && (v & 0x7fffu);
    if (neg == negative_part) out |= v << (16 * h);
  }
  return out;
}

template <int D, bool F16>
__global__ void __launch_bounds__(kScoreWarps * 32) score_kernel(const ScoreArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int page0 = blockIdx.x * kScorePagesPerCta + warp * 16;
  griddep_launch_dependents();
  griddep_wait();
  if (page0 >= a.P) return;

  // Contraction index k (0..2d) runs over the concatenation [M | m]; thread
  // (g, t4) owns 16-byte chunks c = t4 + 4 s of it, each giving two k-steps.
  constexpr int kChunks = D / 16;  // per thread per row
  // B operand: [q+ | q-] of head g (zero for g >= G).
  uint32_t bq[kChunks][4];
  {
    const bool hv = g < a.G;
    const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + b * a.q_sb +
                           static_cast<int64_t>(kvh * a.G + (hv ? g : 0)) * a.q_sh;
#pragma unroll
    for (int s = 0; s < kChunks; ++s) {
      const int c = t4 + 4 * s;
      const bool neg_part = c >= D / 8;
      const int ch = 8 * (neg_part ? c - D / 8 : c);
      uint4 w = hv ? *reinterpret_cast<const uint4*>(qrow + ch) : make_uint4(0, 0, 0, 0);
      bq[s][0] = keep_sign(w.x, neg_part);
      bq[s][1] = keep_sign(w.y, neg_part);
      bq[s][2] = keep_sign(w.z, neg_part);
      bq[s][3] = keep_sign(w.w, neg_part);
    }
  }
  // A operand: rows g and g + 8 are pages page0 + g and page0 + g + 8.
  const int64_t mbase = (static_cast<int64_t>(b) * a.Hkv + kvh) * a.P;
  const uint16_t* mmax = static_cast<const uint16_t*>(a.meta_max);
  const uint16_t* mmin = static_cast<const uint16_t*>(a.meta_min);
  uint4 ra[2][kChunks];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int page = page0 + g + 8 * hr;
    const bool pv = page < a.P;
#pragma unroll
    for (int s = 0; s < kChunks; ++s) {
      const int c = t4 + 4 * s;
      const uint16_t* src = (c < D / 8) ? mmax + (mbase + page) * D + 8 * c
                                        : mmin + (mbase + page) * D + 8 * (c - D / 8);
      ra[hr][s] = pv ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
    }
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < kChunks; ++s) {
    mma16816<F16>(acc, ra[0][s].x, ra[1][s].x, ra[0][s].y, ra[1][s].y, bq[s][0], bq[s][1]);
    mma16816<F16>(acc, ra[0][s].z, ra[1][s].z, ra[0][s].w, ra[1][s].w, bq[s][2], bq[s][3]);
  }
  // acc: [page g][head 2t4], [g][2t4+1], [g+8][2t4], [g+8][2t4+1]
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int head = 2 * t4 + (e & 1);
    const int page = page0 + g + 8 * (e >> 1);
    if (head < a.G && page < a.P)
      a.scores[(static_cast<int64_t>(b) * a.Hq + kvh * a.G + head) * a.P + page] = acc[e];
  }
}

// Order-preserving key of an fp32 score (-0 taken as +0).
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kTopkThreads = 256;
constexpr size_t kTopkSmemKeyBytes = 160 * 1024;  // rows of up to 40960 pages
constexpr int kTopkMaxWordsSmem = 2048;           // bitmap words built in shared memory

// Block-wide exclusive prefix sum of v.
__device__ __forceinline__ long long block_excl_sum(long long v, long long* warp_tot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  long long before = 0;
#pragma unroll
  for (int w = 0; w < kTopkThreads / 32; ++w) before += (w < warp) ? warp_tot[w] : 0;
  return before + incl - v;
}

// Keys of one row: staged in shared memory once when they fit, else re-read
// (order-preserving transform applied on the fly) from global memory.
template <bool SMEM>
struct RowKeys {
  const float* r;
  const uint32_t* s;
  __device__ __forceinline__ uint32_t operator()(int j) const {
    if constexpr (SMEM) return s[j];
    return score_key(__ldcg(r + j));
  }
};

// One CTA per (b, h) row.  Radix select on 8-bit digits, most significant
// first: each pass histograms the digit of the keys that still match the
// prefix (one shared atomic per distinct digit per warp), and warp 0 finds the
// digit that holds the K-th largest key.  Then every thread takes a contiguous
// range of pages: keys above the threshold are in, keys equal to it are in for
// the first `need` of them in page order; one block scan gives every thread
// its output position, so pages come out ascending.
template <bool SMEM>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkArgs a) {
  extern __shared__ uint32_t s_keys[];
  __shared__ uint32_t hist[256];
  __shared__ long long warp_tot[kTopkThreads / 32];
  __shared__ uint32_t s_digit, s_above;
  __shared__ uint32_t s_bits[kTopkMaxWordsSmem];
  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  griddep_launch_dependents();
  griddep_wait();  // the scores come from the previous kernel
  const float* r = a.scores + static_cast<int64_t>(row) * a.P;
  if constexpr (SMEM) {
#pragma unroll 8
    for (int j = tid; j < a.P; j += kTopkThreads) s_keys[j] = score_key(__ldcg(r + j));
  }
  const RowKeys<SMEM> key{r, s_keys};
  const int P_round = (a.P + kTopkThreads - 1) / kTopkThreads * kTopkThreads;

  uint32_t prefix = 0, mask = 0;
  int need = a.kk;  // still to choose among keys matching `prefix` under `mask`
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    hist[tid] = 0;
    __syncthreads();
    for (int j = tid; j < P_round; j += kTopkThreads) {
      const uint32_t k = (j < a.P) ? key(j) : 0u;
      const bool in = (j < a.P) && (k & mask) == prefix;
      const uint32_t digit = (k >> shift) & 0xffu;
      const uint32_t act = __ballot_sync(0xffffffffu, in);
      if (in) {
        const uint32_t peers = __match_any_sync(act, digit);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(peers)));
      }
    }
    __syncthreads();
    if (tid < 32) {
      // lane L owns digits 255-8L .. 248-8L (descending).
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        c[u] = hist[255 - 8 * tid - u];
        sum += c[u];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
        if (tid >= off) incl += t;
      }
      uint32_t above = incl - sum;  // keys with a larger digit
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (above < static_cast<uint32_t>(need) && above + c[u] >= static_cast<uint32_t>(need)) {
          s_digit = 255 - 8 * tid - u;
          s_above = above;
        }
        above += c[u];
      }
    }
    __syncthreads();
    const uint32_t digit = s_digit;
    need -= static_cast<int>(s_above);
    prefix |= digit << shift;
    mask |= 0xffu << shift;
    const bool all_taken = hist[digit] == static_cast<uint32_t>(need);
    __syncthreads();
    if (all_taken) break;
  }

  // Contiguous page range of this thread; counts of keys above / equal.
  const int per = (a.P + kTopkThreads - 1) / kTopkThreads;
  const int j0 = min(a.P, tid * per), j1 = min(a.P, j0 + per);
  int gt = 0, eq = 0;
  for (int j = j0; j < j1; ++j) {
    const uint32_t k = key(j) & mask;
    gt += k > prefix;
    eq += k == prefix;
  }
  const bool bits_in_smem = a.W32 <= kTopkMaxWordsSmem;
  if (bits_in_smem)
    for (int w = tid; w < a.W32; w += kTopkThreads) s_bits[w] = 0u;
  // One scan of (gt << 32 | eq): both sums stay below 2^31.
  const long long before =
      block_excl_sum((static_cast<long long>(gt) << 32) | static_cast<long long>(eq), warp_tot);
  int gt_before = static_cast<int>(before >> 32);
  int eq_before = static_cast<int>(before & 0xffffffffll);
  for (int j = j0; j < j1; ++j) {
    const uint32_t k = key(j) & mask;
    bool sel = false;
    if (k > prefix) {
      sel = true;
    } else if (k == prefix) {
      sel = eq_before < need;
      ++eq_before;
    }
    if (sel) {
      const int pos = gt_before + min(eq_before - (k == prefix ? 1 : 0), need);
      a.selected[static_cast<int64_t>(row) * a.kk + pos] = j;
      if (bits_in_smem) atomicOr(&s_bits[j >> 5], 1u << (j & 31));
      else atomicOr(&a.bitmaps[static_cast<int64_t>(row) * a.W32 + (j >> 5)], 1u << (j & 31));
      if (k > prefix) ++gt_before;
    }
  }
  if (bits_in_smem) {
    __syncthreads();
    for (int w = tid; w < a.W32; w += kTopkThreads)
      a.bitmaps[static_cast<int64_t>(row) * a.W32 + w] = s_bits[w];
  }
}

}  // namespace

cudaError_t launch_score(int d, bool f16, const ScoreArgs& a, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(ceil_div(a.P, kScorePagesPerCta)), a.Hkv, a.B);
  dim3 block(kScoreWarps * 32);
  if (d == 128) {
    return f16 ? launch_pdl(score_kernel<128, true>, grid, block, 0, s, a)
               : launch_pdl(score_kernel<128, false>, grid, block, 0, s, a);
  }
  return f16 ? launch_pdl(score_kernel<64, true>, grid, block, 0, s, a)
             : launch_pdl(score_kernel<64, false>, grid, block, 0, s, a);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
  const size_t key_bytes = sizeof(uint32_t) * static_cast<size_t>(a.P);
  if (key_bytes <= kTopkSmemKeyBytes) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kTopkSmemKeyBytes));
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_kernel<true>, dim3(a.rows), dim3(kTopkThreads), key_bytes, s, a);
  }
  // Large rows set their bitmap bits straight in global memory: clear it first.
  if (a.W32 > kTopkMaxWordsSmem) {
    cudaError_t e = cudaMemsetAsync(a.bitmaps, 0,
                                    sizeof(uint32_t) * static_cast<size_t>(a.rows) * a.W32, s);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(topk_kernel<false>, dim3(a.rows), dim3(kTopkThreads), 0, s, a);
}

}  // namespace dkv

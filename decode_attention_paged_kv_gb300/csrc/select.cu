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
constexpr size_t kTopkSmemKeyBytes = 192 * 1024;  // rows of up to 49152 pages

// Block-wide exclusive prefix count of `flag`; *total gets the block total.
__device__ __forceinline__ int block_excl_count(bool flag, int* warp_tot, int* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(bal);
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kTopkThreads / 32; ++w) {
    const int v = warp_tot[w];
    before += (w < warp) ? v : 0;
    tot += v;
  }
  __syncthreads();
  *total = tot;
  return before + in_warp;
}

// Keys of one row: staged in shared memory once when they fit, else re-read
// (order-preserving transform applied on the fly) from global memory.
template <bool SMEM>
struct RowKeys {
  const float* r;
  const uint32_t* s;
  __device__ __forceinline__ uint32_t operator()(int j) const {
    if constexpr (SMEM) return s[j];
    return score_key(r[j]);
  }
};

template <bool SMEM>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkArgs a) {
  extern __shared__ uint32_t s_keys[];
  __shared__ uint32_t hist[256];
  __shared__ int warp_tot[kTopkThreads / 32];
  __shared__ uint32_t s_digit, s_above;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  griddep_launch_dependents();
  griddep_wait();  // the scores come from the previous kernel
  const float* r = a.scores + static_cast<int64_t>(row) * a.P;
  if constexpr (SMEM) {
#pragma unroll 8
    for (int j = tid; j < a.P; j += kTopkThreads) s_keys[j] = score_key(__ldcg(r + j));
  }
  const RowKeys<SMEM> key{r, s_keys};

  uint32_t prefix = 0, mask = 0;
  int need = a.kk;  // still to choose among keys matching `prefix` under `mask`
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    hist[tid] = 0;
    __syncthreads();
    for (int j = tid; j < a.P; j += kTopkThreads) {
      const uint32_t k = key(j);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 0xffu], 1u);
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

  // Keys above the threshold prefix are in; of those equal to it, the first
  // `need` in ascending page order.  Emit ascending.
  int eq_before = 0, sel_before = 0;
  for (int base = 0; base < a.P; base += kTopkThreads) {
    const int j = base + tid;
    const uint32_t k = (j < a.P) ? (key(j) & mask) : 0u;
    const bool gt = (j < a.P) && k > prefix;
    const bool eq = (j < a.P) && k == prefix;
    int eq_tot, sel_tot;
    const int eq_rank = eq_before + block_excl_count(eq, warp_tot, &eq_tot);
    const bool sel = gt || (eq && eq_rank < need);
    const int pos = sel_before + block_excl_count(sel, warp_tot, &sel_tot);
    if (sel && pos < a.kk) a.selected[static_cast<int64_t>(row) * a.kk + pos] = j;
    const uint32_t bal = __ballot_sync(0xffffffffu, sel);
    const int word = (base >> 5) + (tid >> 5);
    if ((tid & 31) == 0 && word < a.W32) a.bitmaps[static_cast<int64_t>(row) * a.W32 + word] = bal;
    eq_before += eq_tot;
    sel_before += sel_tot;
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
  return launch_pdl(topk_kernel<false>, dim3(a.rows), dim3(kTopkThreads), 0, s, a);
}

}  // namespace dkv

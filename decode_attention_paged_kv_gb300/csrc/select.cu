// select.cu -- query-aware page selection: bound scores, per-head top-K and
// the union of a query group's selected pages.
//
// Bound score ("TinyServe: Query-Aware Cache Selection for Efficient LLM
// Serving", 相关性函数实例化; Algorithm 1 step 1):
//   r(q, phi_j) = sum_i (q_i >= 0 ? q_i M_ji : q_i m_ji)
// Because the two cases are exclusive it equals  q+ . M_j + q- . m_j  with
// q+ = max(q, 0), q- = min(q, 0): one dot product of length 2d between the
// page's concatenated metadata [M_j | m_j] and [q+ | q-].  score_tile runs it
// for 16 pages x (up to 8) query heads per mma.sync m16n8k16 step: pages on the
// M side straight from global memory (16-byte loads, coalesced rows), the G
// query heads of the group on the N side.  bf16 x bf16 products are exact in
// the fp32 accumulator.
//
// Top-K (问题公式化定义: S_t = TopK_j r, |S_t| = K; Algorithm 1 step 2, "radix
// select"): radix selection of the K largest scores of one (b, h) on
// order-preserving 32-bit keys (8-bit digits, most significant first), then
// the selected pages in ascending order; among equal scores the lower page
// index is taken first.
//
// Union: the pages any query head of a group selected, ascending, each with a
// bit per head that chose it -- the list the sparse attention gathers (each
// page once for the whole group).
//
// Three kernels, chained with programmatic dependent launch: score_kernel
// (scores to global memory), topk_kernel (one CTA per (b, h): selection and
// its bitmap) and union_kernel (one CTA per (batch, kv head)).

#include <math.h>

#include "select_warp.cuh"
#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {
namespace {

constexpr int kScoreWarps = 4;
constexpr int kScorePagesPerCta = 16 * kScoreWarps;
constexpr int kSelThreads = 256;  // top-K and union CTAs
constexpr int kSelWarps = kSelThreads / 32;
constexpr size_t kTopkSmemKeyBytes = 160 * 1024;  // stage rows of up to 40960 pages

// B operand of the score MMA for lane (g, t4): [q+ | q-] of query head g of the
// group (zero for g >= G).  The contraction index runs over the concatenation
// [M | m]; the lane owns 16-byte chunks c = t4 + 4 s of it, two k-steps each.
template <int D>
__device__ __forceinline__ void load_q_pm(const void* q, int64_t q_sb, int64_t q_sh, int b,
                                          int kvh, int G, int lane,
                                          uint32_t (&bq)[D / 16][4]) {
  const int g = lane >> 2, t4 = lane & 3;
  const bool hv = g < G;
  const uint16_t* qrow = static_cast<const uint16_t*>(q) + b * q_sb +
                         static_cast<int64_t>(kvh * G + (hv ? g : 0)) * q_sh;
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    const int c = t4 + 4 * s;
    const bool neg_part = c >= D / 8;
    const int ch = 8 * (neg_part ? c - D / 8 : c);
    const uint4 w = hv ? *reinterpret_cast<const uint4*>(qrow + ch) : make_uint4(0, 0, 0, 0);
    bq[s][0] = keep_sign(w.x, neg_part);
    bq[s][1] = keep_sign(w.y, neg_part);
    bq[s][2] = keep_sign(w.z, neg_part);
    bq[s][3] = keep_sign(w.w, neg_part);
  }
}

// Bound scores of pages page0 .. page0+15 (< P) of one (batch, kv head) for the
// group's query heads: acc = [page g][head 2t4], [g][2t4+1], [g+8][2t4],
// [g+8][2t4+1].  mmax / mmin point at the unit's [P, d] metadata.
template <int D, bool F16>
__device__ __forceinline__ void score_tile(const uint32_t (&bq)[D / 16][4], const uint16_t* mmax,
                                           const uint16_t* mmin, int page0, int P, int lane,
                                           float (&acc)[4]) {
  const int g = lane >> 2, t4 = lane & 3;
  // Every load is issued before the first MMA (rows past P read a valid page
  // and are zeroed afterwards), so a lane has 2 d / 8 16-byte loads in flight.
  uint4 ra[2][D / 16];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int page = min(page0 + g + 8 * hr, P - 1);
#pragma unroll
    for (int s = 0; s < D / 16; ++s) {
      const int c = t4 + 4 * s;
      const uint16_t* src = (c < D / 8) ? mmax + static_cast<int64_t>(page) * D + 8 * c
                                        : mmin + static_cast<int64_t>(page) * D + 8 * (c - D / 8);
      ra[hr][s] = __ldg(reinterpret_cast<const uint4*>(src));
    }
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    if (page0 + g + 8 * hr >= P) {
#pragma unroll
      for (int s = 0; s < D / 16; ++s) ra[hr][s] = make_uint4(0, 0, 0, 0);
    }
  }
  acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    mma16816<F16>(acc, ra[0][s].x, ra[1][s].x, ra[0][s].y, ra[1][s].y, bq[s][0], bq[s][1]);
    mma16816<F16>(acc, ra[0][s].z, ra[1][s].z, ra[0][s].w, ra[1][s].w, bq[s][2], bq[s][3]);
  }
}

// Two tiles (pages page0.. and page1.. , both < P rows clamped) with every
// load of both issued before the first MMA.
template <int D, bool F16>
__device__ __forceinline__ void score_tile2(const uint32_t (&bq)[D / 16][4], const uint16_t* mmax,
                                            const uint16_t* mmin, int page0, int page1, int P,
                                            int lane, float (&acc0)[4], float (&acc1)[4]) {
  const int g = lane >> 2, t4 = lane & 3;
  uint4 ra[2][2][D / 16];
#pragma unroll
  for (int tt = 0; tt < 2; ++tt) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int page = min((tt ? page1 : page0) + g + 8 * hr, P - 1);
#pragma unroll
      for (int s = 0; s < D / 16; ++s) {
        const int c = t4 + 4 * s;
        const uint16_t* src = (c < D / 8) ? mmax + static_cast<int64_t>(page) * D + 8 * c
                                          : mmin + static_cast<int64_t>(page) * D + 8 * (c - D / 8);
        ra[tt][hr][s] = __ldg(reinterpret_cast<const uint4*>(src));
      }
    }
  }
  acc0[0] = acc0[1] = acc0[2] = acc0[3] = 0.f;
  acc1[0] = acc1[1] = acc1[2] = acc1[3] = 0.f;
#pragma unroll
  for (int s = 0; s < D / 16; ++s) {
    mma16816<F16>(acc0, ra[0][0][s].x, ra[0][1][s].x, ra[0][0][s].y, ra[0][1][s].y, bq[s][0],
                  bq[s][1]);
    mma16816<F16>(acc0, ra[0][0][s].z, ra[0][1][s].z, ra[0][0][s].w, ra[0][1][s].w, bq[s][2],
                  bq[s][3]);
    mma16816<F16>(acc1, ra[1][0][s].x, ra[1][1][s].x, ra[1][0][s].y, ra[1][1][s].y, bq[s][0],
                  bq[s][1]);
    mma16816<F16>(acc1, ra[1][0][s].z, ra[1][1][s].z, ra[1][0][s].w, ra[1][1][s].w, bq[s][2],
                  bq[s][3]);
  }
}

struct SelScratch {
  uint32_t hist[256];
  long long warp_tot[kSelWarps];
  uint32_t digit, above;
};

// Radix selection (block of kSelThreads) of the kk largest of P keys.  On
// return: keys with (key & mask) > prefix are selected, and of the keys with
// (key & mask) == prefix the first `need` in index order.
template <typename KeyFn>
__device__ void block_radix_select(const KeyFn& key, int P, int kk, SelScratch& sc,
                                   uint32_t& prefix, uint32_t& mask, int& need) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int P_round = (P + kSelThreads - 1) / kSelThreads * kSelThreads;
  prefix = 0;
  mask = 0;
  need = kk;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    sc.hist[tid] = 0;
    __syncthreads();
    for (int j = tid; j < P_round; j += kSelThreads) {
      const uint32_t k = (j < P) ? key(j) : 0u;
      const bool in = (j < P) && (k & mask) == prefix;
      const uint32_t digit = (k >> shift) & 0xffu;
      const uint32_t act = __ballot_sync(0xffffffffu, in);
      if (in) {  // one shared atomic per distinct digit per warp
        const uint32_t peers = __match_any_sync(act, digit);
        if (lane == __ffs(peers) - 1)
          atomicAdd(&sc.hist[digit], static_cast<uint32_t>(__popc(peers)));
      }
    }
    __syncthreads();
    if (tid < 32) {
      // lane L owns digits 255-8L .. 248-8L (descending).
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        c[u] = sc.hist[255 - 8 * tid - u];
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
          sc.digit = 255 - 8 * tid - u;
          sc.above = above;
        }
        above += c[u];
      }
    }
    __syncthreads();
    const uint32_t digit = sc.digit;
    need -= static_cast<int>(sc.above);
    prefix |= digit << shift;
    mask |= 0xffu << shift;
    const bool all_taken = sc.hist[digit] == static_cast<uint32_t>(need);
    __syncthreads();
    if (all_taken) break;
  }
}

// Writes the selection in ascending page order to sel_row[0 .. kk) and its
// bitmap word by word (word_out(w, bits)).  Warp w walks a contiguous range of
// pages 32 at a time; one block scan of the per-warp counts places it.
template <typename KeyFn, typename WordOut>
__device__ void block_emit(const KeyFn& key, int P, uint32_t prefix, uint32_t mask, int need,
                           int32_t* sel_row, const WordOut& word_out, SelScratch& sc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int span = (P + 32 * kSelWarps - 1) / (32 * kSelWarps) * 32;
  const int j0 = warp * span, j1 = min(P, j0 + span);
  int gt = 0, eq = 0;
  for (int base = j0; base < j1; base += 32) {
    const int j = base + lane;
    const uint32_t k = (j < j1) ? (key(j) & mask) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, j < j1 && k > prefix));
    eq += __popc(__ballot_sync(0xffffffffu, j < j1 && k == prefix));
  }
  if (lane == 0) sc.warp_tot[warp] = (static_cast<long long>(gt) << 32) | eq;
  __syncthreads();
  long long before = 0;
  for (int w = 0; w < warp; ++w) before += sc.warp_tot[w];
  int gt_before = static_cast<int>(before >> 32);
  int eq_before = static_cast<int>(before & 0xffffffffll);
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = j0; base < j1; base += 32) {
    const int j = base + lane;
    const uint32_t k = (j < j1) ? (key(j) & mask) : 0u;
    const bool is_gt = j < j1 && k > prefix, is_eq = j < j1 && k == prefix;
    const uint32_t gtm = __ballot_sync(0xffffffffu, is_gt);
    const uint32_t eqm = __ballot_sync(0xffffffffu, is_eq);
    const int eq_rank = eq_before + __popc(eqm & lt);
    const bool sel = is_gt || (is_eq && eq_rank < need);
    const uint32_t selm = __ballot_sync(0xffffffffu, sel);
    if (sel) sel_row[gt_before + __popc(gtm & lt) + min(eq_rank, need)] = j;
    if (lane == 0) word_out(base >> 5, selm);
    gt_before += __popc(gtm);
    eq_before += __popc(eqm);
  }
  __syncthreads();  // the scratch may be reused
}

// The union of G heads' selection bitmaps (word(h, w)), ascending, with a bit
// per head: out[0 .. count) = (page, mask); *count_out = count.
template <typename WordFn>
__device__ void block_union(const WordFn& word, int G, int W32, int2* out, int* count_out,
                            SelScratch& sc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int span = (W32 + 32 * kSelWarps - 1) / (32 * kSelWarps) * 32;  // words per warp
  const int w0 = warp * span, w1 = min(W32, w0 + span);
  int cnt = 0;
  for (int wi = w0 + lane; wi < w1; wi += 32) {
    uint32_t u = 0;
    for (int h = 0; h < G; ++h) u |= word(h, wi);
    cnt += __popc(u);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
  if (lane == 0) sc.warp_tot[warp] = cnt;
  __syncthreads();
  int before = 0, total = 0;
  for (int w = 0; w < kSelWarps; ++w) {
    before += (w < warp) ? static_cast<int>(sc.warp_tot[w]) : 0;
    total += static_cast<int>(sc.warp_tot[w]);
  }
  for (int base = w0; base < w1; base += 32) {
    const int wi = base + lane;
    uint32_t hw[8];
    uint32_t u = 0;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      hw[h] = (h < G && wi < w1) ? word(h, wi) : 0u;
      u |= hw[h];
    }
    const int c = __popc(u);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    int pos = before + incl - c;
    while (u) {
      const int bit = __ffs(u) - 1;
      u &= u - 1;
      uint32_t m = 0;
#pragma unroll
      for (int h = 0; h < 8; ++h) m |= ((hw[h] >> bit) & 1u) << h;
      out[pos++] = make_int2(wi * 32 + bit, static_cast<int>(m));
    }
    before += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (threadIdx.x == 0) *count_out = total;
  __syncthreads();
}

// ---------------------------------------------------------------- kernels
template <int D, bool F16>
__global__ void __launch_bounds__(kScoreWarps * 32) score_kernel(const ScoreArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int page0 = blockIdx.x * kScorePagesPerCta + warp * 16;
  griddep_launch_dependents();
  griddep_wait();
  if (page0 >= a.P) return;
  uint32_t bq[D / 16][4];
  load_q_pm<D>(a.q, a.q_sb, a.q_sh, b, kvh, a.G, lane, bq);
  const int64_t mbase = (static_cast<int64_t>(b) * a.Hkv + kvh) * a.P * D;
  float acc[4];
  score_tile<D, F16>(bq, static_cast<const uint16_t*>(a.meta_max) + mbase,
                     static_cast<const uint16_t*>(a.meta_min) + mbase, page0, a.P, lane, acc);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int head = 2 * t4 + (e & 1);
    const int page = page0 + g + 8 * (e >> 1);
    if (head < a.G && page < a.P)
      a.scores[(static_cast<int64_t>(b) * a.Hq + kvh * a.G + head) * a.P + page] = acc[e];
  }
}

template <bool SMEM>
__global__ void __launch_bounds__(kSelThreads) topk_kernel(const TopkArgs a) {
  extern __shared__ uint32_t s_keys[];
  __shared__ SelScratch sc;
  const int row = blockIdx.x;
  griddep_launch_dependents();
  griddep_wait();  // the scores come from the previous kernel
  const float* r = a.scores + static_cast<int64_t>(row) * a.P;
  if constexpr (SMEM) {
    for (int j = threadIdx.x; j < a.P; j += kSelThreads) s_keys[j] = score_key(__ldcg(r + j));
    __syncthreads();
  }
  auto key = [&](int j) {
    if constexpr (SMEM) return s_keys[j];
    return score_key(__ldcg(r + j));
  };
  uint32_t* bits = a.bitmaps + static_cast<int64_t>(row) * a.W32;
  auto word_out = [&](int w, uint32_t v) { bits[w] = v; };
  uint32_t prefix, mask;
  int need;
  block_radix_select(key, a.P, a.kk, sc, prefix, mask, need);
  block_emit(key, a.P, prefix, mask, need, a.selected + static_cast<int64_t>(row) * a.kk,
             word_out, sc);
}

__global__ void __launch_bounds__(kSelThreads) union_kernel(const UnionArgs a) {
  __shared__ SelScratch sc;
  griddep_launch_dependents();
  griddep_wait();  // the bitmaps come from the previous kernel
  const int unit = blockIdx.x;
  const int b = unit / a.Hkv, kvh = unit % a.Hkv;
  const uint32_t* bm = a.bitmaps + (static_cast<int64_t>(b) * a.Hq + kvh * a.G) * a.W32;
  auto word = [&](int h, int w) { return __ldcg(bm + static_cast<int64_t>(h) * a.W32 + w); };
  block_union(word, a.G, a.W32, a.union_list + static_cast<int64_t>(unit) * a.union_stride,
              a.union_count + unit, sc);
}

// ------------------------------------------------------- one CTA per unit
// unit_select_kernel: the bound scores, per-head top-K and union of one
// (batch, kv head) in one CTA of kUnitWarps warps.  The scores stay in shared
// memory as order-preserving keys [G][P]; warp h selects head h (and h + 8)
// from them (select_warp.cuh); warp 0 then builds
// the union from the heads' bitmaps.  Scoring streams the unit's metadata with
// two 16-page tiles in flight per warp.
constexpr int kUnitWarps = 8;

template <int D, bool F16>
__global__ void __launch_bounds__(kUnitWarps * 32, 1) unit_select_kernel(const UnitSelectArgs a) {
  extern __shared__ __align__(16) uint8_t usm[];
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(usm);                     // [G][P]
  uint32_t* s_bm = s_keys + static_cast<size_t>(a.G) * a.P;                // [G][kSelBitmapWords]
  uint8_t* s_cand = reinterpret_cast<uint8_t*>(s_bm + a.G * kSelBitmapWords);  // per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int unit = blockIdx.x;
  const int b = unit / a.Hkv, kvh = unit % a.Hkv;
  griddep_launch_dependents();
  griddep_wait();
  uint32_t bq[D / 16][4];
  load_q_pm<D>(a.q, a.q_sb, a.q_sh, b, kvh, a.G, lane, bq);
  const int64_t mbase = static_cast<int64_t>(unit) * a.P * D;
  const uint16_t* mmax = static_cast<const uint16_t*>(a.meta_max) + mbase;
  const uint16_t* mmin = static_cast<const uint16_t*>(a.meta_min) + mbase;
  const int tiles = static_cast<int>(ceil_div(a.P, 16));
  for (int t = warp; t < tiles; t += 2 * kUnitWarps) {
    float acc0[4], acc1[4];
    const int t1 = t + kUnitWarps;
    score_tile2<D, F16>(bq, mmax, mmin, 16 * t, 16 * min(t1, tiles - 1), a.P, lane, acc0, acc1);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int head = 2 * t4 + (e & 1);
      const int p0 = 16 * t + g + 8 * (e >> 1), p1 = 16 * t1 + g + 8 * (e >> 1);
      if (head < a.G && p0 < a.P) s_keys[head * a.P + p0] = score_key(acc0[e]);
      if (head < a.G && t1 < tiles && p1 < a.P) s_keys[head * a.P + p1] = score_key(acc1[e]);
    }
  }
  __syncthreads();
  uint32_t* cand_key = reinterpret_cast<uint32_t*>(s_cand + warp * kCandCap * 6);
  uint16_t* cand_page = reinterpret_cast<uint16_t*>(s_cand + warp * kCandCap * 6 + kCandCap * 4);
  const int W = static_cast<int>(ceil_div(a.P, 32));
  for (int h = warp; h < a.G; h += kUnitWarps) {
    uint32_t* bm = s_bm + h * kSelBitmapWords;
    for (int w = lane; w < kSelBitmapWords; w += 32) bm[w] = 0u;
    __syncwarp();
    const uint32_t* keys = s_keys + h * a.P;
    warp_topk_head([keys](int j) { return keys[j]; }, a.P, a.kk, bm, cand_key, cand_page);
    __syncwarp();
    const int64_t row = static_cast<int64_t>(b) * a.Hq + kvh * a.G + h;
    warp_emit_row(bm, W, a.selected + row * a.kk, nullptr);
  }
  __syncthreads();
  if (warp == 0) {
    const int count = warp_union(s_bm, kSelBitmapWords, a.G, W,
                                 a.union_list + static_cast<int64_t>(unit) * a.union_stride,
                                 false);
    if (lane == 0) a.union_count[unit] = count;
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
    return launch_pdl(topk_kernel<true>, dim3(a.rows), dim3(kSelThreads), key_bytes, s, a);
  }
  return launch_pdl(topk_kernel<false>, dim3(a.rows), dim3(kSelThreads), 0, s, a);
}

size_t unit_select_smem(int G, int P) {
  return static_cast<size_t>(G) * P * 4 + static_cast<size_t>(G) * kSelBitmapWords * 4 +
         static_cast<size_t>(kUnitWarps) * kCandCap * 6;
}

cudaError_t launch_unit_select(int d, bool f16, const UnitSelectArgs& a, cudaStream_t s) {
  const size_t smem = unit_select_smem(a.G, a.P);
  const dim3 grid(a.B * a.Hkv), block(kUnitWarps * 32);
  auto kern = d == 128 ? (f16 ? unit_select_kernel<128, true> : unit_select_kernel<128, false>)
                       : (f16 ? unit_select_kernel<64, true> : unit_select_kernel<64, false>);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, block, smem, s, a);
}

cudaError_t launch_union(const UnionArgs& a, int units, cudaStream_t s) {
  return launch_pdl(union_kernel, dim3(units), dim3(kSelThreads), 0, s, a);
}

}  // namespace dkv

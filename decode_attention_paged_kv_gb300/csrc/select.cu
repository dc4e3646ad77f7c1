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

// The union of G heads' selection bitmaps (word(h, w)) over selection pages of
// S tokens, ascending, with a bit per head, each selection page written as its
// cache pages (S / 16 of them, fewer for the last page of a sequence of n
// tokens): out[0 .. count) = (cache page, mask); *count_out = count.
template <typename WordFn>
__device__ void block_union(const WordFn& word, int G, int W32, int S, int n, int2* out,
                            int* count_out, SelScratch& sc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int span = (W32 + 32 * kSelWarps - 1) / (32 * kSelWarps) * 32;  // words per warp
  const int w0 = warp * span, w1 = min(W32, w0 + span);
  const int msub = S / kPage, last = static_cast<int>(ceil_div(n, S)) - 1;
  auto pages_of = [&](uint32_t u, int wi) {  // cache pages of word wi's selection pages
    int c = __popc(u) * msub;
    if (wi == (last >> 5) && ((u >> (last & 31)) & 1u)) c -= msub - cache_pages_in(last, S, n);
    return c;
  };
  int cnt = 0;
  for (int wi = w0 + lane; wi < w1; wi += 32) {
    uint32_t u = 0;
    for (int h = 0; h < G; ++h) u |= word(h, wi);
    cnt += pages_of(u, wi);
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
    const int c = pages_of(u, wi);
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
      const int ps = wi * 32 + bit;
      const int k = msub == 1 ? 1 : cache_pages_in(ps, S, n);
      for (int i = 0; i < k; ++i) out[pos++] = make_int2(ps * msub + i, static_cast<int>(m));
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
  // One selection per kv head group: every row of the group sums the group's
  // scores, head by head in order, so the group's rows select identically.
  const int r0 = row - (row % a.Hq) % a.group;
  const float* r = a.scores + static_cast<int64_t>(r0) * a.P;
  auto score = [&](int j) {
    float s = __ldcg(r + j);
    for (int h = 1; h < a.group; ++h) s = __fadd_rn(s, __ldcg(r + static_cast<int64_t>(h) * a.P + j));
    return s;
  };
  if constexpr (SMEM) {
    for (int j = threadIdx.x; j < a.P; j += kSelThreads) s_keys[j] = score_key(score(j));
    __syncthreads();
  }
  auto key = [&](int j) {
    if constexpr (SMEM) return s_keys[j];
    return score_key(score(j));
  };
  uint32_t* bits = a.bitmaps + static_cast<int64_t>(row) * a.W32;
  auto word_out = [&](int w, uint32_t v) { bits[w] = v; };
  // a shorter sequence: its own pages only, and possibly fewer than kk kept
  const int Pb = static_cast<int>(ceil_div(seq_len_of(a.lens, row / a.Hq, a.N), a.S));
  const int kkb = min(a.kk, Pb);
  uint32_t prefix, mask;
  int need;
  block_radix_select(key, Pb, kkb, sc, prefix, mask, need);
  int32_t* sel_row = a.selected + static_cast<int64_t>(row) * a.kk;
  block_emit(key, Pb, prefix, mask, need, sel_row, word_out, sc);
  for (int w = static_cast<int>(ceil_div(Pb, 32)) + threadIdx.x; w < a.W32; w += kSelThreads)
    bits[w] = 0u;
  for (int i = kkb + threadIdx.x; i < a.kk; i += kSelThreads) sel_row[i] = -1;
}

__global__ void __launch_bounds__(kSelThreads) union_kernel(const UnionArgs a) {
  __shared__ SelScratch sc;
  griddep_launch_dependents();
  griddep_wait();  // the bitmaps come from the previous kernel
  const int unit = blockIdx.x;
  const int b = unit / a.Hkv, kvh = unit % a.Hkv;
  const uint32_t* bm = a.bitmaps + (static_cast<int64_t>(b) * a.Hq + kvh * a.G) * a.W32;
  auto word = [&](int h, int w) { return __ldcg(bm + static_cast<int64_t>(h) * a.W32 + w); };
  block_union(word, a.G, a.W32, a.S, seq_len_of(a.lens, b, a.N),
              a.union_list + static_cast<int64_t>(unit) * a.union_stride, a.union_count + unit,
              sc);
}

// ------------------------------------------------------- one CTA per unit
// unit_select_kernel: the bound scores, per-head top-K and union of one
// (batch, kv head) in one CTA.  Warp 8 streams the unit's metadata with TMA
// tensor copies, 64 pages of [M] and [m] per stage (128-byte swizzle); a stage
// goes to consumer warps 0-3 or 4-7 (alternately), each of which scores one
// 16-page tile of it on tensor cores: S[head][page] = q+ . M + q- . m, as in
// the score kernel but with the pages' metadata read by ldmatrix.  The scores
// stay in shared memory as order-preserving keys [G][P]; then warp h selects
// head h (select_warp.cuh); warps 0-3 build the union from the heads' bitmaps
// while warps 4-7 write the per-head rows.  Every wait is bounded.
constexpr int kUnitConsumers = 8;
constexpr int kUnitThreads = (kUnitConsumers + 1) * 32;
constexpr int kUnitBoxPages = 64;

template <int D>
struct UnitCfg {
  static constexpr int kBoxBytes = kUnitBoxPages * D * 2;  // one of [M] / [m]
  static constexpr int kStageBytes = 2 * kBoxBytes;
  static constexpr int kStages = (128 * 1024) / kStageBytes;  // 128 KiB in flight
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kKeysOffset = kBarOffset + 2 * kStages * 8 + 16;  // + abort flag
};

// Shared address of channels [c, c+8) of page row t of a metadata box
// {64 channels, 64 pages, D/64 halves} written with 128-byte swizzle.
__device__ __forceinline__ uint32_t box_addr(uint32_t base, int t, int c) {
  const int row = (c >> 6) * kUnitBoxPages + t;
  const int chunk = ((c & 63) >> 3) ^ (row & 7);
  return base + static_cast<uint32_t>(row * 128 + chunk * 16);
}

__device__ __forceinline__ void unit_consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kUnitConsumers * 32) : "memory");
}

// The union is built by warps 0-3 (warps 4-7 write the per-head rows meanwhile).
constexpr int kUnionWarps = 4;
__device__ __forceinline__ void union_sync() {
  asm volatile("bar.sync 2, %0;" ::"r"(kUnionWarps * 32) : "memory");
}

template <int D, bool F16>
__global__ void __launch_bounds__(kUnitThreads, 1)
    unit_select_kernel(const UnitSelectArgs a, const __grid_constant__ CUtensorMap mmx,
                       const __grid_constant__ CUtensorMap mmn) {
  using C = UnitCfg<D>;
  extern __shared__ uint8_t usm_raw[];
  uint8_t* usm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(usm_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(usm);
  const uint32_t full0 = sbase + C::kBarOffset, empty0 = full0 + 8 * C::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(usm + C::kBarOffset + 16 * C::kStages);
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(usm + C::kKeysOffset);      // [G][P]
  uint32_t* s_bm = s_keys + static_cast<size_t>(a.G) * a.P;                  // [G][kSelBitmapWords]
  // [0..7] / [8..15]: each head's largest / smallest key; [16] / [17]: the
  // group score's (one selection per group)
  uint32_t* s_kext = s_bm + static_cast<size_t>(a.G) * kSelBitmapWords;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;
  const int b = unit / a.Hkv, kvh = unit % a.Hkv;
  // selection pages of this sequence (all P without per-sequence lengths)
  const int Nb = seq_len_of(a.lens, b, a.N);
  const int Pb = static_cast<int>(ceil_div(Nb, a.S));
  const int n_boxes = static_cast<int>(ceil_div(Pb, kUnitBoxPages));
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 4);  // the four warps that score the stage
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < 18) s_kext[threadIdx.x] = (threadIdx.x < 8 || threadIdx.x == 16) ? 0u : ~0u;
  if (warp == kUnitConsumers && lane == 0) {
    prefetch_tensormap(&mmx);
    prefetch_tensormap(&mmn);
  }
  griddep_launch_dependents();
  griddep_wait();
  __syncthreads();

  if (warp == kUnitConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (int i = 0; i < n_boxes; ++i) {
        const int s = i % C::kStages;
        if (i >= C::kStages &&
            !mbar_wait_bounded(empty0 + 8 * s, ((i / C::kStages) - 1) & 1, a.wait_limit_ns,
                               abort_flag)) {
          if (*abort_flag == 0) {
            set_status(a.status, kStatusTimeout);
            *abort_flag = 1;
          }
          break;
        }
        const uint32_t dst = sbase + s * C::kStageBytes;
        mbar_arrive_expect_tx(full0 + 8 * s, C::kStageBytes);
        tma_load_5d_hint(dst, &mmx, full0 + 8 * s, 0, i * kUnitBoxPages, 0, kvh, b, pol);
        tma_load_5d_hint(dst + C::kBoxBytes, &mmn, full0 + 8 * s, 0, i * kUnitBoxPages, 0, kvh, b,
                         pol);
        issued = i + 1;
      }
      // The last copies issued have landed before this warp leaves (so no copy
      // is still writing when the consumers stop early); each wait is bounded.
      const uint64_t deadline = globaltimer_ns() + 200000000ull;
      for (int j = max(0, issued - C::kStages); j < issued; ++j) {
        const uint64_t now = globaltimer_ns();
        if (now >= deadline) break;
        mbar_wait_bounded(full0 + 8 * (j % C::kStages), (j / C::kStages) & 1, deadline - now,
                          nullptr);
      }
    }
    return;
  }

  // -------------------------------------------------------------- scoring
  const int g = lane >> 2, t4 = lane & 3;
  const bool head_ok = g < a.G;
  const int mtx = lane >> 3, mrow = lane & 7;
  uint32_t qp[D / 16][2], qm[D / 16][2];  // A fragments of q+ and q- (rows = heads)
  {
    const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + b * a.q_sb +
                           static_cast<int64_t>(kvh * a.G + (head_ok ? g : 0)) * a.q_sh;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint32_t w0 =
          head_ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t4) : 0u;
      const uint32_t w1 =
          head_ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t4 + 8) : 0u;
      qp[ks][0] = keep_sign(w0, false);
      qm[ks][0] = keep_sign(w0, true);
      qp[ks][1] = keep_sign(w1, false);
      qm[ks][1] = keep_sign(w1, true);
    }
  }
  const int half = warp >> 2, tile = warp & 3;  // boxes of parity `half`, tile `tile` of each
  bool ok = true;
  uint32_t kmx = 0u, kmn = ~0u;  // extremes of head g's keys this lane wrote
  for (int i = half; i < n_boxes; i += 2) {
    const int s = i % C::kStages;
    ok = mbar_wait_bounded(full0 + 8 * s, (i / C::kStages) & 1, a.wait_limit_ns, abort_flag);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    const uint32_t mb = sbase + s * C::kStageBytes, nb = mb + C::kBoxBytes;
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t r0, r1, r2, r3;
      const int row = 16 * tile + 8 * (mtx >> 1) + mrow, ch = 16 * ks + 8 * (mtx & 1);
      ldsm_x4(box_addr(mb, row, ch), r0, r1, r2, r3);
      mma16816<F16>(sc[0], qp[ks][0], 0u, qp[ks][1], 0u, r0, r1);
      mma16816<F16>(sc[1], qp[ks][0], 0u, qp[ks][1], 0u, r2, r3);
      ldsm_x4(box_addr(nb, row, ch), r0, r1, r2, r3);
      mma16816<F16>(sc[0], qm[ks][0], 0u, qm[ks][1], 0u, r0, r1);
      mma16816<F16>(sc[1], qm[ks][0], 0u, qm[ks][1], 0u, r2, r3);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    if (head_ok) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int p = i * kUnitBoxPages + 16 * tile + 8 * (e >> 1) + 2 * t4 + (e & 1);
        if (p < Pb) {
          const uint32_t key = score_key(sc[e >> 1][e & 1]);
          s_keys[g * a.P + p] = key;
          kmx = max(kmx, key);
          kmn = min(kmn, key);
        }
      }
    }
  }
  // each head's largest and smallest key, for the selection's common prefix
  kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, 1));
  kmx = max(kmx, __shfl_xor_sync(0xffffffffu, kmx, 2));
  kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, 1));
  kmn = min(kmn, __shfl_xor_sync(0xffffffffu, kmn, 2));
  if (head_ok && t4 == 0) {
    atomicMax(s_kext + g, kmx);
    atomicMin(s_kext + 8 + g, kmn);
  }
  // (a warp that timed out tells the others through the abort flag)
  if (!ok && lane == 0 && *abort_flag == 0) {
    set_status(a.status, kStatusTimeout);
    *abort_flag = 1;
  }
  unit_consumers_sync();
  if (*abort_flag) {
    if (threadIdx.x == 0) a.union_count[unit] = 0;  // gather nothing for this unit
    return;
  }

  // ------------------------------------------------------------ selection
  const int W = static_cast<int>(ceil_div(Pb, 32));
  const int kkb = min(a.kk, Pb);  // pages kept (a shorter sequence may have fewer than kk)
  if (a.group) {
    // One selection per group: page j's key becomes that of the heads' scores
    // summed in head order (row 0 of the keys; only this thread reads or
    // writes page j).
    uint32_t gmx = 0u, gmn = ~0u;
    for (int j = threadIdx.x; j < Pb; j += kUnitConsumers * 32) {
      float sum = key_score(s_keys[j]);
      for (int h = 1; h < a.G; ++h) sum = __fadd_rn(sum, key_score(s_keys[h * a.P + j]));
      const uint32_t k = score_key(sum);
      s_keys[j] = k;
      gmx = max(gmx, k);
      gmn = min(gmn, k);
    }
    gmx = __reduce_max_sync(0xffffffffu, gmx);
    gmn = __reduce_min_sync(0xffffffffu, gmn);
    if (lane == 0) {
      atomicMax(s_kext + 16, gmx);
      atomicMin(s_kext + 17, gmn);
    }
    unit_consumers_sync();
  }
  const int n_sel = a.group ? 1 : a.G;  // selections: one per head, or one per group
  for (int h = warp; h < n_sel; h += kUnitConsumers) {
    uint32_t* bm = s_bm + h * kSelBitmapWords;
    const uint32_t* keys = s_keys + h * a.P;
    warp_topk_head([keys](int j) { return keys[j]; }, Pb, kkb, bm,
                   s_kext[a.group ? 16 : h], s_kext[a.group ? 17 : 8 + h]);
  }
  unit_consumers_sync();
  if (warp >= kUnionWarps) {
    // Warps 4-7 write each head's ascending row while warps 0-3 build the union.
    for (int h = warp - kUnionWarps; h < a.G; h += kUnitConsumers - kUnionWarps) {
      const int64_t row = static_cast<int64_t>(b) * a.Hq + kvh * a.G + h;
      warp_emit_row(s_bm + (a.group ? 0 : h) * kSelBitmapWords, W, a.selected + row * a.kk,
                    nullptr);
      for (int i = kkb + lane; i < a.kk; i += 32) a.selected[row * a.kk + i] = -1;
    }
    return;
  }
  // Union of the heads' bitmaps, ascending, with a bit per head: warp w ORs
  // words w * wpw .. (one per lane), the per-warp counts place them.  Each
  // selection page becomes its S / 16 cache pages (fewer for the sequence's
  // last).
  {
    const int wpw = static_cast<int>(ceil_div(W, kUnionWarps));
    const int wi = warp * wpw + lane;
    const bool own = lane < wpw && wi < W;
    uint32_t hw[8];
    uint32_t u = 0;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      hw[h] = (own && h < a.G) ? s_bm[(a.group ? 0 : h) * kSelBitmapWords + wi] : 0u;
      u |= hw[h];
    }
    const int msub = a.S / kPage;  // cache pages per selection page
    const int last = Pb - 1;
    int c = __popc(u) * msub;
    if (own && wi == (last >> 5) && ((u >> (last & 31)) & 1u))
      c -= msub - cache_pages_in(last, a.S, Nb);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    int* wtot = reinterpret_cast<int*>(s_keys);  // (the keys are no longer needed)
    if (lane == 31) wtot[warp] = incl;
    union_sync();
    int before = 0, count = 0;
#pragma unroll
    for (int v = 0; v < kUnionWarps; ++v) {
      before += v < warp ? wtot[v] : 0;
      count += wtot[v];
    }
    int2* out = a.union_list + static_cast<int64_t>(unit) * a.union_stride;
    int at = before + incl - c;
    auto put = [&](int ps, uint32_t m) {  // selection page ps -> its cache pages
      const int n = msub == 1 ? 1 : cache_pages_in(ps, a.S, Nb);
      for (int i = 0; i < n; ++i) out[at++] = make_int2(ps * msub + i, static_cast<int>(m));
    };
    if (a.G <= 4) {
      while (u) {
        const int bit = __ffs(u) - 1;
        u &= u - 1;
        uint32_t m = 0;
#pragma unroll
        for (int h = 0; h < 4; ++h) m |= ((hw[h] >> bit) & 1u) << h;
        put(wi * 32 + bit, m);
      }
    } else {
      while (u) {
        const int bit = __ffs(u) - 1;
        u &= u - 1;
        uint32_t m = 0;
#pragma unroll
        for (int h = 0; h < 8; ++h) m |= ((hw[h] >> bit) & 1u) << h;
        put(wi * 32 + bit, m);
      }
    }
    if (threadIdx.x == 0) a.union_count[unit] = count;
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

size_t unit_select_smem(int d, int G, int P) {
  const size_t keys_off = d == 128 ? UnitCfg<128>::kKeysOffset : UnitCfg<64>::kKeysOffset;
  return 1024 + keys_off + static_cast<size_t>(G) * P * 4 +
         static_cast<size_t>(G) * kSelBitmapWords * 4 + 32 * 4;
}

cudaError_t launch_unit_select(int d, bool f16, const UnitSelectArgs& a, const CUtensorMap& mmx,
                               const CUtensorMap& mmn, cudaStream_t s) {
  const size_t smem = unit_select_smem(d, a.G, a.P);
  const dim3 grid(a.B * a.Hkv), block(kUnitThreads);
  auto kern = d == 128 ? (f16 ? unit_select_kernel<128, true> : unit_select_kernel<128, false>)
                       : (f16 ? unit_select_kernel<64, true> : unit_select_kernel<64, false>);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, block, smem, s, a, mmx, mmn);
}

cudaError_t launch_union(const UnionArgs& a, int units, cudaStream_t s) {
  return launch_pdl(union_kernel, dim3(units), dim3(kSelThreads), 0, s, a);
}

}  // namespace dkv

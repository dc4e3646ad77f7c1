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
// order-preserving 32-bit keys, most significant bits first -- one bit at a
// time by a warp over keys in registers (select_warp.cuh) or by a block; for
// long rows a sample bracket first narrows the K-th key to a bucket of a few
// thousand keys, searched with 8-bit digits -- then the selected pages in
// ascending order; among equal scores the lower page index is taken first.
//
// Union: the pages any query head of a group selected, ascending, each with a
// bit per head that chose it -- the list the sparse attention gathers (each
// page once for the whole group).
//
// Contexts of 256 to 2048 pages: unit_select_kernel does all three for a
// (batch, kv head) in one CTA.  Otherwise three kernels, chained with
// programmatic dependent launch: score_kernel (scores to global memory),
// topk_kernel (one CTA per (b, h): selection and its bitmap) and
// union_kernel (one CTA per (batch, kv head)).

#include <math.h>

#include "select_warp.cuh"
#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {
namespace {

constexpr int kScoreWarps = 4;
constexpr int kScorePagesPerCta = 16 * kScoreWarps;
// Top-K and union CTAs: up to kSelMaxThreads threads (the block functions
// read the block's size at run time; shared scratch is laid out for the most).
constexpr int kSelMaxThreads = 1024;
constexpr int kSelMaxWarps = kSelMaxThreads / 32;
static_assert(kSelMaxWarps <= 32, "one warp partial a lane");
__device__ __forceinline__ int sel_threads() { return static_cast<int>(blockDim.x); }
__device__ __forceinline__ int sel_warps() { return static_cast<int>(blockDim.x) >> 5; }

// Per-warp partials part[0 .. warps) summed by every warp, one partial a
// lane: over all warps, or over the warps before the calling one.
__device__ __forceinline__ int warps_total(const uint32_t* part) {
  const int lane = threadIdx.x & 31;
  return __reduce_add_sync(0xffffffffu, lane < sel_warps() ? static_cast<int>(part[lane]) : 0);
}
__device__ __forceinline__ int warps_before(const uint32_t* part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  return __reduce_add_sync(0xffffffffu, lane < warp ? static_cast<int>(part[lane]) : 0);
}
constexpr size_t kTopkSmemKeyBytes = 160 * 1024;  // stage rows of up to 40960 pages

// B operand of the score MMA for lane (g, t4): [q+ | q-] of query head g of the
// group (zero for g >= G).  The contraction index runs over the concatenation
// [M | m]; the lane owns 16-byte chunks c = t4 + 4 s of it, two k-steps each.
// EXACT: plain q over the d channels (rows of single keys, m = M = k: the
// bound is the dot product itself, computed once).
template <int D, bool EXACT = false>
__device__ __forceinline__ void load_q_pm(const void* q, int64_t q_sb, int64_t q_sh, int b,
                                          int kvh, int G, int lane,
                                          uint32_t (&bq)[D / 16][4]) {
  const int g = lane >> 2, t4 = lane & 3;
  const bool hv = g < G;
  const uint16_t* qrow = static_cast<const uint16_t*>(q) + b * q_sb +
                         static_cast<int64_t>(kvh * G + (hv ? g : 0)) * q_sh;
  if constexpr (EXACT) {
#pragma unroll
    for (int s = 0; s < D / 32; ++s) {
      const uint4 w = hv ? *reinterpret_cast<const uint4*>(qrow + 8 * (t4 + 4 * s))
                         : make_uint4(0, 0, 0, 0);
      bq[s][0] = w.x;
      bq[s][1] = w.y;
      bq[s][2] = w.z;
      bq[s][3] = w.w;
    }
  } else {
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
}

// Bound scores of pages page0 .. page0+15 (< P) of one (batch, kv head) for the
// group's query heads: acc = [page g][head 2t4], [g][2t4+1], [g+8][2t4],
// [g+8][2t4+1].  mmax / mmin point at the unit's [P, d] metadata.
template <int D, bool F16, bool EXACT = false>
__device__ __forceinline__ void score_tile(const uint32_t (&bq)[D / 16][4], const uint16_t* mmax,
                                           const uint16_t* mmin, int page0, int P, int lane,
                                           float (&acc)[4]) {
  const int g = lane >> 2, t4 = lane & 3;
  constexpr int NS = EXACT ? D / 32 : D / 16;  // 16-byte chunks a lane contracts
  // Every load is issued before the first MMA (rows past P read a valid page
  // and are zeroed afterwards), so a lane has 2 NS 16-byte loads in flight.
  uint4 ra[2][D / 16];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int page = min(page0 + g + 8 * hr, P - 1);
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      const int c = t4 + 4 * s;
      const uint16_t* src = (EXACT || c < D / 8)
                                ? mmax + static_cast<int64_t>(page) * D + 8 * c
                                : mmin + static_cast<int64_t>(page) * D + 8 * (c - D / 8);
      ra[hr][s] = __ldg(reinterpret_cast<const uint4*>(src));
    }
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    if (page0 + g + 8 * hr >= P) {
#pragma unroll
      for (int s = 0; s < NS; ++s) ra[hr][s] = make_uint4(0, 0, 0, 0);
    }
  }
  acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    mma16816<F16>(acc, ra[0][s].x, ra[1][s].x, ra[0][s].y, ra[1][s].y, bq[s][0], bq[s][1]);
    mma16816<F16>(acc, ra[0][s].z, ra[1][s].z, ra[0][s].w, ra[1][s].w, bq[s][2], bq[s][3]);
  }
}

constexpr int kSelCompCap = 4096;  // bucket keys the block top-K compacts
struct SelScratch {
  uint32_t hist[256];
  uint32_t warp_gt[kSelMaxWarps];      // per-warp counts (emit: keys > prefix,
  uint32_t warp_eq[kSelMaxWarps];      // == prefix; union: pages)
  uint32_t res[4];                     // the bucket search's verdicts
  uint32_t comp[kSelCompCap];
};

// Stores v at p (global) or addr (shared) when c holds: one predicated store,
// so a warp whose lanes differ on c takes no branch.
__device__ __forceinline__ void st_global_if(void* p, uint32_t v, bool c) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.global.u32 [%0], %1;\n\t}"
               :
               : "l"(p), "r"(v), "r"(static_cast<uint32_t>(c))
               : "memory");
}
__device__ __forceinline__ void st_shared_if(uint32_t addr, uint32_t v, bool c) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.shared.u32 [%0], %1;\n\t}"
               :
               : "r"(addr), "r"(v), "r"(static_cast<uint32_t>(c))
               : "memory");
}

// Selection (by the whole block) of the kk largest of P keys: the K-th
// largest key found bit by bit below the keys' common prefix (radix selection
// with 1-bit digits, as the per-head warp top-K), every pass one count over the
// block, stopping as soon as exactly kk keys are >= the candidate.  On return:
// keys with (key & mask) > prefix are selected, and of the keys with
// (key & mask) == prefix the first `need` in index order.
template <typename KeyFn>
__device__ void block_radix_select(const KeyFn& key, int P, int kk, SelScratch& sc,
                                   uint32_t& prefix, uint32_t& mask, int& need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* wcnt = sc.hist;            // per-warp counts
  uint32_t* wmax = sc.hist + kSelMaxWarps;
  uint32_t* wmin = sc.hist + 2 * kSelMaxWarps;
  const int nt = sel_threads(), nw = sel_warps();
  // the keys' largest and smallest: the bits they all share are skipped
  uint32_t mx = 0u, mn = ~0u;
  for (int j = tid; j < P; j += nt) {
    const uint32_t k = key(j);
    mx = max(mx, k);
    mn = min(mn, k);
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  if (lane == 0) {
    wmax[warp] = mx;
    wmin[warp] = mn;
  }
  __syncthreads();
  const uint32_t kmax = __reduce_max_sync(0xffffffffu, lane < nw ? wmax[lane] : 0u);
  const uint32_t kmin = __reduce_min_sync(0xffffffffu, lane < nw ? wmin[lane] : ~0u);
  __syncthreads();
  // keys >= x over the block (four partial sums a thread, then warps in order)
  auto block_sum = [&](int mine) {
    const int wsum = __reduce_add_sync(0xffffffffu, mine);
    if (lane == 0) wcnt[warp] = static_cast<uint32_t>(wsum);
    __syncthreads();
    const int tot = warps_total(wcnt);
    __syncthreads();
    return tot;
  };
  auto count_ge = [&](uint32_t x) {
    int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
    int j = tid;
    for (; j + 3 * nt < P; j += 4 * nt) {
      c0 -= minus_borrow(key(j), x);
      c1 -= minus_borrow(key(j + nt), x);
      c2 -= minus_borrow(key(j + 2 * nt), x);
      c3 -= minus_borrow(key(j + 3 * nt), x);
    }
    for (; j < P; j += nt) c0 -= minus_borrow(key(j), x);
    const int below = (c0 + c1) + (c2 + c3);
    return block_sum(max(static_cast<int>(ceil_div(P - tid, nt)), 0) - below);
  };
  // Once the keys that agree with the bits fixed so far (the bucket) are few,
  // they are copied to sc.comp; counts are then `base` (keys above the bucket)
  // plus the bucket's keys >= x.
  int ncomp = -1, base = 0;
  auto count_comp = [&](uint32_t x) {
    int c = 0;
    for (int j = tid; j < ncomp; j += nt) c -= minus_borrow(sc.comp[j], x);
    return base + block_sum(max(static_cast<int>(ceil_div(ncomp - tid, nt)), 0) - c);
  };
  uint32_t T;
  int ge = -1;
  if (kmax == kmin) {
    T = kmax;  // all equal: a tie at T
  } else {
    const int top = 31 - __clz(kmax ^ kmin);
    T = top == 31 ? 0u : (kmax >> (top + 1)) << (top + 1);
    int geT = P, above = 0;  // keys >= T; keys above the bucket
    for (int bit = top; bit >= 0; --bit) {
      if (ncomp < 0 && geT - above <= kSelCompCap) {
        // the bucket: keys whose bits above `bit` equal T's; each thread
        // counts its own, a block scan places them, then each writes its own
        const int sh = bit + 1;
        auto in_bucket = [&](uint32_t k) { return sh == 32 || (k >> sh) == (T >> sh); };
        int mine = 0;
        for (int j = tid; j < P; j += nt) mine += in_bucket(key(j)) ? 1 : 0;
        int incl = mine;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += t;
        }
        if (lane == 31) wcnt[warp] = static_cast<uint32_t>(incl);
        __syncthreads();
        int at = incl - mine + warps_before(wcnt);
        ncomp = warps_total(wcnt);
        for (int j = tid; j < P; j += nt) {
          const uint32_t k = key(j);
          if (in_bucket(k)) sc.comp[at++] = k;
        }
        base = above;
        __syncthreads();
      }
      const uint32_t cand = T | (1u << bit);
      const int c = ncomp >= 0 ? count_comp(cand) : count_ge(cand);
      if (c >= kk) {
        T = cand;
        ge = geT = c;
        if (c == kk) break;
      } else {
        above = c;
      }
    }
  }
  mask = ~0u;
  if (ge == kk) {
    // exactly kk keys are >= T (T >= 1 here): all of them
    prefix = T - 1u;
    need = 0;
  } else {
    // a tie at the kk-th key T: the keys above T, then the first equal ones
    const int gt = T == ~0u ? 0 : (ncomp >= 0 ? count_comp(T + 1u) : count_ge(T + 1u));
    prefix = T;
    need = kk - gt;
  }
}

// Warp w of block_emit takes pages [w span, (w + 1) span).
__device__ __forceinline__ int emit_span(int P) {
  return (P + 32 * sel_warps() - 1) / (32 * sel_warps()) * 32;
}

constexpr int kSampleMinP = 4096;

// The sample ranks of the two splitters for kk of P keys: hi at rank r_hi
// (none when r_hi < 1), lo at rank r_lo; false when r_lo passes the sample.
__device__ __forceinline__ bool sample_ranks(int kk, int P, int& r_hi, int& r_lo) {
  const float pk = static_cast<float>(kk) / static_cast<float>(P);
  const float rho = 1024.f * pk, margin = 3.f * sqrtf(1024.f * pk * (1.f - pk)) + 8.f;
  r_hi = static_cast<int>(floorf(rho - margin));
  r_lo = static_cast<int>(ceilf(rho + margin));
  return r_lo <= 1024;
}

// One warp: the splitter of rank r among 1024 sampled keys (sample i = 32 m +
// lane is key i * stride + lane % stride, stride = P / 1024), to *out; ~0 when
// r < 1 (no upper splitter).  The keys are those of the score rows r, r + rs,
// ... (group of them summed in order, as the staged keys), fetched sixteen a
// lane at a time through stash[0 .. 1024) (shared memory).
__device__ void sample_splitter(const float* r, int64_t rs, int group, int P, int rank,
                                uint32_t* stash, uint32_t* out) {
  const int lane = threadIdx.x & 31;
  const int stride = P >> 10;
  const int off = lane % stride;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    float v[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) v[m] = __ldcg(r + (32 * (16 * b + m) + lane) * stride + off);
    for (int h = 1; h < group; ++h) {
      const float* rh = r + h * rs;
#pragma unroll
      for (int m = 0; m < 16; ++m)
        v[m] = __fadd_rn(v[m], __ldcg(rh + (32 * (16 * b + m) + lane) * stride + off));
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) stash[32 * (16 * b + m) + lane] = score_key(v[m]);
  }
  __syncwarp();
  uint32_t smp[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) smp[m] = stash[32 * m + lane];
  uint32_t smax = 0u, smin = ~0u;
#pragma unroll
  for (int m = 0; m < 32; ++m) {
    smax = max(smax, smp[m]);
    smin = min(smin, smp[m]);
  }
  smax = __reduce_max_sync(0xffffffffu, smax);
  smin = __reduce_min_sync(0xffffffffu, smin);
  uint32_t t = ~0u;
  if (rank >= 1) {
    if (smax == smin) {
      t = smax;
    } else {
      const int top = 31 - __clz(smax ^ smin);
      const uint32_t t0 = top == 31 ? 0u : (smax >> (top + 1)) << (top + 1);
      int ge;
      t = warp_threshold(smp, rank, rank + 2, ge, t0, top);
    }
  }
  if (lane == 0) *out = t;
}

// Where the two splitters sit in SelScratch::hist (hi, then lo).
constexpr int kSplitOffset = 2 * kSelMaxWarps;

// Block top-K of P >= kSampleMinP keys (load4(q): keys 4 q .. 4 q + 3, zero
// from P up to a multiple of 4; staged in shared memory or read from the
// score row) by a sample bracket.  1024 keys, one from each
// of 1024 equal windows, give two splitters lo < hi between which the kk-th
// largest key most likely lies: the sample ranks of that key's expected
// place, kk * 1024 / P, minus and plus three binomial standard deviations and
// 8 (sample_splitter, run by two warps while the others stage the keys, leaves
// them in sc.hist + kSplitOffset).  One pass over the
// keys counts A = #(>= hi) and the bucket [lo, hi); when A < kk <= A +
// #bucket and the bucket fits kSelCompCap, a second pass copies the bucket out
// and the bit search runs on the bucket alone (counts are A plus the bucket's
// keys >= x).  Otherwise it returns false, having written nothing, and the
// full search runs.  The splitters only decide which keys are compacted, so
// the selection is the same exact one either way.  Output as
// block_radix_select, plus block_emit's per-warp counts in sc.warp_gt and
// sc.warp_eq (the passes walk the keys in block_emit's warp ranges).
template <typename Load4>
__device__ bool block_sample_select(const Load4& load4, int P, int kk, SelScratch& sc,
                                    uint32_t& prefix, uint32_t& mask, int& need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* wcnt = sc.hist;               // per-warp bucket counts
  uint32_t* wabove = sc.hist + kSelMaxWarps;  // per-warp counts of keys >= hi
  const uint32_t* split = sc.hist + kSplitOffset;
  const uint32_t hi = split[0], lo = max(split[1], 1u);
  // pass 1: keys >= hi and keys in [lo, hi) (zero padding is below both);
  // warp w takes the keys block_emit gives it, four at a time
  const int span = emit_span(P);
  const int q0 = (warp * span) >> 2, q1 = (min(P, warp * span + span) + 3) >> 2;
  int below_hi = 0, inb = 0, seen = 0;
  auto tally = [&](uint32_t k) {
    const int bh = minus_borrow(k, hi), bl = minus_borrow(k, lo);
    below_hi -= bh;
    inb += bl - bh;
  };
  for (int j = q0 + lane; j < q1; j += 32) {
    const uint4 v = load4(j);
    tally(v.x);
    tally(v.y);
    tally(v.z);
    tally(v.w);
    seen += 4;
  }
  int incl = inb;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  const int wa = __reduce_add_sync(0xffffffffu, seen - below_hi);
  if (lane == 31) wcnt[warp] = static_cast<uint32_t>(incl);
  if (lane == 0) wabove[warp] = static_cast<uint32_t>(wa);
  __syncthreads();
  int at = incl - inb + warps_before(wcnt);
  const int nb = warps_total(wcnt), A = warps_total(wabove);
  const int my_above = static_cast<int>(wabove[warp]);
  __syncthreads();
  if (!(A < kk && kk <= A + nb && nb <= kSelCompCap)) return false;
  const int my0 = at, my1 = at + inb;  // this thread's bucket keys in sc.comp
  // pass 2: the bucket to sc.comp (in any order)
  const uint32_t comp = smem_u32(sc.comp);
  auto put = [&](uint32_t k) {
    const bool in = k >= lo && k < hi;
    st_shared_if(comp + 4u * static_cast<uint32_t>(at), k, in);
    at += in ? 1 : 0;
  };
  for (int j = q0 + lane; j < q1; j += 32) {
    const uint4 v = load4(j);
    put(v.x);
    put(v.y);
    put(v.z);
    put(v.w);
  }
  __syncthreads();
  // The (kk - A)-th largest bucket key T by radix selection over the bucket,
  // 8 bits a pass below the bits all bucket keys share (those of lo and
  // hi - 1), by the whole block: a shared histogram of the next digit of the
  // keys that agree with T so far, then warp 0 finds the digit holding the
  // rank (and zeroes the histogram for the next pass).  After the last pass r
  // is T's rank among the keys equal to it and cnt their number.
  uint32_t* hist = sc.hist;
  for (int i = tid; i < 256; i += sel_threads()) hist[i] = 0u;
  const uint32_t hm1 = hi - 1u;
  const int top = lo == hm1 ? -1 : 31 - __clz(lo ^ hm1);  // highest bit that may differ
  uint32_t fixed = top < 0 ? ~0u : (top >= 31 ? 0u : ~((2u << top) - 1u));  // bits settled
  uint32_t T = lo & fixed;
  int r = kk - A, cnt = nb;
  __syncthreads();
  for (int hb = top; hb >= 0; hb -= 8) {
    const int lb = hb >= 7 ? hb - 7 : 0;
    const uint32_t dmask = (2u << (hb - lb)) - 1u;
    for (int j = tid; j < nb; j += sel_threads()) {
      const uint32_t k = sc.comp[j];
      if ((k & fixed) == T) atomicAdd(hist + ((k >> lb) & dmask), 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds digits 8 l .. 8 l + 7; the digit d where the count of
      // digits >= d first reaches r, counting from the top
      uint32_t h[8];
      int tot = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        h[e] = hist[8 * lane + e];
        hist[8 * lane + e] = 0u;
        tot += static_cast<int>(h[e]);
      }
      int incl = tot;  // digits of this lane and the lanes above
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_down_sync(0xffffffffu, incl, off);
        if (lane + off < 32) incl += t;
      }
      const int above = incl - tot;
      if (above < r && r <= incl) {  // exactly one lane
        int run = above, d = 0;
        uint32_t hd = 0u;
        bool found = false;
#pragma unroll
        for (int e = 7; e >= 0; --e) {
          if (!found && run + static_cast<int>(h[e]) >= r) {
            found = true;
            d = e;
            hd = h[e];
          } else if (!found) {
            run += static_cast<int>(h[e]);
          }
        }
        sc.res[0] = static_cast<uint32_t>(8 * lane + d);
        sc.res[1] = static_cast<uint32_t>(r - run);
        sc.res[2] = hd;
      }
    }
    __syncthreads();
    T |= sc.res[0] << lb;
    r = static_cast<int>(sc.res[1]);
    cnt = static_cast<int>(sc.res[2]);
    fixed |= dmask << lb;
  }
  // keys > T, and of the cnt keys equal to T the first r: all of them when
  // r == cnt (then the selection is every key >= T, T >= lo >= 1)
  mask = ~0u;
  prefix = r == cnt ? T - 1u : T;
  need = r == cnt ? 0 : r;
  // block_emit's per-warp counts: keys > prefix are the warp's keys >= hi and
  // its bucket keys > prefix (prefix >= lo - 1); keys == prefix matter only
  // when need > 0, where prefix = T >= lo and they all lie in the bucket
  int gt = 0, eq = 0;
  for (int i = my0; i < my1; ++i) {
    const uint32_t k = sc.comp[i];
    gt += k > prefix ? 1 : 0;
    eq += k == prefix ? 1 : 0;
  }
  gt = __reduce_add_sync(0xffffffffu, gt) + my_above;
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (lane == 0) {
    sc.warp_gt[warp] = static_cast<uint32_t>(gt);
    sc.warp_eq[warp] = static_cast<uint32_t>(eq);
  }
  __syncthreads();
  return true;
}

// block_emit's first pass: per warp, the keys > prefix and == prefix, to
// sc.warp_gt and sc.warp_eq.
template <typename KeyFn>
__device__ void block_emit_counts(const KeyFn& key, int P, uint32_t prefix, uint32_t mask,
                                  SelScratch& sc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int span = emit_span(P);
  const int j0 = warp * span, j1 = min(P, j0 + span);
  int gt = 0, eq = 0;
  for (int base = j0; base < j1; base += 256) {
    uint32_t k[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = base + 32 * u + lane;
      k[u] = j < j1 ? key(j) & mask : 0u;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = base + 32 * u + lane;
      gt += (j < j1 && k[u] > prefix) ? 1 : 0;
      eq += (j < j1 && k[u] == prefix) ? 1 : 0;
    }
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (lane == 0) {
    sc.warp_gt[warp] = static_cast<uint32_t>(gt);
    sc.warp_eq[warp] = static_cast<uint32_t>(eq);
  }
  __syncthreads();
}

// Writes the selection in ascending page order to sel_row[0 .. kk) and its
// bitmap to bits[0 .. ceil(P / 32)), given the per-warp counts in
// sc.warp_gt / sc.warp_eq.  Warp w walks its range 256 keys at a time; the
// counts of the warps before it place it.  load4(q): keys 4 q .. 4 q + 3 (zero
// from P up to a multiple of 4), called for q < ceil(P / 4) only.  Without a
// partial tie (no key equal to the prefix is left out) a page is selected by
// its own key alone.
template <typename KeyFn, typename Load4>
__device__ void block_emit(const KeyFn& key, const Load4& load4, int P, uint32_t prefix,
                           uint32_t mask, int need, int32_t* sel_row, uint32_t* bits,
                           SelScratch& sc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int span = emit_span(P);
  const int j0 = warp * span, j1 = min(P, j0 + span);
  int gt_before = warps_before(sc.warp_gt);
  int eq_before = warps_before(sc.warp_eq);
  const uint32_t lt = (1u << lane) - 1u;
  if (need == 0 || need == warps_total(sc.warp_eq)) {
    // every key > prefix, and the keys == prefix all or none (need == 0 only
    // with prefix = T - 1 for a T >= 1, so prefix + 1 does not wrap)
    int at = gt_before + (need == 0 ? 0 : eq_before);
    const uint32_t cut = need == 0 ? prefix + 1u : prefix;  // selected: key & mask >= cut
    // lane l takes the 8 keys base + 8 l .. base + 8 l + 7: one count, one
    // warp scan and one bitmap byte a lane per 256 keys
    const int pad = 4 * static_cast<int>(ceil_div(P, 4));  // keys with zero padding
    for (int base = j0; base < j1; base += 256) {
      const int jb = base + 8 * lane;  // a multiple of 8
      uint32_t k[8];
      const uint4 z = make_uint4(0, 0, 0, 0);
      const uint4 a4 = jb + 4 <= pad ? load4(jb >> 2) : z;
      const uint4 b4 = jb + 8 <= pad ? load4((jb >> 2) + 1) : z;
      k[0] = a4.x;
      k[1] = a4.y;
      k[2] = a4.z;
      k[3] = a4.w;
      k[4] = b4.x;
      k[5] = b4.y;
      k[6] = b4.z;
      k[7] = b4.w;
      uint32_t m8 = 0u;
#pragma unroll
      for (int u = 0; u < 8; ++u) m8 |= (jb + u < j1 && (k[u] & mask) >= cut) ? 1u << u : 0u;
      const int c = __popc(m8);
      int incl = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
      }
      // bitmap word i of the 8: the bytes of lanes 4 i .. 4 i + 3
      uint32_t w = m8 << (8 * (lane & 3));
      w |= __shfl_xor_sync(0xffffffffu, w, 1);
      w |= __shfl_xor_sync(0xffffffffu, w, 2);
      st_global_if(bits + (base >> 5) + (lane >> 2), w, (lane & 3) == 0 && base + 8 * lane < j1);
      int pos = at + incl - c;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const bool sel = (m8 >> u) & 1u;
        st_global_if(sel_row + pos, static_cast<uint32_t>(jb + u), sel);
        pos += sel ? 1 : 0;
      }
      at += __shfl_sync(0xffffffffu, incl, 31);
    }
  } else {
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
      if (lane == 0) bits[base >> 5] = selm;
      gt_before += __popc(gtm);
      eq_before += __popc(eqm);
    }
  }
  __syncthreads();  // the scratch may be reused
}

// Selection pages of S = 16 / sub tokens (sub = 2 or 4): the bits of word u
// that start a cache page with at least one selected sub-page.
__device__ __forceinline__ uint32_t subpage_groups(uint32_t u, int sub) {
  return sub == 2 ? (u | (u >> 1)) & 0x55555555u
                  : (u | (u >> 1) | (u >> 2) | (u >> 3)) & 0x11111111u;
}

// The union of G heads' selection bitmaps (word(h, w)) over selection pages of
// S tokens, ascending, with a bit per head, each selection page written as its
// cache pages (S / 16 of them, fewer for the last page of a sequence of n
// tokens): out[0 .. count) = (cache page, mask); *count_out = count.  Pages of
// S = 4 or 8 tokens: each cache page holding a selected one is written once,
// its mask holding 16 / S bits per head (bit h * 16 / S + sub-page).
template <typename WordFn>
__device__ void block_union(const WordFn& word, int G, int W32, int S, int n, int2* out,
                            int* count_out, SelScratch& sc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int span = (W32 + 32 * sel_warps() - 1) / (32 * sel_warps()) * 32;  // words per warp
  const int w0 = warp * span, w1 = min(W32, w0 + span);
  const int msub = S / kPage, last = static_cast<int>(ceil_div(n, S)) - 1;
  const int sub = S < kPage ? kPage / S : 1;  // selection pages per cache page
  auto pages_of = [&](uint32_t u, int wi) {  // cache pages of word wi's selection pages
    if (sub > 1) return __popc(subpage_groups(u, sub));
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
  if (lane == 0) sc.warp_gt[warp] = static_cast<uint32_t>(cnt);
  __syncthreads();
  int before = warps_before(sc.warp_gt);
  const int total = warps_total(sc.warp_gt);
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
    if (sub > 1) {
      uint32_t gm = subpage_groups(u, sub);
      const uint32_t sub_mask = (1u << sub) - 1u;
      while (gm) {
        const int bit = __ffs(gm) - 1;  // first sub-page of a cache page
        gm &= gm - 1;
        uint32_t m = 0;
#pragma unroll
        for (int h = 0; h < 8; ++h) m |= ((hw[h] >> bit) & sub_mask) << (h * sub);
        out[pos++] = make_int2((wi * 32 + bit) / sub, static_cast<int>(m));
      }
    } else {
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
    }
    before += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (threadIdx.x == 0) *count_out = total;
  __syncthreads();
}

// ---------------------------------------------------------------- kernels
template <int D, bool F16, bool EXACT>
__global__ void __launch_bounds__(kScoreWarps * 32) score_kernel(const ScoreArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int page0 = blockIdx.x * kScorePagesPerCta + warp * 16;
  griddep_launch_dependents();
  griddep_wait();
  if (page0 >= a.P) return;
  uint32_t bq[D / 16][4];
  load_q_pm<D, EXACT>(a.q, a.q_sb, a.q_sh, b, kvh, a.G, lane, bq);
  const int64_t mbase = (static_cast<int64_t>(b) * a.Hkv + kvh) * a.P * D;
  float acc[4];
  score_tile<D, F16, EXACT>(bq, static_cast<const uint16_t*>(a.meta_max) + mbase,
                     static_cast<const uint16_t*>(a.meta_min) + mbase, page0, a.P, lane, acc);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int head = 2 * t4 + (e & 1);
    const int page = page0 + g + 8 * (e >> 1);
    if (head < a.G && page < a.P)
      a.scores[(static_cast<int64_t>(b) * a.Hq + kvh * a.G + head) * a.P + page] = acc[e];
  }
}

// Bound scores over 8-bit metadata ("TinyServe" 相关性函数实例化 with the
// outward-rounded grid of the 8-bit format): with dec(c) = lo + c * step,
//   r = sum_i q_i dec(c_i) = lo * sum_i q_i + step * (q+ . code_max + q- . code_min).
// The codes (0..255) are exact in bf16 and fp16, so both dot products run on
// tensor cores: query heads on the M side (rows 0-7), eight pages a tile on
// the N side.  Inside k-step ks, lane (g, t4) holds k positions 2 t4, 2 t4 + 1,
// 2 t4 + 8, 2 t4 + 9; they carry channels D/4 * t4 + 4 ks + 0..3, for q and
// codes alike (the order of a dot product's terms does not change it), so a
// lane reads its D/4 code bytes of a page as contiguous 16-byte vectors.
constexpr int kScore8Warps = 4;
constexpr int kScore8TilesPerWarp = 4;
constexpr int kScore8PagesPerCta = 8 * kScore8TilesPerWarp * kScore8Warps;

// Two code bytes (bytes `first`, first + 1 of w) as an exact fp16 pair: each
// byte under the high byte 0x64 of 1024 (one byte permute) is 1024 + c;
// subtracting 1024 leaves c.
__device__ __forceinline__ uint32_t codes_h2(uint32_t w, int first) {
  const uint32_t bits = __byte_perm(w, 0x64646464u, first == 0 ? 0x4140u : 0x4342u);
  const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&bits),
                            __half2half2(__ushort_as_half(0x6400)));
  return *reinterpret_cast<const uint32_t*>(&c);
}

template <bool F16>
__device__ __forceinline__ uint32_t codes_pair(uint32_t w, int first) {
  // two code bytes as exact 16-bit floats: each byte placed under the exponent
  // of 2^23 (one byte permute gives the fp32 2^23 + c), minus 2^23
  const float c0 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650u | first)) - 8388608.f;
  const float c1 = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650u | (first + 1))) - 8388608.f;
  if constexpr (F16) {
    const __half2 h = __floats2half2_rn(c0, c1);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(c0, c1);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

template <int D, bool F16>
__global__ void __launch_bounds__(kScore8Warps * 32) score8_kernel(const Score8Args a) {
  constexpr int KS = D / 16, CPL = D / 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int b = blockIdx.z, kvh = blockIdx.y;
  griddep_launch_dependents();
  griddep_wait();
  const int page0 = (blockIdx.x * kScore8Warps + warp) * kScore8TilesPerWarp * 8;
  if (page0 >= a.P) return;
  const bool head_ok = g < a.G;
  // A fragments of q+ and q- for head g, and the lane's part of sum_i q_i
  uint32_t qp[KS][2], qm[KS][2];
  float qsum = 0.f;
  {
    const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + b * a.q_sb +
                           static_cast<int64_t>(kvh * a.G + (head_ok ? g : 0)) * a.q_sh +
                           CPL * t4;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint2 w = make_uint2(0u, 0u);
      if (head_ok) {
        w.x = *reinterpret_cast<const uint32_t*>(qrow + 4 * ks);
        w.y = *reinterpret_cast<const uint32_t*>(qrow + 4 * ks + 2);
      }
      qp[ks][0] = keep_sign(w.x, false);
      qm[ks][0] = keep_sign(w.x, true);
      qp[ks][1] = keep_sign(w.y, false);
      qm[ks][1] = keep_sign(w.y, true);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t h = (((e < 2) ? w.x : w.y) >> (16 * (e & 1))) & 0xffffu;
        qsum += F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(h)))
                    : __uint_as_float(h << 16);
      }
    }
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
  }
  const int64_t pbase = (static_cast<int64_t>(b) * a.Hkv + kvh) * a.P;
#pragma unroll 1
  for (int t = 0; t < kScore8TilesPerWarp; ++t) {
    const int tile0 = page0 + 8 * t;
    if (tile0 >= a.P) break;
    const int pn = tile0 + g;  // this lane's page on the N side
    uint4 vmx[CPL / 16], vmn[CPL / 16];
#pragma unroll
    for (int v = 0; v < CPL / 16; ++v) {
      if (pn < a.P) {
        const int64_t off = (pbase + pn) * D + CPL * t4 + 16 * v;
        vmx[v] = __ldcs(reinterpret_cast<const uint4*>(a.code_max + off));
        vmn[v] = __ldcs(reinterpret_cast<const uint4*>(a.code_min + off));
      } else {
        vmx[v] = make_uint4(0u, 0u, 0u, 0u);
        vmn[v] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      // k-step ks: code bytes 4 ks .. 4 ks + 3 of the lane's run
      const uint4& X = vmx[ks / 4];
      const uint4& Y = vmn[ks / 4];
      const uint32_t wx = (ks & 3) == 0 ? X.x : (ks & 3) == 1 ? X.y : (ks & 3) == 2 ? X.z : X.w;
      const uint32_t wy = (ks & 3) == 0 ? Y.x : (ks & 3) == 1 ? Y.y : (ks & 3) == 2 ? Y.z : Y.w;
      mma16816<F16>(sc, qp[ks][0], 0u, qp[ks][1], 0u, codes_pair<F16>(wx, 0),
                    codes_pair<F16>(wx, 2));
      mma16816<F16>(sc, qm[ks][0], 0u, qm[ks][1], 0u, codes_pair<F16>(wy, 0),
                    codes_pair<F16>(wy, 2));
    }
    // head g, pages tile0 + 2 t4 + e
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int page = tile0 + 2 * t4 + e;
      if (head_ok && page < a.P) {
        const float lo = a.lo[pbase + page], st = a.step[pbase + page];
        a.scores[(static_cast<int64_t>(b) * a.Hq + kvh * a.G + g) * a.P + page] =
            __fmaf_rn(st, sc[e], lo * qsum);
      }
    }
  }
}

// One query head per kv head and 16-token pages: a unit's union is its one
// row, ascending, each page with mask 1, so the top-K kernel writes it (row
// b * Hq + h is unit b * Hkv + h) and the union kernel is not launched.  The
// row's kkb entries are read back from L2 after the barrier that ordered
// their writes; threads t, t + nt, ... of the row take them.
__device__ __forceinline__ void write_row_union(const int32_t* sel_row, int kkb, int row,
                                                const TopkArgs& a, int t, int nt) {
  int2* ul = a.union_list + static_cast<int64_t>(row) * a.union_stride;
  for (int i = t; i < kkb; i += nt) ul[i] = make_int2(__ldcg(sel_row + i), 1);
  if (t == 0) a.union_count[row] = kkb;
}

template <bool SMEM>
__global__ void __launch_bounds__(kSelMaxThreads) topk_kernel(const TopkArgs a) {
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
  // a shorter sequence: its own pages only, and possibly fewer than kk kept
  const int Pb = static_cast<int>(ceil_div(seq_len_of(a.lens, row / a.Hq, a.N), a.S));
  const int kkb = min(a.kk, Pb);
  auto key = [&](int j) {
    if constexpr (SMEM) return s_keys[j];
    return score_key(score(j));
  };
  // keys 4 q .. 4 q + 3, zero from Pb on: staged, or from the score row (one
  // 16-byte load when the row is one head's and 16-byte aligned)
  const bool vec_row = a.group == 1 && (a.P & 3) == 0;
  auto load4 = [&](int q) -> uint4 {
    if constexpr (SMEM) return *reinterpret_cast<const uint4*>(s_keys + 4 * q);
    uint4 k;
    if (vec_row && 4 * q + 3 < Pb) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(r) + q);
      k = make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
    } else {
      k.x = 4 * q < Pb ? key(4 * q) : 0u;
      k.y = 4 * q + 1 < Pb ? key(4 * q + 1) : 0u;
      k.z = 4 * q + 2 < Pb ? key(4 * q + 2) : 0u;
      k.w = 4 * q + 3 < Pb ? key(4 * q + 3) : 0u;
    }
    return k;
  };
  uint32_t prefix, mask;
  int need;
  bool found = false;
  if constexpr (SMEM) {
    // Keys 0 .. Pb - 1 to shared memory, zero from Pb up to a multiple of 4
    // (the sample bracket's vector passes).  With the sample bracket, warps 0
    // and 1 pick its splitters from the score row meanwhile.
    int r_hi = 0, r_lo = 0;
    const bool sampled = Pb >= kSampleMinP && sample_ranks(kkb, Pb, r_hi, r_lo);
    const int t0 = sampled ? 64 : 0, nt = sel_threads() - t0;
    const int tid = static_cast<int>(threadIdx.x);
    if (tid < t0) {
      sample_splitter(r, a.P, a.group, Pb, tid < 32 ? r_hi : r_lo, sc.comp + 1024 * (tid >> 5),
                      sc.hist + kSplitOffset + (tid >> 5));
    } else if (a.group == 1 && (a.P & 3) == 0) {
      // one score row: 16-byte loads, eight in flight a thread
      const float4* r4 = reinterpret_cast<const float4*>(r);
      const int n4 = a.P / 4;
#pragma unroll 8
      for (int j = tid - t0; j < n4; j += nt) {
        const float4 v = __ldcg(r4 + j);
        uint4 k = make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
        if (4 * j + 3 >= Pb) {
          k.x = 4 * j < Pb ? k.x : 0u;
          k.y = 4 * j + 1 < Pb ? k.y : 0u;
          k.z = 4 * j + 2 < Pb ? k.z : 0u;
          k.w = 0u;
        }
        *reinterpret_cast<uint4*>(s_keys + 4 * j) = k;
      }
    } else {
#pragma unroll 8
      for (int j = tid - t0; j < a.P; j += nt) s_keys[j] = j < Pb ? score_key(score(j)) : 0u;
      // past P (up to a multiple of 4): no thread stages there
      if (tid - t0 < 3 && a.P + tid - t0 < 4 * static_cast<int>(ceil_div(Pb, 4)))
        s_keys[a.P + tid - t0] = 0u;
    }
    __syncthreads();
    if (sampled) found = block_sample_select(load4, Pb, kkb, sc, prefix, mask, need);
  } else {
    // rows longer than the staging area: keys read from the score row (in L2
    // after the score kernel) in every pass, with the same sample bracket
    int r_hi = 0, r_lo = 0;
    if (Pb >= kSampleMinP && sample_ranks(kkb, Pb, r_hi, r_lo)) {
      const int tid = static_cast<int>(threadIdx.x);
      if (tid < 64)
        sample_splitter(r, a.P, a.group, Pb, tid < 32 ? r_hi : r_lo, sc.comp + 1024 * (tid >> 5),
                        sc.hist + kSplitOffset + (tid >> 5));
      __syncthreads();
      found = block_sample_select(load4, Pb, kkb, sc, prefix, mask, need);
    }
  }
  uint32_t* bits = a.bitmaps + static_cast<int64_t>(row) * a.W32;
  if (!found) block_radix_select(key, Pb, kkb, sc, prefix, mask, need);
  int32_t* sel_row = a.selected + static_cast<int64_t>(row) * a.kk;
  if (!found) block_emit_counts(key, Pb, prefix, mask, sc);
  block_emit(key, load4, Pb, prefix, mask, need, sel_row, bits, sc);  // ends in a block barrier
  for (int w = static_cast<int>(ceil_div(Pb, 32)) + threadIdx.x; w < a.W32; w += sel_threads())
    bits[w] = 0u;
  for (int i = kkb + threadIdx.x; i < a.kk; i += sel_threads()) sel_row[i] = -1;
  if (a.union_list != nullptr)
    write_row_union(sel_row, kkb, row, a, static_cast<int>(threadIdx.x), sel_threads());
}

// One warp per (b, h) row of at most kUnitMaxP keys: the row's scores (summed
// over the group's rows, head by head in order, as topk_kernel) become keys in
// the warp's shared-memory slot, the warp top-K of the per-unit kernel selects
// (keys in registers), and the warp writes the ascending row and the bitmap.
constexpr int kTopkWarpRows = 8;
__global__ void __launch_bounds__(kTopkWarpRows * 32) topk_warp_kernel(const TopkArgs a) {
  extern __shared__ uint32_t s_slots[];
  griddep_launch_dependents();
  griddep_wait();  // the scores come from the previous kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kTopkWarpRows + warp;
  if (row >= a.rows) return;
  const int Pr = static_cast<int>(ceil_div(a.P, 32)) * 32;
  uint32_t* keys = s_slots + warp * (Pr + kSelBitmapWords);
  uint32_t* bm = keys + Pr;
  const int r0 = row - (row % a.Hq) % a.group;
  const float* r = a.scores + static_cast<int64_t>(r0) * a.P;
  const int Pb = static_cast<int>(ceil_div(seq_len_of(a.lens, row / a.Hq, a.N), a.S));
  const int kkb = min(a.kk, Pb);
  uint32_t mx = 0u, mn = ~0u;
#pragma unroll 8
  for (int j = lane; j < Pb; j += 32) {
    float x = __ldcg(r + j);
    for (int h = 1; h < a.group; ++h) x = __fadd_rn(x, __ldcg(r + static_cast<int64_t>(h) * a.P + j));
    const uint32_t k = score_key(x);
    keys[j] = k;
    mx = max(mx, k);
    mn = min(mn, k);
  }
  mx = __reduce_max_sync(0xffffffffu, mx);
  mn = __reduce_min_sync(0xffffffffu, mn);
  __syncwarp();
  warp_topk_head([keys](int j) { return keys[j]; }, Pb, kkb, bm, mx, mn);
  __syncwarp();
  const int W = static_cast<int>(ceil_div(Pb, 32));
  uint32_t* bits = a.bitmaps + static_cast<int64_t>(row) * a.W32;
  int32_t* sel_row = a.selected + static_cast<int64_t>(row) * a.kk;
  warp_emit_row(bm, W, sel_row, bits);
  for (int w = W + lane; w < a.W32; w += 32) bits[w] = 0u;
  for (int i = kkb + lane; i < a.kk; i += 32) sel_row[i] = -1;
  if (a.union_list != nullptr) {
    __syncwarp();  // the row's entries, written by the warp's lanes
    write_row_union(sel_row, kkb, row, a, lane, 32);
  }
}

__global__ void __launch_bounds__(kSelMaxThreads) union_kernel(const UnionArgs a) {
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

// ------------------------------------------------------- units of a CTA
// unit_select_kernel: the bound scores, per-head top-K and union of each
// (batch, kv head) unit, one unit at a time per CTA of a persistent grid.  Warp 8 streams the unit's metadata with TMA
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

// TWO: two CTAs a streaming multiprocessor (for more units than SMs), each with
// half the ring, so the SM keeps the same bytes in flight.
template <int D, bool M8 = false, bool TWO = false>
struct UnitCfg {
  // one of [M] / [m] (16-bit), or of the code bytes [cM] / [cm] (8-bit)
  static constexpr int kBoxBytes = kUnitBoxPages * D * (M8 ? 1 : 2);
  static constexpr int kStageBytes = 2 * kBoxBytes;
  static constexpr int kStages = ((TWO ? 64 : 128) * 1024) / kStageBytes;  // bytes in flight
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

// Shared address of the 16 code bytes (channels) [16 c, 16 c + 16) of page row
// t of an 8-bit box {D bytes, 64 pages} written with D-byte swizzle (D = 128:
// 128-byte swizzle, the chunk XORed with t % 8; D = 64: 64-byte swizzle, the
// chunk XORed with (t / 2) % 4).
template <int D>
__device__ __forceinline__ uint32_t box8_addr(uint32_t base, int t, int c) {
  const int chunk = D == 128 ? (c ^ (t & 7)) : (c ^ ((t >> 1) & 3));
  return base + static_cast<uint32_t>(t * D + chunk * 16);
}

__device__ __forceinline__ void unit_consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kUnitConsumers * 32) : "memory");
}

// The union is built by warps 0-3 (warps 4-7 write the per-head rows meanwhile).
constexpr int kUnionWarps = 4;
__device__ __forceinline__ void union_sync() {
  asm volatile("bar.sync 2, %0;" ::"r"(kUnionWarps * 32) : "memory");
}

// M8: the scores come from 8-bit metadata (codes in the boxes, lo / step per
// page from global memory).
template <int D, bool F16, bool M8, bool TWO = false>
__global__ void __launch_bounds__(kUnitThreads, TWO ? 2 : 1)
    unit_select_kernel(const UnitSelectArgs a, const __grid_constant__ CUtensorMap mmx,
                       const __grid_constant__ CUtensorMap mmn) {
  using C = UnitCfg<D, M8, TWO>;
  extern __shared__ uint8_t usm_raw[];
  uint8_t* usm = usm_raw + ((1024u - (smem_u32(usm_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(usm);
  const uint32_t full0 = sbase + C::kBarOffset, empty0 = full0 + 8 * C::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(usm + C::kBarOffset + 16 * C::kStages);
  uint32_t* s_keys = reinterpret_cast<uint32_t*>(usm + C::kKeysOffset);      // [G][P]
  uint32_t* s_bm = s_keys + static_cast<size_t>(a.G) * a.P;                  // [G][kSelBitmapWords]
  // [0..7] / [8..15]: each head's largest / smallest key; [16] / [17]: the
  // group score's (one selection per group)
  uint32_t* s_kext = s_bm + static_cast<size_t>(a.G) * kSelBitmapWords;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = a.B * a.Hkv;
  // This CTA's units: blockIdx.x, blockIdx.x + gridDim.x, ...  The producer
  // warp streams their metadata back to back (box gi of the CTA, counted over
  // all its units, goes to stage gi % kStages), so the next unit's boxes are
  // in flight while the consumers select and build the current one's union.
  auto unit_pages = [&](int u) {  // selection pages of unit u's sequence
    return static_cast<int>(ceil_div(seq_len_of(a.lens, u / a.Hkv, a.N), a.S));
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 4);  // the four warps that score the stage
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kUnitConsumers && lane == 0) {
    prefetch_tensormap(&mmx);
    prefetch_tensormap(&mmn);
  }
  griddep_wait();
  // The attention grid may start as soon as every CTA here has passed this
  // point, and then reads the units' ready flags: clear this CTA's first (the
  // previous call's attention has finished with them once the wait returns).
  if (threadIdx.x == 0 && a.unit_ready != nullptr) {
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) a.unit_ready[u] = 0u;
    __threadfence();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kUnitConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int gi = 0;  // boxes issued by this CTA
      bool failed = false;
      for (int u = blockIdx.x; u < n_units && !failed; u += gridDim.x) {
        const int ub = u / a.Hkv, ukvh = u % a.Hkv;
        const int nb = static_cast<int>(ceil_div(unit_pages(u), kUnitBoxPages));
        for (int i = 0; i < nb; ++i, ++gi) {
          const int s = gi % C::kStages;
          if (gi >= C::kStages &&
              !mbar_wait_bounded(empty0 + 8 * s, ((gi / C::kStages) - 1) & 1, a.wait_limit_ns,
                                 abort_flag)) {
            if (*abort_flag == 0) {
              set_status(a.status, kStatusTimeout);
              *abort_flag = 1;
            }
            failed = true;
            break;
          }
          const uint32_t dst = sbase + s * C::kStageBytes;
          mbar_arrive_expect_tx(full0 + 8 * s, C::kStageBytes);
          tma_load_5d_hint(dst, &mmx, full0 + 8 * s, 0, i * kUnitBoxPages, 0, ukvh, ub, pol);
          tma_load_5d_hint(dst + C::kBoxBytes, &mmn, full0 + 8 * s, 0, i * kUnitBoxPages, 0,
                           ukvh, ub, pol);
        }
      }
      // The last copies issued have landed before this warp leaves (so no copy
      // is still writing when the consumers stop early); each wait is bounded.
      const uint64_t deadline = globaltimer_ns() + 200000000ull;
      for (int j = max(0, gi - C::kStages); j < gi; ++j) {
        const uint64_t now = globaltimer_ns();
        if (now >= deadline) break;
        mbar_wait_bounded(full0 + 8 * (j % C::kStages), (j / C::kStages) & 1, deadline - now,
                          nullptr);
      }
    }
    return;
  }

  const int g = lane >> 2, t4 = lane & 3;
  const bool head_ok = g < a.G;
  const int mtx = lane >> 3, mrow = lane & 7;
  const int half = warp >> 2, tile = warp & 3;  // boxes of parity `half`, tile `tile` of each
  int gbase = 0;  // boxes of this CTA's earlier units
  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
  const int b = unit / a.Hkv, kvh = unit % a.Hkv;
  const int Nb = seq_len_of(a.lens, b, a.N);
  const int Pb = unit_pages(unit);
  const int n_boxes = static_cast<int>(ceil_div(Pb, kUnitBoxPages));
  if (threadIdx.x < 18) s_kext[threadIdx.x] = (threadIdx.x < 8 || threadIdx.x == 16) ? 0u : ~0u;
  unit_consumers_sync();

  // -------------------------------------------------------------- scoring
  // 8-bit metadata: lo and step of the lane's four pages of a box, loaded one
  // of this warp's boxes ahead (box i + 2), so their latency hides behind the
  // box wait instead of following each tile's MMAs.
  float lo_n[4] = {0.f, 0.f, 0.f, 0.f}, st_n[4] = {0.f, 0.f, 0.f, 0.f};
  auto load_lo_step = [&](int box) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int p = box * kUnitBoxPages + 16 * tile + 8 * (e >> 1) + 2 * t4 + (e & 1);
      const int64_t pi = static_cast<int64_t>(unit) * a.P + p;
      lo_n[e] = (head_ok && p < Pb) ? __ldg(a.lo + pi) : 0.f;
      st_n[e] = (head_ok && p < Pb) ? __ldg(a.step + pi) : 0.f;
    }
  };
  if constexpr (M8) {
    if (half < n_boxes) load_lo_step(half);  // (its latency overlaps the query loads)
  }
  uint32_t qp[D / 16][2], qm[D / 16][2];  // A fragments of q+ and q- (rows = heads)
  float qsum = 0.f;  // 8-bit metadata: sum_i q_i of head g
  float qscale = 1.f;  // 8-bit metadata: the scores' factor 2^k (q was scaled by 2^-k)
  if constexpr (M8) {
    // 8-bit metadata: fp16 MMAs.  The codes widen to fp16 exactly (1024 + c,
    // minus 1024); q is scaled by 2^-k per head, k such that its largest
    // component lands in [2^14, 2^15), which fp16 holds exactly for every
    // bf16 component within 2^31 of that largest one (the rest, below 2^-17
    // after scaling, round to the fp16 grid of 2^-24).  Channels of k-step
    // ks: 16 ks + 4 t4 + 0..3, the bytes an ldmatrix row fragment of the code
    // box gives the lane.
    const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + b * a.q_sb +
                           static_cast<int64_t>(kvh * a.G + (head_ok ? g : 0)) * a.q_sh;
    float qmax = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint2 w = head_ok ? *reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * t4)
                              : make_uint2(0u, 0u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t h = (((e < 2) ? w.x : w.y) >> (16 * (e & 1))) & 0xffffu;
        const float x = F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(h)))
                            : __uint_as_float(h << 16);
        qsum += x;
        qmax = fmaxf(qmax, fabsf(x));
      }
    }
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
    qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
    qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
    const int k = (F16 || qmax == 0.f) ? 0 : ((__float_as_int(qmax) >> 23) & 0xff) - 127 - 14;
    const float down = __int_as_float((127 - k) << 23);  // 2^-k
    qscale = __int_as_float((127 + k) << 23);            // 2^k
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint2 w = head_ok ? *reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * t4)
                              : make_uint2(0u, 0u);
      uint32_t h2[2];
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const uint32_t ww = v ? w.y : w.x;
        if constexpr (F16) {
          h2[v] = ww;
        } else {
          const __half2 hh = __floats2half2_rn(__uint_as_float(ww << 16) * down,
                                               __uint_as_float(ww & 0xffff0000u) * down);
          h2[v] = *reinterpret_cast<const uint32_t*>(&hh);
        }
      }
      qp[ks][0] = keep_sign(h2[0], false);
      qm[ks][0] = keep_sign(h2[0], true);
      qp[ks][1] = keep_sign(h2[1], false);
      qm[ks][1] = keep_sign(h2[1], true);
    }
  } else {
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
  bool ok = true;
  uint32_t kmx = 0u, kmn = ~0u;  // extremes of head g's keys this lane wrote
  for (int i = half; i < n_boxes; i += 2) {
    float lo_c[4], st_c[4];
    if constexpr (M8) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        lo_c[e] = lo_n[e];
        st_c[e] = st_n[e];
      }
      if (i + 2 < n_boxes) load_lo_step(i + 2);
    }
    const int gi = gbase + i;
    const int s = gi % C::kStages;
    ok = mbar_wait_bounded(full0 + 8 * s, (gi / C::kStages) & 1, a.wait_limit_ns, abort_flag);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    const uint32_t mb = sbase + s * C::kStageBytes, nb = mb + C::kBoxBytes;
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if constexpr (M8) {
      // Matrices of one ldmatrix.x4: pages 16 tile + 0..7 / + 8..15 (n tiles
      // 0 / 1) of code chunks ks and ks + 1; lane (g, t4) gets the four code
      // bytes 4 t4 .. 4 t4 + 3 of its page g of each.
      const int row = 16 * tile + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < D / 16; ks += 2) {
        uint32_t x0, x1, x2, x3, y0, y1, y2, y3;
        ldsm_x4(box8_addr<D>(mb, row, ks + (lane >> 4)), x0, x1, x2, x3);
        ldsm_x4(box8_addr<D>(nb, row, ks + (lane >> 4)), y0, y1, y2, y3);
        mma16816<true>(sc[0], qp[ks][0], 0u, qp[ks][1], 0u, codes_h2(x0, 0), codes_h2(x0, 2));
        mma16816<true>(sc[1], qp[ks][0], 0u, qp[ks][1], 0u, codes_h2(x1, 0), codes_h2(x1, 2));
        mma16816<true>(sc[0], qm[ks][0], 0u, qm[ks][1], 0u, codes_h2(y0, 0), codes_h2(y0, 2));
        mma16816<true>(sc[1], qm[ks][0], 0u, qm[ks][1], 0u, codes_h2(y1, 0), codes_h2(y1, 2));
        mma16816<true>(sc[0], qp[ks + 1][0], 0u, qp[ks + 1][1], 0u, codes_h2(x2, 0),
                       codes_h2(x2, 2));
        mma16816<true>(sc[1], qp[ks + 1][0], 0u, qp[ks + 1][1], 0u, codes_h2(x3, 0),
                       codes_h2(x3, 2));
        mma16816<true>(sc[0], qm[ks + 1][0], 0u, qm[ks + 1][1], 0u, codes_h2(y2, 0),
                       codes_h2(y2, 2));
        mma16816<true>(sc[1], qm[ks + 1][0], 0u, qm[ks + 1][1], 0u, codes_h2(y3, 0),
                       codes_h2(y3, 2));
      }
    } else {
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
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    if (head_ok) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int p = i * kUnitBoxPages + 16 * tile + 8 * (e >> 1) + 2 * t4 + (e & 1);
        if (p < Pb) {
          float sv = sc[e >> 1][e & 1];
          if constexpr (M8) sv = __fmaf_rn(st_c[e], sv * qscale, lo_c[e] * qsum);
          const uint32_t key = score_key(sv);
          s_keys[g * a.P + p] = key;
          kmx = max(kmx, key);
          kmn = min(kmn, key);
        }
      }
    }
  }
  gbase += n_boxes;
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
    if (threadIdx.x == 0) {
      // gather nothing for this unit or this CTA's later ones
      for (int u = unit; u < n_units; u += gridDim.x) {
        a.union_count[u] = 0;
        if (a.unit_ready != nullptr) {
          __threadfence();
          st_release_gpu(a.unit_ready + u, 1u);
        }
      }
    }
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
    // (the short-head copies only where d = 64 contexts run short)
    warp_topk_head<D == 64>([keys](int j) { return keys[j]; }, Pb, kkb, bm,
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
  } else {
  // Union of the heads' bitmaps, ascending, with a bit per head: warp w ORs
  // words w * wpw .. (one per lane), the per-warp counts place them.  Each
  // selection page becomes its S / 16 cache pages (fewer for the sequence's
  // last).
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
    if (a.unit_ready != nullptr) {
      // publish the unit: every writer's list entries, then the count, then
      // the flag the attention kernel waits on
      __threadfence();
      union_sync();
      if (threadIdx.x == 0) {
        a.union_count[unit] = count;
        __threadfence();
        st_release_gpu(a.unit_ready + unit, 1u);
      }
    } else if (threadIdx.x == 0) {
      a.union_count[unit] = count;
    }
  }
  unit_consumers_sync();  // keys, bitmaps and extremes are free for the next unit
  }
}

}  // namespace

cudaError_t launch_score(int d, bool f16, const ScoreArgs& a, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>(ceil_div(a.P, kScorePagesPerCta)), a.Hkv, a.B);
  dim3 block(kScoreWarps * 32);
  if (a.exact) {
    if (d == 128)
      return f16 ? launch_pdl(score_kernel<128, true, true>, grid, block, 0, s, a)
                 : launch_pdl(score_kernel<128, false, true>, grid, block, 0, s, a);
    return f16 ? launch_pdl(score_kernel<64, true, true>, grid, block, 0, s, a)
               : launch_pdl(score_kernel<64, false, true>, grid, block, 0, s, a);
  }
  if (d == 128) {
    return f16 ? launch_pdl(score_kernel<128, true, false>, grid, block, 0, s, a)
               : launch_pdl(score_kernel<128, false, false>, grid, block, 0, s, a);
  }
  return f16 ? launch_pdl(score_kernel<64, true, false>, grid, block, 0, s, a)
             : launch_pdl(score_kernel<64, false, false>, grid, block, 0, s, a);
}

cudaError_t launch_score8(int d, bool f16, const Score8Args& a, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(ceil_div(a.P, kScore8PagesPerCta)), a.Hkv, a.B);
  const dim3 block(kScore8Warps * 32);
  if (d == 128)
    return f16 ? launch_pdl(score8_kernel<128, true>, grid, block, 0, s, a)
               : launch_pdl(score8_kernel<128, false>, grid, block, 0, s, a);
  return f16 ? launch_pdl(score8_kernel<64, true>, grid, block, 0, s, a)
             : launch_pdl(score8_kernel<64, false>, grid, block, 0, s, a);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
  if (a.P <= kUnitMaxP) {  // a warp a row, keys in registers
    const size_t smem = sizeof(uint32_t) * kTopkWarpRows *
                        (static_cast<size_t>(ceil_div(a.P, 32)) * 32 + kSelBitmapWords);
    cudaError_t e = cudaFuncSetAttribute(topk_warp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_warp_kernel, dim3(static_cast<unsigned>(ceil_div(a.rows, kTopkWarpRows))),
                      dim3(kTopkWarpRows * 32), smem, s, a);
  }
  const size_t key_bytes = 16 * static_cast<size_t>(ceil_div(a.P, 4));  // zero-padded to 4
  if (key_bytes <= kTopkSmemKeyBytes) {
    cudaError_t e = cudaFuncSetAttribute(topk_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kTopkSmemKeyBytes));
    if (e != cudaSuccess) return e;
    // rows long enough for the sample bracket get 1024 threads; shorter rows
    // 256 (their passes are short, and fewer warps meet at each barrier)
    const int threads = a.P >= kSampleMinP ? kSelMaxThreads : 256;
    return launch_pdl(topk_kernel<true>, dim3(a.rows), dim3(threads), key_bytes, s, a);
  }
  return launch_pdl(topk_kernel<false>, dim3(a.rows), dim3(kSelMaxThreads), 0, s, a);
}

namespace {
template <int D, bool M8, bool TWO>
size_t unit_smem_t(int G, int P) {
  return 1024 + UnitCfg<D, M8, TWO>::kKeysOffset + static_cast<size_t>(G) * P * 4 +
         static_cast<size_t>(G) * kSelBitmapWords * 4 + 32 * 4;
}
// Shared memory a CTA may take when two share a multiprocessor.
constexpr size_t kUnitTwoSmemLimit = 112 * 1024;

template <int D, bool F16, bool M8, bool TWO>
cudaError_t launch_unit_t(const UnitSelectArgs& a, const CUtensorMap& mmx, const CUtensorMap& mmn,
                          int grid, cudaStream_t s) {
  const size_t smem = unit_smem_t<D, M8, TWO>(a.G, a.P);
  auto kern = unit_select_kernel<D, F16, M8, TWO>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kUnitThreads), smem, s, a, mmx, mmn);
}
}  // namespace

size_t unit_select_smem(int d, bool m8, int G, int P) {
  return d == 128 ? (m8 ? unit_smem_t<128, true, false>(G, P) : unit_smem_t<128, false, false>(G, P))
                  : (m8 ? unit_smem_t<64, true, false>(G, P) : unit_smem_t<64, false, false>(G, P));
}

cudaError_t launch_unit_select(int d, bool f16, bool m8, const UnitSelectArgs& a,
                               const CUtensorMap& mmx, const CUtensorMap& mmn, cudaStream_t s) {
  // One CTA per SM at most (a CTA takes most of an SM's shared memory), each
  // taking units blockIdx.x, + gridDim.x, ...: with fewer CTAs the metadata
  // scan streams from too few SMs (measured: 64, 80, 96, 112 CTAs for 128
  // units were slower than 128).  With more units than SMs at d = 64, two
  // CTAs of half the ring share each SM, so every unit starts at once.
  const int units = a.B * a.Hkv;
  if (d == 64 && units > a.num_sms &&
      (m8 ? unit_smem_t<64, true, true>(a.G, a.P) : unit_smem_t<64, false, true>(a.G, a.P)) <=
          kUnitTwoSmemLimit) {
    const int grid = units < 2 * a.num_sms ? units : 2 * a.num_sms;
    return m8 ? (f16 ? launch_unit_t<64, true, true, true>(a, mmx, mmn, grid, s)
                     : launch_unit_t<64, false, true, true>(a, mmx, mmn, grid, s))
              : (f16 ? launch_unit_t<64, true, false, true>(a, mmx, mmn, grid, s)
                     : launch_unit_t<64, false, false, true>(a, mmx, mmn, grid, s));
  }
  const int grid = units < a.num_sms ? units : a.num_sms;
  if (d == 128)
    return m8 ? (f16 ? launch_unit_t<128, true, true, false>(a, mmx, mmn, grid, s)
                     : launch_unit_t<128, false, true, false>(a, mmx, mmn, grid, s))
              : (f16 ? launch_unit_t<128, true, false, false>(a, mmx, mmn, grid, s)
                     : launch_unit_t<128, false, false, false>(a, mmx, mmn, grid, s));
  return m8 ? (f16 ? launch_unit_t<64, true, true, false>(a, mmx, mmn, grid, s)
                   : launch_unit_t<64, false, true, false>(a, mmx, mmn, grid, s))
            : (f16 ? launch_unit_t<64, true, false, false>(a, mmx, mmn, grid, s)
                   : launch_unit_t<64, false, false, false>(a, mmx, mmn, grid, s));
}

cudaError_t launch_union(const UnionArgs& a, int units, cudaStream_t s) {
  return launch_pdl(union_kernel, dim3(units), dim3(256), 0, s, a);
}

}  // namespace dkv

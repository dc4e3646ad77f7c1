// attn.cu -- decode attention over pages of a KV cache (exact and page-sparse)
// and the merge of its split-K partials.
//
// What it computes (per query head h of batch b, kv head h / G):
//   out = sum_t softmax_t(scale * q . k_t) v_t
// over all N tokens ("论文阅读：HeadInfer", 核心 idea; "TinyServe: Query-Aware
// Cache Selection for Efficient LLM Serving", 标准Transformer解码层的注意力计算)
// or over the tokens of the pages selected for h (TinyServe, 问题公式化定义,
// Algorithm 1 steps 3-4: gather the selected pages, then softmax-weighted sum).
//
// attn_kernel is persistent: kAttnCtasPerSm CTAs per SM pull work items --
// (batch, kv head, chunk of pages) -- from an atomic counter until none are
// left.  Inside a CTA:
//   * warp 4 (producer) takes the next item, turns it into a page list (in the
//     sparse path: its slice of the group's union of selected pages, each with
//     a bit per query head that chose it; slices past the union are skipped
//     unpublished), publishes it
//     through a two-slot descriptor ring and streams the pages' K and V into
//     shared-memory stages with TMA tensor copies (cp.async.bulk.tensor, 128B
//     swizzle), one full / empty mbarrier pair per stage.  It runs ahead
//     across item boundaries, so the copy engine never drains between items.
//   * warps 0-3 (consumers): page j of an item goes to warp j % 4, through that
//     warp's own sub-ring of stages.  Each stage is therefore filled and drained
//     by one fixed pair (producer, warp) in strict order, so no waiter is ever
//     more than one phase behind a barrier (parity waits cannot alias).  A warp
//     computes a 16-token page for all G <= 8 query heads at once on tensor
//     cores: S[8 heads x 16 tokens] = Q K^T with mma.sync m16n8k16 (heads on the
//     M side), an online softmax in fp32 (log2 domain), then O += P V with P
//     split into a high and a low 16-bit half (A rows 0-7 / 8-15) so the
//     weights keep ~16 significant bits.  At the end of an item warps 1-3 hand
//     their (max, sum, o) to warp 0 through shared memory, which merges them
//     with its own and writes the item's partial.
// merge_small_kernel (units of up to 32 chunks) or merge_kernel then combines
// the chunks of every (b, h) in a fixed order and writes out.  Its structure,
// like the chunking, depends only on (P, d), and partials do not depend on
// which CTA computed them, so results are deterministic and one kv head at a
// time gives bitwise the all-heads result.  The sparse 4-bit path with one
// chunk per unit (unions of up to 32 pages at d = 128, 64 at d = 64) skips
// the merge: warp 0 writes O / L itself, the value the merge would write
// (its weight is 2^0 = 1).  The other instantiations keep the partials only:
// the extra epilogue costs them more in registers and code than the merge's
// round trip (4% on the 4-bit exact kernel, 3% on the dense sparse one).
// The last CTA to stop fetching work resets the work counter.
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the status word, stops issuing, drains the copies it issued and exits.

#include <math.h>
#include <string.h>

#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {
namespace {

constexpr uint64_t kDrainLimitNs = 200000000ull;  // 200 ms for the whole drain

struct ItemDesc {
  int item;     // work item, -1: no more work
  int n_pages;  // pages in the item (0 for an empty sparse chunk)
  int seq0;     // producer sequence number of the item's first page
  int pad;
};

// QUAD: four pages a stage (the dense 4-bit path, whose pages are consecutive).
// MHA: the 4-bit single-head layout, three CTAs per SM (fewer stages each --
// two consecutive pages a stage in the dense path -- and a merge area of
// one row).
template <int D, bool Q4, bool QUAD, bool MHA = false>
struct AttnCfg {
  static constexpr int kCtasPerSm = MHA ? 3 : kAttnCtasPerSm;
  static constexpr int kPageBytes = kPage * D * 2;          // one 16-bit page tile
  static constexpr int kCodeBytes = kPage * D / 2;          // 4-bit: one tensor's page of codes
  static constexpr int kGroupBytes = kPage * (D / 64) * 2;  // 4-bit: one page of gmin (or gmax)
  // A 4-bit stage holds one page, or four pages of one consumer warp in the
  // dense path (consecutive pages of the cache move with one copy per part):
  //   K codes [q][page] | V codes [q][page] | K min | K max | V min | V max,
  // each bound array [q][page], q = kPagesPerStage.
  static constexpr int kPagesPerStage = QUAD ? (MHA ? 2 : 4) : 1;
  static constexpr int kQ4PageBytes = 2 * kCodeBytes + 4 * kGroupBytes;
  static constexpr int kQ4VCodeOffset = kPagesPerStage * kCodeBytes;
  static constexpr int kQ4BoundsOffset = 2 * kPagesPerStage * kCodeBytes;
  static constexpr int kStageBytes =
      Q4 ? (kPagesPerStage * kQ4PageBytes + 127) / 128 * 128 : 2 * kPageBytes;
  // 4-bit pages are a quarter the size: more of them in flight.
  static constexpr int kStages =
      Q4 ? (MHA ? (D == 128 ? 24 : 48) : (D == 128 ? 32 : 48)) / kPagesPerStage : attn_stages(D);
  static constexpr int kSub = kStages / kConsumerWarps;             // stages per consumer warp
  static constexpr int kBarOffset = (kStages * kStageBytes + 15) / 16 * 16;
  static constexpr int kStageMetaOffset = kBarOffset + (2 * kStages + 4) * 8;
  static constexpr int kDescOffset = kStageMetaOffset + kStages * kPagesPerStage * 8;
  static constexpr int kMergeOffset = kDescOffset + 2 * 16;
  static constexpr int kMergeRow = D + 2;                           // o[D], max, sum
  static constexpr int kMergeBytes = (kConsumerWarps - 1) * (MHA ? 1 : 8) * kMergeRow * 4;
  static constexpr int kListOffset = kMergeOffset + kMergeBytes;
  static constexpr int kBlockOffset = kListOffset + 8 * kMaxSelectList;  // paged: pool blocks
  static constexpr int kMiscOffset = kBlockOffset + 4 * kMaxSelectList;
  static constexpr int kSmemBytes = 1024 + kMiscOffset + 16;
  static_assert(Q4 || kPageBytes % 1024 == 0, "TMA stages must stay 1024-byte aligned");
  static_assert(kStages % kConsumerWarps == 0, "one sub-ring per consumer warp");
  static_assert((kSmemBytes + 1024) * kCtasPerSm <= 228 * 1024, "the CTAs fit an SM");
};

// Shared address of channels [c, c+8) of token t in a page tile written by the
// TMA box {64 channels, 16 tokens, d/64 halves} with 128-byte swizzle: row
// (half * 16 + t) holds 64 channels in 128 bytes, and the 16-byte chunk index
// is XORed with row % 8.
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int t, int c) {
  const int row = (c >> 6) * 16 + t;
  const int chunk = ((c & 63) >> 3) ^ (row & 7);
  return base + static_cast<uint32_t>(row * 128 + chunk * 16);
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
}

// Barrier over the consumer warps that also ORs `flag` across them, so every
// consumer takes the same branch afterwards.
__device__ __forceinline__ bool consumers_any(bool flag) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(res)
      : "r"(static_cast<uint32_t>(flag)), "r"(kConsumerWarps * 32)
      : "memory");
  return res != 0;
}

// 4-bit path, producer.  A run of r consecutive whole pages of the cache,
// going to stage slots slot0 .. slot0 + r - 1, moves by six 1-D bulk copies,
// one per issuing lane: part 0 K codes, 1 V codes, 2-5 K min, K max, V min,
// V max.
template <typename C, int D>
__device__ __forceinline__ void q4_copy_run(const AttnArgs& a, int b, int kvh, int page0, int r,
                                            int slot0, int part, uint32_t dst, uint32_t bar) {
  constexpr int ng = D / 64;
  const int64_t t0 = static_cast<int64_t>(page0) * kPage;
  if (part < 2) {
    const Q4View& v = part == 0 ? a.k4 : a.v4;
    bulk_load(dst + part * C::kQ4VCodeOffset + slot0 * C::kCodeBytes,
              v.codes + b * v.sb + kvh * v.sh + t0 * (D / 2), r * C::kCodeBytes, bar);
  } else {
    const int i = part - 2;
    const Q4View& v = i < 2 ? a.k4 : a.v4;
    const __half* src = ((i & 1) ? v.gmax : v.gmin) + b * v.gsb + kvh * v.gsh + t0 * ng;
    bulk_load(dst + C::kQ4BoundsOffset + (i * C::kPagesPerStage + slot0) * C::kGroupBytes, src,
              r * C::kGroupBytes, bar);
  }
}

// 4-bit path, producer: the ragged last page (nt < 16 tokens), by one lane,
// into stage slot `slot`.  The valid tokens' group bounds are loaded with plain
// loads (released by the caller's barrier arrival, which counts the codes'
// 2 * nt * d/2 bytes) and the missing tokens' bounds zeroed, so whatever codes
// their rows hold dequantise to 0 (a zero-width group: step 0; the page takes
// the consumers' tiny-group path); then only the valid tokens' codes are
// copied, so nothing is read past the cache.
template <typename C, int D>
__device__ __forceinline__ void q4_ragged_bounds(const AttnArgs& a, int b, int kvh, int page,
                                                 int nt, int slot, uint8_t* stage) {
  constexpr int ng = D / 64;
  const int64_t t0 = static_cast<int64_t>(page) * kPage;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const Q4View& v = i < 2 ? a.k4 : a.v4;
    const __half* src = ((i & 1) ? v.gmax : v.gmin) + b * v.gsb + kvh * v.gsh + t0 * ng;
    __half* gb = reinterpret_cast<__half*>(stage + C::kQ4BoundsOffset +
                                           (i * C::kPagesPerStage + slot) * C::kGroupBytes);
    for (int e = 0; e < kPage * ng; ++e) gb[e] = e < nt * ng ? src[e] : __ushort_as_half(0);
  }
}
template <typename C, int D>
__device__ __forceinline__ void q4_ragged_codes(const AttnArgs& a, int b, int kvh, int page,
                                                int nt, int slot, uint32_t dst, uint32_t bar) {
  const int64_t t0 = static_cast<int64_t>(page) * kPage;
  const uint32_t cb = static_cast<uint32_t>(nt * (D / 2));
  bulk_load(dst + slot * C::kCodeBytes, a.k4.codes + b * a.k4.sb + kvh * a.k4.sh + t0 * (D / 2),
            cb, bar);
  bulk_load(dst + C::kQ4VCodeOffset + slot * C::kCodeBytes,
            a.v4.codes + b * a.v4.sb + kvh * a.v4.sh + t0 * (D / 2), cb, bar);
}

// 4-bit path, consumer warp.  The codes go straight from the stage into MMA
// fragments in registers; no dequantised tile is written.  Channel orders are
// chosen so that every lane's codes are contiguous:
//   * S = Q K^T: lane (g, t4) holds tokens g and g + 8 of channels
//     [D/4 t4, D/4 (t4 + 1)).  Code word j of that block (channels
//     D/4 t4 + 8 j + n, nibble n) feeds k-steps 2 j (nibble pairs (0, 4) and
//     (1, 5)) and 2 j + 1 ((2, 6) and (3, 7)); the query's A fragments take the
//     same channel order.
//   * O += P V: lane (g, t4) holds tokens 2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9 of
//     channels [D/8 g, D/8 (g + 1)); output tile cn, column n is channel
//     D/8 n + cn.
// A nibble masked into the mantissa of 1024 (bits 0-3) or 64 (bits 4-7) gives
// bias + code exactly; subtracting the bias leaves the code, then
// x = fp16(code * step + mn) by one fp16 FMA -- the dequantisation of the
// 4-bit format, bit for bit.  The steps come from the stage, where the owning
// warp computed each group's once (q4_stage_steps).  A stage with a tiny group
// (range below 451 * 2^-24: its step is an fp32 value) keeps its maxes and
// takes a slower path that dequantises every pair from its group's min and
// max.
template <int D>
struct Q4Page {
  uint32_t kc[2][D / 32];  // K codes, tokens g and g + 8
  uint32_t vc[4][D / 64];  // V codes, tokens 2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9
  __half kmn[2], kx[2];    // K group min and step (group max on a tiny stage), tokens g, g + 8
  uint32_t vmn[2], vx[2];  // V: the same as half pairs, tokens (2 t4, 2 t4 + 1) and + 8
  bool tiny;               // warp-uniform: the page's stage has a tiny group
};

template <typename C, int D>
__device__ __forceinline__ void q4_load(const uint8_t* st, int slot, int g, int t4, bool tiny,
                                        Q4Page<D>& r) {
  r.tiny = tiny;
  constexpr int ng = D / 64;
  constexpr int kBound = C::kPagesPerStage * kPage * ng;  // halves from one bound array to the next
  const __half* gb =
      reinterpret_cast<const __half*>(st + C::kQ4BoundsOffset + slot * C::kGroupBytes);
  const int gk = (D / 4) * t4 / 64;  // group of the lane's K channels
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = g + 8 * h;
    const uint8_t* src = st + slot * C::kCodeBytes + t * (D / 2) + (D / 8) * t4;
    if constexpr (D == 128) {
      const uint4 w = *reinterpret_cast<const uint4*>(src);
      r.kc[h][0] = w.x;
      r.kc[h][1] = w.y;
      r.kc[h][2] = w.z;
      r.kc[h][3] = w.w;
    } else {
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      r.kc[h][0] = w.x;
      r.kc[h][1] = w.y;
    }
    r.kmn[h] = gb[t * ng + gk];
    r.kx[h] = gb[kBound + t * ng + gk];
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = 2 * t4 + (i & 1) + 8 * (i >> 1);
    const uint8_t* src = st + C::kQ4VCodeOffset + slot * C::kCodeBytes + t * (D / 2) + (D / 16) * g;
    if constexpr (D == 128) {
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      r.vc[i][0] = w.x;
      r.vc[i][1] = w.y;
    } else {
      r.vc[i][0] = *reinterpret_cast<const uint32_t*>(src);
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = 2 * t4 + 8 * h;  // the pair (t, t + 1)
    const __half* vmn = gb + 2 * kBound + t * ng;
    const __half* vmx = gb + 3 * kBound + t * ng;
    if constexpr (D == 128) {
      const int gv = (D / 8) * g / 64;  // group of the lane's V channels
      const uint2 lo = *reinterpret_cast<const uint2*>(vmn);
      const uint2 hi = *reinterpret_cast<const uint2*>(vmx);
      r.vmn[h] = __byte_perm(lo.x, lo.y, gv ? 0x7632 : 0x5410);
      r.vx[h] = __byte_perm(hi.x, hi.y, gv ? 0x7632 : 0x5410);
    } else {
      r.vmn[h] = *reinterpret_cast<const uint32_t*>(vmn);
      r.vx[h] = *reinterpret_cast<const uint32_t*>(vmx);
    }
  }
}

// A landed 4-bit stage of `cnt` pages: the owning warp replaces every group's
// max by its fp16 step, each group once, unless a group of the stage is tiny
// (then the maxes stay and the stage's pages take the tiny-group path).
// Returns that warp-uniform flag.  The generic-proxy writes are fenced before
// the stage is handed back to the producer's bulk copies (q4_stage_release).
template <typename C, int D>
__device__ __forceinline__ bool q4_stage_steps(uint8_t* st, int cnt, int lane) {
  constexpr int ng = D / 64;
  constexpr int kBound = C::kPagesPerStage * kPage * ng;  // halves per bound array
  constexpr int kPer = (kBound + 31) / 32;                // groups per lane per tensor
  __half* gb = reinterpret_cast<__half*>(st + C::kQ4BoundsOffset);
  const int n = cnt * kPage * ng;  // groups per tensor in this stage
  __half step[2][kPer];
  bool tiny = false;
#pragma unroll
  for (int v = 0; v < 2; ++v) {  // K, V
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      step[v][i] = __ushort_as_half(0);
      if (e < n) {
        const float range = q4_range(gb[2 * v * kBound + e], gb[(2 * v + 1) * kBound + e]);
        tiny |= range < kQ4TinyRange;
        step[v][i] = q4_step16(fmaxf(range, kQ4TinyRange));
      }
    }
  }
  tiny = __any_sync(0xffffffffu, tiny);
  if (!tiny) {
#pragma unroll
    for (int v = 0; v < 2; ++v)
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (lane + 32 * i < n) gb[(2 * v + 1) * kBound + lane + 32 * i] = step[v][i];
  }
  __syncwarp();
  return tiny;
}

// Before a stage the consumers wrote to goes back to the producer's bulk
// copies: order those generic-proxy writes before the async proxy's.
__device__ __forceinline__ void q4_stage_release() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// (bits & mask) | bias, minus the bias: the masked nibbles as exact fp16 codes.
__device__ __forceinline__ __half2 q4_codes(uint32_t w, uint32_t mask, uint32_t bias) {
  const uint32_t x = (w & mask) | bias;
  return __hsub2(*reinterpret_cast<const __half2*>(&x), *reinterpret_cast<const __half2*>(&bias));
}

// A pair of codes of normal groups: fp16(code * step + mn), one rounding.
__device__ __forceinline__ uint32_t q4_value(__half2 code, __half2 step, __half2 mn) {
  const __half2 x = __hfma2(code, step, mn);
  return *reinterpret_cast<const uint32_t*>(&x);
}

// A pair of codes whose halves belong to the groups (mn.lo, mx.lo) and
// (mn.hi, mx.hi), normal or tiny.
__device__ __forceinline__ uint32_t q4_value_any(__half2 code, __half2 mn, __half2 mx) {
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const __half m = i ? __high2half(mn) : __low2half(mn);
    const __half M = i ? __high2half(mx) : __low2half(mx);
    const __half c = i ? __high2half(code) : __low2half(code);
    const float range = q4_range(m, M);
    const __half x =
        range >= kQ4TinyRange
            ? __hfma(c, q4_step16(range), m)
            : q4_level32(static_cast<uint32_t>(__half2float(c)), q4_step32(range, m, M),
                         __half2float(m));
    out |= static_cast<uint32_t>(__half_as_ushort(x)) << (16 * i);
  }
  return out;
}

constexpr uint32_t kNib0 = 0x000f000fu, kNib1 = 0x00f000f0u;
constexpr uint32_t kBias1024 = 0x64006400u, kBias64 = 0x54005400u;

// Query A fragments in the 4-bit path's channel order (see Q4Page).
template <int D>
__device__ __forceinline__ void q4_query(const uint16_t* qrow, bool head_ok, int t4,
                                         uint32_t (&qa)[D / 16][2]) {
#pragma unroll
  for (int j = 0; j < D / 32; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      w[u] = head_ok ? *reinterpret_cast<const uint32_t*>(qrow + (D / 4) * t4 + 8 * j + 2 * u)
                     : 0u;
    qa[2 * j][0] = __byte_perm(w[0], w[2], 0x5410);      // channels 0, 4
    qa[2 * j][1] = __byte_perm(w[0], w[2], 0x7632);      // 1, 5
    qa[2 * j + 1][0] = __byte_perm(w[1], w[3], 0x5410);  // 2, 6
    qa[2 * j + 1][1] = __byte_perm(w[1], w[3], 0x7632);  // 3, 7
  }
}

// S = Q K^T for a 4-bit page (sc[h]: tokens 8 h + 2 t4 + e, as the 16-bit path).
template <int D, bool TINY>
__device__ __forceinline__ void q4_scores_t(const Q4Page<D>& r, const uint32_t (&qa)[D / 16][2],
                                            float (&sc)[2][4]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const __half2 x2 = __half2half2(r.kx[h]), mn2 = __half2half2(r.kmn[h]);
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      const uint32_t w = r.kc[h][j], w8 = w >> 8;
      uint32_t b[4];
      const __half2 c[4] = {q4_codes(w, kNib0, kBias1024), q4_codes(w, kNib1, kBias64),
                            q4_codes(w8, kNib0, kBias1024), q4_codes(w8, kNib1, kBias64)};
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] = TINY ? q4_value_any(c[i], mn2, x2) : q4_value(c[i], x2, mn2);
      mma16816<true>(sc[h], qa[2 * j][0], 0u, qa[2 * j][1], 0u, b[0], b[1]);
      mma16816<true>(sc[h], qa[2 * j + 1][0], 0u, qa[2 * j + 1][1], 0u, b[2], b[3]);
    }
  }
}
template <int D>
__device__ __forceinline__ void q4_scores(const Q4Page<D>& r, const uint32_t (&qa)[D / 16][2],
                                          float (&sc)[2][4]) {
  if (r.tiny)
    q4_scores_t<D, true>(r, qa, sc);
  else
    q4_scores_t<D, false>(r, qa, sc);
}

// O += P V for a 4-bit page (a0-a3: the P fragments).
template <int D, bool TINY>
__device__ __forceinline__ void q4_pv_t(const Q4Page<D>& r, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, float (&acc)[D / 8][4]) {
#pragma unroll
  for (int j = 0; j < D / 64; ++j) {
    uint32_t bv[2][8];  // [token pair][nibble]: B fragments of tiles 8 j + nibble
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2 mn = *reinterpret_cast<const __half2*>(&r.vmn[h]);
      const __half2 x2 = *reinterpret_cast<const __half2*>(&r.vx[h]);
      const uint32_t wa = r.vc[2 * h][j], wb = r.vc[2 * h + 1][j];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        // Nibbles 4 hh .. 4 hh + 3 of both tokens, token 2 t4 (+ 8 h) in the low half.
        const uint32_t u = __byte_perm(wa, wb, hh ? 0x7632 : 0x5410), u8 = u >> 8;
        const __half2 c[4] = {q4_codes(u, kNib0, kBias1024), q4_codes(u, kNib1, kBias64),
                              q4_codes(u8, kNib0, kBias1024), q4_codes(u8, kNib1, kBias64)};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          bv[h][4 * hh + i] = TINY ? q4_value_any(c[i], mn, x2) : q4_value(c[i], x2, mn);
      }
    }
#pragma unroll
    for (int n = 0; n < 8; ++n) mma16816<true>(acc[8 * j + n], a0, a1, a2, a3, bv[0][n], bv[1][n]);
  }
}
template <int D>
__device__ __forceinline__ void q4_pv(const Q4Page<D>& r, uint32_t a0, uint32_t a1, uint32_t a2,
                                      uint32_t a3, float (&acc)[D / 8][4]) {
  if (r.tiny)
    q4_pv_t<D, true>(r, a0, a1, a2, a3, acc);
  else
    q4_pv_t<D, false>(r, a0, a1, a2, a3, acc);
}

// One query head per kv head (G = 1): the head-group MMA layout above would
// fill 1 of its 16 A rows.  Instead the page's tokens take the M side of
// S = K q (A = the K fragments the lane already builds, B = the query
// fragments, column 0) and its channels the M side of O^T = V^T P (A = the V
// fragments, B = the softmax weights as two columns, hi and lo): 16 MMAs a
// page instead of 32, and 32 accumulators instead of 64.  Scores land in
// lanes t4 = 0 (d[0]: token g, d[2]: token g + 8); output tile 4 j + m of
// lane (g, 0) holds channels D/8 g + 8 j + 2 m (d[0] + d[1]) and + 1
// (d[2] + d[3]).  (Layouts checked by a CPU emulation of the fragments.)
template <int D, bool TINY>
__device__ __forceinline__ void q4_scores_mha_t(const Q4Page<D>& r,
                                                const uint32_t (&qa)[D / 16][2], float (&sc)[4]) {
  __half2 x2[2], mn2[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    x2[h] = __half2half2(r.kx[h]);
    mn2[h] = __half2half2(r.kmn[h]);
  }
#pragma unroll
  for (int j = 0; j < D / 32; ++j) {
    uint32_t v[2][4];  // [token g, g + 8][nibble pairs (0,4) (1,5) (2,6) (3,7)]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t w = r.kc[h][j], w8 = w >> 8;
      const __half2 c[4] = {q4_codes(w, kNib0, kBias1024), q4_codes(w, kNib1, kBias64),
                            q4_codes(w8, kNib0, kBias1024), q4_codes(w8, kNib1, kBias64)};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        v[h][i] = TINY ? q4_value_any(c[i], mn2[h], x2[h]) : q4_value(c[i], x2[h], mn2[h]);
    }
    mma16816<true>(sc, v[0][0], v[1][0], v[0][1], v[1][1], qa[2 * j][0], qa[2 * j][1]);
    mma16816<true>(sc, v[0][2], v[1][2], v[0][3], v[1][3], qa[2 * j + 1][0], qa[2 * j + 1][1]);
  }
}
template <int D>
__device__ __forceinline__ void q4_scores_mha(const Q4Page<D>& r, const uint32_t (&qa)[D / 16][2],
                                              float (&sc)[4]) {
  if (r.tiny)
    q4_scores_mha_t<D, true>(r, qa, sc);
  else
    q4_scores_mha_t<D, false>(r, qa, sc);
}

template <int D, bool TINY>
__device__ __forceinline__ void q4_pv_mha_t(const Q4Page<D>& r, uint32_t b0, uint32_t b1,
                                            float (&acc)[D / 16][4]) {
#pragma unroll
  for (int j = 0; j < D / 64; ++j) {
    uint32_t bv[2][8];  // [token pair][nibble]: channel D/8 g + 8 j + nibble
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2 mn = *reinterpret_cast<const __half2*>(&r.vmn[h]);
      const __half2 x2 = *reinterpret_cast<const __half2*>(&r.vx[h]);
      const uint32_t wa = r.vc[2 * h][j], wb = r.vc[2 * h + 1][j];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t u = __byte_perm(wa, wb, hh ? 0x7632 : 0x5410), u8 = u >> 8;
        const __half2 c[4] = {q4_codes(u, kNib0, kBias1024), q4_codes(u, kNib1, kBias64),
                              q4_codes(u8, kNib0, kBias1024), q4_codes(u8, kNib1, kBias64)};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          bv[h][4 * hh + i] = TINY ? q4_value_any(c[i], mn, x2) : q4_value(c[i], x2, mn);
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m)
      mma16816<true>(acc[4 * j + m], bv[0][2 * m], bv[0][2 * m + 1], bv[1][2 * m],
                     bv[1][2 * m + 1], b0, b1);
  }
}
template <int D>
__device__ __forceinline__ void q4_pv_mha(const Q4Page<D>& r, uint32_t b0, uint32_t b1,
                                          float (&acc)[D / 16][4]) {
  if (r.tiny)
    q4_pv_mha_t<D, true>(r, b0, b1, acc);
  else
    q4_pv_mha_t<D, false>(r, b0, b1, acc);
}

__device__ __forceinline__ void store_out(void* out, int out_dtype, int64_t off, float v) {
  if (out_dtype == 2) {
    static_cast<float*>(out)[off] = v;
  } else if (out_dtype == 1) {
    static_cast<__half*>(out)[off] = __float2half_rn(v);
  } else {
    static_cast<__nv_bfloat16*>(out)[off] = __float2bfloat16_rn(v);
  }
}

// MHA: the 4-bit path's single-head layout (q4_scores_mha), for G = 1.
template <int D, bool F16, bool SPARSE, bool Q4, bool MHA = false>
__global__ void __launch_bounds__(kAttnThreads, MHA ? 3 : (D == 64 ? kAttnCtasPerSm : 0))
    attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mv) {
  using C = AttnCfg<D, Q4, Q4 && !SPARSE, MHA>;
  static_assert(!Q4 || F16, "a 4-bit cache is dequantised to fp16");
  static_assert(!MHA || Q4, "the single-head layout is the 4-bit path's");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full0 = sbase + C::kBarOffset;
  const uint32_t empty0 = full0 + 8 * C::kStages;
  const uint32_t dfull0 = empty0 + 8 * C::kStages;
  const uint32_t dempty0 = dfull0 + 16;
  int2* stage_meta = reinterpret_cast<int2*>(smem + C::kStageMetaOffset);
  volatile ItemDesc* desc = reinterpret_cast<volatile ItemDesc*>(smem + C::kDescOffset);
  float* mrg = reinterpret_cast<float*>(smem + C::kMergeOffset);
  int2* list = reinterpret_cast<int2*>(smem + C::kListOffset);
  int* blocks = reinterpret_cast<int*>(smem + C::kBlockOffset);  // paged: the item's pool blocks
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(dfull0 + 8 * s, 1);
      mbar_init(dempty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (!Q4 && warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&mk);
    prefetch_tensormap(&mv);
  }
  griddep_launch_dependents();
  // q, K, V, the selection and the work counter come from earlier kernels.
  // With per-unit ready flags the sparse path instead waits for each unit's
  // selection as it takes the unit's items (the selection kernel lets this
  // grid start only once every earlier kernel has finished).
  const bool unit_flags = SPARSE && a.unit_ready != nullptr;
  if (!unit_flags) griddep_wait();
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // Lane 0 fetches items and publishes their descriptors; the other lanes
    // help issue the copies.  Page j of an item goes to consumer warp j % 4.
    // 16-bit pages: lanes 0-7 issue one page (two tensor copies) each per
    // round, so lane l always feeds warp l % 4 (lanes l and l + 4 fill
    // consecutive slots of that warp's sub-ring).  4-bit pages: lanes
    // 6 w .. 6 w + 5 move the page of warp w, one bulk copy each, four pages per
    // round; lane 6 w waits for the free slot and arms its barrier first.  One
    // issuing thread would cap a CTA at a few copies per microsecond, far below
    // HBM bandwidth for pages of 1-8 KiB.
    static_assert(kConsumerWarps == 4, "four consumer sub-rings");
    constexpr int kIssueLanes = 8;
    constexpr int kQ4Parts = 6, kQ4IssueLanes = kQ4Parts * kConsumerWarps;
    const uint64_t pol = l2_evict_first_policy();
    const uint64_t pol_keep = l2_evict_last_policy();
    const bool hot = SPARSE && !Q4 && a.hot_stamp != nullptr;
    unsigned long long hot_loads = 0, hot_hits = 0;  // lane 0's running totals
    // consumer warp this lane feeds
    const int my_w = Q4 ? (lane < kQ4IssueLanes ? lane / kQ4Parts : 0) : (lane & 3);
    const int part = lane % kQ4Parts;  // 4-bit: which of the page's copies
    const bool drainer = Q4 ? (lane < kQ4IssueLanes && part == 0) : (lane < kConsumerWarps);
    int wc = 0;                     // pages issued so far to warp my_w
    int seq = 0;
    bool failed = false;            // a lane gave up waiting for a free slot
    for (int k = 0;; ++k) {
      // Next work item with pages (sparse chunks past a unit's union are
      // skipped here and never published).
      int item = 0, n = 0, b = 0, kvh = 0, first = 0;
      bool keep = false;  // reuse: the item's pages stay in L2 for the next step
      while (true) {
        if (lane == 0) item = static_cast<int>(atomicAdd(a.work_counter, 1u));
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item >= a.n_items) {
          item = -1;
          break;
        }
        const int chunk = item % a.n_chunks;
        const int unit = item / a.n_chunks;
        kvh = unit % a.Hkv;
        b = unit / a.Hkv;
        first = chunk * a.pages_per_chunk;
        if constexpr (SPARSE) {
          if (unit_flags) {
            int rdy = 1;
            if (lane == 0) rdy = flag_wait_bounded(a.unit_ready + unit, a.wait_limit_ns, abort_flag);
            if (!__shfl_sync(0xffffffffu, rdy, 0)) {
              if (lane == 0 && *abort_flag == 0) {
                set_status(a.status, kStatusTimeout);
                *abort_flag = 1;
              }
              item = -1;  // stop: publish the end of work
              break;
            }
          }
          const int count = __ldcg(a.union_count + unit);
          n = max(0, min(count - first, a.pages_per_chunk));
          if (n == 0) continue;
          const int2* src = a.union_list + static_cast<int64_t>(unit) * a.union_stride + first;
          for (int j = lane; j < n; j += 32) list[j] = __ldcg(src + j);
          if (hot) {
            // Cross-step reuse: each page of a unit's union is in exactly one
            // item, so its stamp has one writer per call.
            uint32_t* stamp = a.hot_stamp + static_cast<int64_t>(unit) * a.hot_pages;
            int hits = 0;
            for (int j = lane; j < n; j += 32) {
              const int page = __ldcg(src + j).x;
              const uint32_t last = stamp[page];
              stamp[page] = a.hot_step;
              hits += last != 0u && last + 1u == a.hot_step;
            }
            hits = __reduce_add_sync(0xffffffffu, hits);
            hot_loads += n;
            hot_hits += hits;
            keep = unit < a.hot_keep_units;
          }
          __syncwarp();
        } else {
          // (with per-sequence lengths, chunks past the sequence are skipped)
          const int Pb = static_cast<int>(ceil_div(seq_len_of(a.lens, b, a.N), kPage));
          n = max(0, min(Pb - first, a.pages_per_chunk));
          if (n == 0) continue;
        }
        if (a.bt != nullptr) {
          // paged cache: the pool block of each of the item's pages.  An
          // entry outside [0, num_blocks) is clamped into it, so no copy
          // leaves the pool, and reported as a failed check.
          for (int j = lane; j < n; j += 32) {
            const int page = SPARSE ? list[j].x : first + j;
            const int blk = a.bt[b * a.bts + page];
            if (blk < 0 || blk >= a.nblocks) set_status(a.status, kStatusCheck);
            blocks[j] = min(max(blk, 0), a.nblocks - 1);
          }
          __syncwarp();
        }
        break;
      }
      const int slot = k & 1;
      int ok = 1;
      if (lane == 0 && k >= 2) {
        ok = mbar_wait_bounded(dempty0 + 8 * slot, ((k >> 1) - 1) & 1, a.wait_limit_ns,
                               abort_flag);
        if (!ok && *abort_flag == 0) {
          set_status(a.status, kStatusTimeout);
          *abort_flag = 1;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (lane == 0) {
        desc[slot].item = item;
        desc[slot].n_pages = n;
        desc[slot].seq0 = seq;
        mbar_arrive(dfull0 + 8 * slot);  // release: consumers see the descriptor
      }
      if (item < 0) break;
      bool lok = true;
      if constexpr (Q4) {
        // Round: quads m0 .. m0 + 3 (quad m = pages 4 m .. 4 m + 3 of the
        // item) go to warps 0-3; lanes 6 w .. 6 w + 5 fill warp w's.
        constexpr int kQ = C::kPagesPerStage;
        for (int j0 = 0; j0 < n; j0 += kConsumerWarps * kQ) {
          const int m = j0 / kQ + my_w;  // this lane group's quad
          const int cnt = lane < kQ4IssueLanes ? max(0, min(kQ, n - m * kQ)) : 0;
          const bool mine = cnt > 0;
          const int c = wc + (m >> 2);   // stages issued to warp my_w so far
          const int s = my_w * C::kSub + c % C::kSub;
          int pg[kQ];
#pragma unroll
          for (int t = 0; t < kQ; ++t)
            pg[t] = t < cnt ? (SPARSE ? list[m * kQ + t].x : first + m * kQ + t) : 0;
          const uint32_t dst = sbase + s * C::kStageBytes;
          int ok = 1;
          if (mine && part == 0) {
            if (c >= C::kSub &&
                !mbar_wait_bounded(empty0 + 8 * s, ((c / C::kSub) - 1) & 1, a.wait_limit_ns,
                                   abort_flag)) {
              ok = 0;
            } else {
              uint32_t bytes = 0;
              for (int t = 0; t < cnt; ++t) {
                stage_meta[s * kQ + t] = make_int2(pg[t], SPARSE ? list[m * kQ + t].y : 0xff);
                const int nt = min(kPage, a.N - pg[t] * kPage);
                if (nt == kPage) {
                  bytes += C::kQ4PageBytes;
                } else {
                  q4_ragged_bounds<C, D>(a, b, kvh, pg[t], nt, t, smem + s * C::kStageBytes);
                  bytes += 2 * nt * (D / 2);
                }
              }
              mbar_arrive_expect_tx(full0 + 8 * s, bytes);  // (releases the plain stores)
            }
          }
          // The slot is free (and its barrier armed) before the quad's other
          // lanes copy into it.
          ok = __shfl_sync(0xffffffffu, ok, lane < kQ4IssueLanes ? my_w * kQ4Parts : lane);
          __syncwarp();
          if (mine && ok) {
            // runs of consecutive whole pages: one copy per part each
            for (int t = 0; t < cnt;) {
              const int nt = min(kPage, a.N - pg[t] * kPage);
              if (nt < kPage) {
                if (part == 0) q4_ragged_codes<C, D>(a, b, kvh, pg[t], nt, t, dst, full0 + 8 * s);
                ++t;
                continue;
              }
              int r = 1;
              while (t + r < cnt && pg[t + r] == pg[t] + r && (pg[t + r] + 1) * kPage <= a.N) ++r;
              q4_copy_run<C, D>(a, b, kvh, pg[t], r, t, part, dst, full0 + 8 * s);
              t += r;
            }
          }
          if (!__all_sync(0xffffffffu, !mine || ok)) {
            lok = false;
            break;
          }
        }
      } else {
        for (int j0 = 0; j0 < n; j0 += kIssueLanes) {
          const int j = j0 + lane;
          if (lane < kIssueLanes && j < n) {
            const int c = wc + (j >> 2);
            const int s = my_w * C::kSub + c % C::kSub;  // warp my_w's sub-ring, in order
            if (c >= C::kSub &&
                !mbar_wait_bounded(empty0 + 8 * s, ((c / C::kSub) - 1) & 1, a.wait_limit_ns,
                                   abort_flag)) {
              lok = false;
            } else {
              const int page = SPARSE ? list[j].x : first + j;
              stage_meta[s] = make_int2(page, SPARSE ? list[j].y : 0xff);
              const uint32_t dst = sbase + s * C::kStageBytes;
              mbar_arrive_expect_tx(full0 + 8 * s, C::kStageBytes);
              // {channel, token, half, kv head, batch} of the cache, or
              // {channel, token in block, half, kv head, block} of a pool
              const int y = a.bt != nullptr ? 0 : page * kPage;
              const int z = a.bt != nullptr ? blocks[j] : b;
              const uint64_t pl = keep ? pol_keep : pol;
              tma_load_5d_hint(dst, &mk, full0 + 8 * s, 0, y, 0, kvh, z, pl);
              tma_load_5d_hint(dst + C::kPageBytes, &mv, full0 + 8 * s, 0, y, 0, kvh, z, pl);
            }
          }
          if (!__all_sync(0xffffffffu, lok)) break;
        }
      }
      if constexpr (Q4) {
        const int nq = static_cast<int>(ceil_div(n, C::kPagesPerStage));  // the item's quads
        wc += nq > my_w ? (nq - my_w + 3) >> 2 : 0;
      } else {
        wc += n > my_w ? (n - my_w + 3) >> 2 : 0;
      }
      seq += n;
      if (!__all_sync(0xffffffffu, lok)) {
        failed = true;
        break;
      }
    }
    if (lane == 0 && failed && *abort_flag == 0) {
      set_status(a.status, kStatusTimeout);
      *abort_flag = 1;
    }
    __syncwarp();
    if (drainer && *abort_flag) {
      // Let every copy this CTA issued land before it exits.  A sub-ring holds
      // at most kSub copies in flight, so lane w waits for the last kSub slots
      // of warp w's sub-ring (slots never issued just run into the deadline).
      const uint64_t deadline = globaltimer_ns() + kDrainLimitNs;
      for (int c = max(0, wc - C::kSub); c < wc; ++c) {
        const uint64_t now = globaltimer_ns();
        if (now >= deadline) break;
        mbar_wait_bounded(full0 + 8 * (my_w * C::kSub + c % C::kSub), (c / C::kSub) & 1,
                          deadline - now, nullptr);
      }
    }
    __syncwarp();
    if (hot && lane == 0 && hot_loads > 0) {
      atomicAdd(a.hot_stats, hot_loads);
      atomicAdd(a.hot_stats + 1, hot_hits);
    }
    if (lane == 0) {
      // This CTA fetches no more work.  The last CTA to get here resets the
      // counters for the next call (every earlier fetch is ordered before its
      // exit ticket by the fence).
      __threadfence();
      if (atomicAdd(a.exit_counter, 1u) == gridDim.x - 1) {
        atomicExch(a.work_counter, 0u);
        atomicExch(a.exit_counter, 0u);
      }
    }
    // The grid ends only after the selection grid has (so the kernels after
    // this one, which wait for this grid alone, see every selection output).
    if (unit_flags) griddep_wait();
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, t4 = lane & 3;
  const bool head_ok = g < a.G;
  // Channel of output tile cn, column 2 t4 + e (the 4-bit path permutes them).
  auto out_channel = [](int cn, int t4_, int e) {
    return Q4 ? (D / 8) * (2 * t4_ + e) + cn : 8 * cn + 2 * t4_ + e;
  };
  const int mtx = lane >> 3, mrow = lane & 7;
  int mycnt = 0;  // pages this warp has taken from its sub-ring
  // Exits are taken by all four consumer warps together (consumers_any), so no
  // warp is ever left waiting at a consumer barrier.
  for (int k = 0;; ++k) {
    const int slot = k & 1;
    const bool dok = mbar_wait_bounded(dfull0 + 8 * slot, (k >> 1) & 1, a.wait_limit_ns,
                                       abort_flag);
    if (consumers_any(!dok)) {
      if (threadIdx.x == 0) {
        set_status(a.status, kStatusTimeout);
        *abort_flag = 1;
      }
      return;
    }
    const int item = desc[slot].item, n_pages = desc[slot].n_pages;
    if (item < 0) return;  // the same descriptor for every consumer warp
    const int chunk = item % a.n_chunks;
    const int unit = item / a.n_chunks;
    const int kvh = unit % a.Hkv, b = unit / a.Hkv;
    const int Nb = seq_len_of(a.lens, b, a.N);  // tokens this sequence attends

    uint32_t qa[D / 16][2];
    {
      const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + b * a.q_sb +
                             static_cast<int64_t>(kvh * a.G + (head_ok ? g : 0)) * a.q_sh;
      if constexpr (Q4) {
        q4_query<D>(qrow, head_ok, t4, qa);
      } else {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          qa[ks][0] = head_ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t4) : 0u;
          qa[ks][1] =
              head_ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t4 + 8) : 0u;
        }
      }
    }
    float m_run = -INFINITY, l_run = 0.f;
    constexpr int kAccTiles = MHA ? D / 16 : D / 8;
    float acc[kAccTiles][4];
#pragma unroll
    for (int cn = 0; cn < kAccTiles; ++cn) acc[cn][0] = acc[cn][1] = acc[cn][2] = acc[cn][3] = 0.f;

    bool aborted = false;
    // Stage q of the item goes to warp q % 4; it holds pages kQ q .. of the item.
    constexpr int kQ = C::kPagesPerStage;
    for (int sq = warp; sq * kQ < n_pages; sq += kConsumerWarps) {
      const int s = warp * C::kSub + mycnt % C::kSub;
      const bool ok = mbar_wait_bounded(full0 + 8 * s, (mycnt / C::kSub) & 1, a.wait_limit_ns,
                                        abort_flag);
      ++mycnt;
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          set_status(a.status, kStatusTimeout);
          *abort_flag = 1;
        }
        aborted = true;
        break;
      }
      const int cnt = min(kQ, n_pages - sq * kQ);
      bool stage_tiny = false;
      if constexpr (Q4) stage_tiny = q4_stage_steps<C, D>(smem + s * C::kStageBytes, cnt, lane);
      for (int t = 0; t < cnt; ++t) {
      const int2 meta = stage_meta[s * kQ + t];
      const int page = meta.x;
      const uint32_t hmask = static_cast<uint32_t>(meta.y);
      const uint32_t kb = sbase + s * C::kStageBytes, vb = kb + C::kPageBytes;

      // S = Q K^T for the page: sc[nt][e] = score of head g, token 8 nt + 2 t4 + e.
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      Q4Page<D> q4;  // 4-bit: the lane's codes and bounds of the page
      if constexpr (Q4) {
        // Everything the warp needs from the page goes to registers; after
        // the stage's last page, the stage is free.
        q4_load<C, D>(smem + s * C::kStageBytes, t, g, t4, stage_tiny, q4);
        if (t == cnt - 1) {
          q4_stage_release();
          __syncwarp();
          if (lane == 0) mbar_arrive(empty0 + 8 * s);
        }
        if constexpr (MHA)
          q4_scores_mha<D>(q4, qa, sc[0]);
        else
          q4_scores<D>(q4, qa, sc);
      } else {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(tile_addr(kb, 8 * (mtx >> 1) + mrow, 16 * ks + 8 * (mtx & 1)), r0, r1, r2, r3);
          mma16816<F16>(sc[0], qa[ks][0], 0u, qa[ks][1], 0u, r0, r1);
          mma16816<F16>(sc[1], qa[ks][0], 0u, qa[ks][1], 0u, r2, r3);
        }
      }

      if constexpr (MHA) {
        // One head: lanes t4 = 0 hold the page's scores, tokens g (sc[0][0])
        // and g + 8 (sc[0][2]).  Token t counts if bit t >> (4 - sub_log2)
        // of the mask is set (head 0's sub-page; bit 0 for whole pages).
        const int sl = SPARSE ? a.sub_log2 : 0;
        const int tk0 = page * kPage + g, tk1 = tk0 + 8;
        const bool on0 = (hmask >> (sl ? (g >> (4 - sl)) : 0)) & 1u;
        const bool on1 = (hmask >> (sl ? ((g + 8) >> (4 - sl)) : 0)) & 1u;
        const float s0 = (t4 == 0 && on0 && tk0 < Nb) ? sc[0][0] * a.scale_log2 : -INFINITY;
        const float s1 = (t4 == 0 && on1 && tk1 < Nb) ? sc[0][2] * a.scale_log2 : -INFINITY;
        // the page's largest score, warp-uniform, by one integer max over
        // order-preserving keys (a float's bits, the magnitude bits flipped
        // when negative; the map is its own inverse)
        const int kb = __float_as_int(fmaxf(s0, s1));
        const int km = __reduce_max_sync(0xffffffffu, kb >= 0 ? kb : kb ^ 0x7fffffff);
        const float pmax = __int_as_float(km >= 0 ? km : km ^ 0x7fffffff);
        const float m_new = fmaxf(m_run, pmax);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = exp2f(m_run - m_use);
        const float p0 = exp2f(s0 - m_use), p1 = exp2f(s1 - m_use);
        l_run = l_run * alpha + (p0 + p1);
        if (m_new != m_run) {
#pragma unroll
          for (int cn = 0; cn < kAccTiles; ++cn) {
            acc[cn][0] *= alpha;
            acc[cn][1] *= alpha;
            acc[cn][2] *= alpha;
            acc[cn][3] *= alpha;
          }
        }
        m_run = m_new;
        // B of O^T += V^T P: the weights of tokens 2 t4, 2 t4 + 1 (b0) and
        // 2 t4 + 8, 2 t4 + 9 (b1), their fp16 hi parts in column 0 (lanes
        // g = 0) and lo parts in column 1 (g = 1).
        const float x0 = __shfl_sync(0xffffffffu, p0, 8 * t4);
        const float x1 = __shfl_sync(0xffffffffu, p0, 8 * t4 + 4);
        const float y0 = __shfl_sync(0xffffffffu, p1, 8 * t4);
        const float y1 = __shfl_sync(0xffffffffu, p1, 8 * t4 + 4);
        uint32_t hx, lx, hy, ly;
        split_pair<true>(x0, x1, hx, lx);
        split_pair<true>(y0, y1, hy, ly);
        const uint32_t b0 = g == 0 ? hx : (g == 1 ? lx : 0u);
        const uint32_t b1 = g == 0 ? hy : (g == 1 ? ly : 0u);
        q4_pv_mha<D>(q4, b0, b1, acc);
      } else {
      // Online softmax (log2 domain) for head g over its 4 tokens of this page.
      // Token t of the page counts for head g if bit (g << sub_log2) +
      // (t >> (4 - sub_log2)) of the mask is set: the head selected its
      // sub-page, or the whole page when sub_log2 = 0.  This lane's tokens
      // 2 t4, 2 t4 + 1 share one sub-page, and 8 + 2 t4, 9 + 2 t4 the one
      // sub_log2 bits above it.
      const int sl = SPARSE ? a.sub_log2 : 0;
      const uint32_t hbits =
          head_ok ? (hmask >> ((g << sl) + (sl == 2 ? (t4 >> 1) : 0))) : 0u;
      const bool on_lo = hbits & 1u, on_hi = (hbits >> sl) & 1u;
      float sv[4];
      float pmax = -INFINITY;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = page * kPage + 8 * (e >> 1) + 2 * t4 + (e & 1);
        const bool on = e < 2 ? on_lo : on_hi;
        sv[e] = (on && tok < Nb) ? sc[e >> 1][e & 1] * a.scale_log2 : -INFINITY;
        pmax = fmaxf(pmax, sv[e]);
      }
      pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, 1));
      pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, 2));
      const float m_new = fmaxf(m_run, pmax);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m_run - m_use);
      float p[4];
      float psum = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p[e] = exp2f(sv[e] - m_use);
        psum += p[e];
      }
      l_run = l_run * alpha + psum;
      if (__any_sync(0xffffffffu, m_new != m_run)) {
#pragma unroll
        for (int cn = 0; cn < D / 8; ++cn) {
          acc[cn][0] *= alpha;
          acc[cn][1] *= alpha;
          acc[cn][2] *= alpha;
          acc[cn][3] *= alpha;
        }
      }
      m_run = m_new;

      // O += P V, with P = hi + lo (A rows 0-7 and 8-15).
      uint32_t a0, a1, a2, a3;
      split_pair<F16>(p[0], p[1], a0, a1);
      split_pair<F16>(p[2], p[3], a2, a3);
      if constexpr (Q4) {
        q4_pv<D>(q4, a0, a1, a2, a3, acc);
      } else {
        if ((a.bt != nullptr || a.lens != nullptr) && (page + 1) * kPage > Nb) {
          // A pool block's slots past N, or a cache's tokens past a shorter
          // sequence's end, hold anything: zero those V rows (their weights
          // are 0, but 0 * NaN is not).  The K rows' scores are masked.
          const int nt = Nb - page * kPage;
          uint8_t* vt = smem + s * C::kStageBytes + C::kPageBytes;
          const int per_half = (kPage - nt) * 8;  // 16-byte chunks
          for (int i = lane; i < (D / 64) * per_half; i += 32) {
            const int h = i / per_half, r = i % per_half;
            *reinterpret_cast<uint4*>(vt + (h * kPage + nt + r / 8) * 128 + (r % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
#pragma unroll
        for (int jn = 0; jn < D / 16; ++jn) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_trans(tile_addr(vb, 8 * (mtx & 1) + mrow, 8 * (2 * jn + (mtx >> 1))), r0, r1,
                        r2, r3);
          mma16816<F16>(acc[2 * jn], a0, a1, a2, a3, r0, r1);
          mma16816<F16>(acc[2 * jn + 1], a0, a1, a2, a3, r2, r3);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
      }
      }
      }
    }

    if constexpr (MHA) {
      // One head: the weight sums of lanes (g, 0) add up over g; lane (g, 0)
      // holds output channels D/8 g + 8 j + 2 m and + 1 of tile 4 j + m.
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 4);
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 8);
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
      auto channel = [g](int tile) { return (D / 8) * g + 8 * (tile >> 2) + 2 * (tile & 3); };
      if (consumers_any(aborted)) return;
      if (warp > 0) {
        float* r = mrg + (warp - 1) * C::kMergeRow;
        if (lane == 0) {
          r[D] = m_run;
          r[D + 1] = l_run;
        }
        if (t4 == 0) {
#pragma unroll
          for (int cn = 0; cn < kAccTiles; ++cn) {
            r[channel(cn)] = acc[cn][0] + acc[cn][1];
            r[channel(cn) + 1] = acc[cn][2] + acc[cn][3];
          }
        }
      }
      consumers_sync();
      if (warp == 0) {
        float M = m_run;
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) M = fmaxf(M, mrg[(w - 1) * C::kMergeRow + D]);
        float f[kConsumerWarps];
        f[0] = (m_run == -INFINITY) ? 0.f : exp2f(m_run - M);
        float L = f[0] * l_run;
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) {
          const float* r = mrg + (w - 1) * C::kMergeRow;
          f[w] = (r[D] == -INFINITY) ? 0.f : exp2f(r[D] - M);
          L += f[w] * r[D + 1];
        }
        const int64_t pi = (static_cast<int64_t>(b) * a.Hq + kvh * a.G) * a.n_chunks + chunk;
        const bool whole = Q4 && SPARSE && a.n_chunks == 1;  // out = O / L
        float* po = a.part_o + pi * D;
        const int64_t oo = b * a.o_sb + kvh * a.G * a.o_sh;
        if (t4 == 0) {
#pragma unroll
          for (int cn = 0; cn < kAccTiles; ++cn) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = channel(cn) + e;
              float O = f[0] * (acc[cn][2 * e] + acc[cn][2 * e + 1]);
#pragma unroll
              for (int w = 1; w < kConsumerWarps; ++w) O += f[w] * mrg[(w - 1) * C::kMergeRow + c];
              if (whole)
                store_out(a.out, a.out_dtype, oo + c, O / L);
              else
                po[c] = O;
            }
          }
        }
        if (lane == 0 && !whole) {
          a.part_ml[2 * pi] = M;
          a.part_ml[2 * pi + 1] = L;
        }
      }
    } else {
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);

    // Warps 1-3 hand their states to warp 0, which merges them with its own
    // (ascending warp order) and writes the item's partial.
    if (consumers_any(aborted)) return;
    if (warp > 0) {
      float* r = mrg + ((warp - 1) * 8 + g) * C::kMergeRow;
      if (t4 == 0) {
        r[D] = m_run;
        r[D + 1] = l_run;
      }
#pragma unroll
      for (int cn = 0; cn < D / 8; ++cn) {
        r[out_channel(cn, t4, 0)] = acc[cn][0] + acc[cn][2];
        r[out_channel(cn, t4, 1)] = acc[cn][1] + acc[cn][3];
      }
    }
    consumers_sync();
    if (warp == 0 && head_ok) {
      float M = m_run;
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w)
        M = fmaxf(M, mrg[((w - 1) * 8 + g) * C::kMergeRow + D]);
      float f[kConsumerWarps];
      f[0] = (m_run == -INFINITY) ? 0.f : exp2f(m_run - M);
      float L = f[0] * l_run;
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) {
        const float* r = mrg + ((w - 1) * 8 + g) * C::kMergeRow;
        f[w] = (r[D] == -INFINITY) ? 0.f : exp2f(r[D] - M);
        L += f[w] * r[D + 1];
      }
      const int64_t pi = (static_cast<int64_t>(b) * a.Hq + kvh * a.G + g) * a.n_chunks + chunk;
      const bool whole = Q4 && SPARSE && a.n_chunks == 1;  // out = O / L
      float* po = a.part_o + pi * D;
      const int64_t oo = b * a.o_sb + (kvh * a.G + g) * a.o_sh;
#pragma unroll
      for (int cn = 0; cn < D / 8; ++cn) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = out_channel(cn, t4, e);
          float O = f[0] * (acc[cn][e] + acc[cn][2 + e]);
#pragma unroll
          for (int w = 1; w < kConsumerWarps; ++w)
            O += f[w] * mrg[((w - 1) * 8 + g) * C::kMergeRow + c];
          if (whole)
            store_out(a.out, a.out_dtype, oo + c, O / L);
          else
            po[c] = O;
        }
      }
      if (t4 == 0 && !whole) {
        a.part_ml[2 * pi] = M;
        a.part_ml[2 * pi + 1] = L;
      }
    }
    }
    consumers_sync();  // merge area free again; the descriptor slot was read by all
    if (threadIdx.x == 0) mbar_arrive(dempty0 + 8 * slot);
  }
}

// One CTA per (b, h) row; D * S threads, S = ceil(n_chunks / 32) slices.
//   1. (m_k, l_k) of all chunks into shared memory; warp 0 takes the max M and
//      the weights w_k = 2^(m_k - M) (0 for empty chunks) and L = sum w_k l_k,
//      each lane over chunks lane, lane + 32, ... then a fixed shuffle tree.
//   2. thread (slice s, channel c) sums w_k o_k[c] over its <= 32 chunks with
//      every load in flight; the S slice sums are added in order.
// out = sum / L.  A fixed order throughout: deterministic.
template <int D>
__global__ void __launch_bounds__(1024) merge_kernel(const MergeArgs m) {
  __shared__ float s_w[kMaxChunks], s_l[kMaxChunks], s_o[kMaxChunks / 32][D];
  __shared__ float s_L;
  griddep_launch_dependents();
  griddep_wait();  // the attention grid has finished writing its partials
  const int row = blockIdx.x, stride = m.n_chunks;
  int nc = stride;  // chunks holding pages
  if (m.union_count != nullptr) {
    const int b = row / m.Hq, h = row % m.Hq;
    const int count = m.union_count[b * m.Hkv + h / m.G];
    nc = min(stride, static_cast<int>(ceil_div(count, m.pages_per_chunk)));
  } else if (m.lens != nullptr) {
    const int Pb = static_cast<int>(ceil_div(seq_len_of(m.lens, row / m.Hq, m.N), kPage));
    nc = min(stride, static_cast<int>(ceil_div(Pb, m.pages_per_chunk)));
  }
  const float* ml = m.part_ml + static_cast<int64_t>(row) * stride * 2;
  for (int k = threadIdx.x; k < nc; k += blockDim.x) {
    s_w[k] = __ldcg(ml + 2 * k);
    s_l[k] = __ldcg(ml + 2 * k + 1);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float M = -INFINITY;
    for (int k = lane; k < nc; k += 32) M = fmaxf(M, s_w[k]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int k = lane; k < nc; k += 32) {
      const float w = (s_w[k] == -INFINITY) ? 0.f : exp2f(s_w[k] - M);
      L += w * s_l[k];
      s_w[k] = w;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) s_L = L;
  }
  __syncthreads();
  const int c = threadIdx.x % D, sl = threadIdx.x / D;
  const int k0 = sl * 32, k1 = min(nc, k0 + 32);
  const float* po = m.part_o + (static_cast<int64_t>(row) * stride + k0) * D + c;
  float x[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) x[i] = (k0 + i < k1) ? __ldcg(po + static_cast<int64_t>(i) * D) : 0.f;
  float O = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float w = (k0 + i < k1) ? s_w[k0 + i] : 0.f;
    O += (w != 0.f) ? w * x[i] : 0.f;  // empty chunks hold no o values
  }
  s_o[sl][c] = O;
  __syncthreads();
  if (threadIdx.x < D) {
    float sum = 0.f;
    for (int i = 0; i < blockDim.x / D; ++i) sum += s_o[i][c];
    const int b = row / m.Hq, h = row % m.Hq;
    store_out(m.out, m.out_dtype, b * m.o_sb + h * m.o_sh + c, sum / s_L);
  }
}

// Units of at most kSmallMergeChunks chunks (the usual case): one thread per
// (row, channel), 256 / D rows per CTA.  Every load a thread needs -- the
// union count, all (m_k, l_k) and its channel of all o_k -- is issued at once,
// so the merge costs one memory round trip; then, in chunk order,
// M = max m_k, w_k = 2^(m_k - M) (0 for empty chunks), L = sum w_k l_k,
// out = (sum w_k o_k) / L.  Deterministic like merge_kernel.
constexpr int kSmallMergeChunks = 32;
constexpr int kSmallMergeThreads = 256;

template <int D>
__global__ void __launch_bounds__(kSmallMergeThreads) merge_small_kernel(const MergeArgs m,
                                                                         int rows) {
  griddep_launch_dependents();
  griddep_wait();  // the attention grid has finished writing its partials
  const int row = blockIdx.x * (kSmallMergeThreads / D) + threadIdx.x / D;
  const int c = threadIdx.x % D;
  if (row >= rows) return;
  const int stride = m.n_chunks;
  const int b = row / m.Hq, h = row % m.Hq;
  const int count = m.union_count != nullptr
                        ? __ldcg(m.union_count + b * m.Hkv + h / m.G)
                        : (m.lens != nullptr
                               ? static_cast<int>(ceil_div(seq_len_of(m.lens, b, m.N), kPage))
                               : 0);
  const float2* ml = reinterpret_cast<const float2*>(m.part_ml) + static_cast<int64_t>(row) * stride;
  const float* po = m.part_o + static_cast<int64_t>(row) * stride * D + c;
  float2 mlv[kSmallMergeChunks];
  float x[kSmallMergeChunks];
#pragma unroll
  for (int k = 0; k < kSmallMergeChunks; ++k) {
    mlv[k] = k < stride ? __ldcg(ml + k) : make_float2(-INFINITY, 0.f);
    x[k] = k < stride ? __ldcg(po + static_cast<int64_t>(k) * D) : 0.f;
  }
  const int nc = (m.union_count != nullptr || m.lens != nullptr)
                     ? min(stride, static_cast<int>(ceil_div(count, m.pages_per_chunk)))
                     : stride;
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kSmallMergeChunks; ++k)
    if (k < nc) M = fmaxf(M, mlv[k].x);
  float L = 0.f, O = 0.f;
#pragma unroll
  for (int k = 0; k < kSmallMergeChunks; ++k) {
    if (k < nc) {
      const float w = (mlv[k].x == -INFINITY) ? 0.f : exp2f(mlv[k].x - M);
      L += w * mlv[k].y;
      O += (w != 0.f) ? w * x[k] : 0.f;  // empty chunks hold no o values
    }
  }
  store_out(m.out, m.out_dtype, b * m.o_sb + h * m.o_sh + c, O / L);
}

// Resident CTAs per SM of one attention instantiation (its registers and shared
// memory as compiled), at most kAttnCtasPerSm; computed once.
template <int D, bool F16, bool SPARSE, bool Q4, bool MHA = false>
cudaError_t attn_ctas_per_sm_t(int* out) {
  using C = AttnCfg<D, Q4, Q4 && !SPARSE, MHA>;
  static int cached = 0;  // benign race: every thread computes the same value
  if (cached > 0) {
    *out = cached;
    return cudaSuccess;
  }
  auto kern = attn_kernel<D, F16, SPARSE, Q4, MHA>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kAttnThreads, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  cached = n < C::kCtasPerSm ? n : C::kCtasPerSm;
  *out = cached;
  return cudaSuccess;
}

template <int D, bool F16, bool SPARSE, bool Q4, bool MHA = false>
cudaError_t launch_attn_t(const AttnArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                          int num_sms, cudaStream_t s) {
  using C = AttnCfg<D, Q4, Q4 && !SPARSE, MHA>;
  int per_sm = 0;
  cudaError_t e = attn_ctas_per_sm_t<D, F16, SPARSE, Q4, MHA>(&per_sm);
  if (e != cudaSuccess) return e;
  const int64_t want = static_cast<int64_t>(num_sms) * per_sm;
  const int grid = static_cast<int>(a.n_items < want ? a.n_items : want);
  return launch_pdl(attn_kernel<D, F16, SPARSE, Q4, MHA>, dim3(grid), dim3(kAttnThreads),
                    C::kSmemBytes, s, a, mk, mv);
}

}  // namespace

cudaError_t launch_attn(int d, bool f16, bool sparse, const AttnArgs& a, const CUtensorMap& mk,
                        const CUtensorMap& mv, int num_sms, cudaStream_t s) {
  if (d == 128) {
    if (f16) return sparse ? launch_attn_t<128, true, true, false>(a, mk, mv, num_sms, s)
                           : launch_attn_t<128, true, false, false>(a, mk, mv, num_sms, s);
    return sparse ? launch_attn_t<128, false, true, false>(a, mk, mv, num_sms, s)
                  : launch_attn_t<128, false, false, false>(a, mk, mv, num_sms, s);
  }
  if (f16) return sparse ? launch_attn_t<64, true, true, false>(a, mk, mv, num_sms, s)
                         : launch_attn_t<64, true, false, false>(a, mk, mv, num_sms, s);
  return sparse ? launch_attn_t<64, false, true, false>(a, mk, mv, num_sms, s)
                : launch_attn_t<64, false, false, false>(a, mk, mv, num_sms, s);
}

cudaError_t launch_attn_q4(int d, bool sparse, const AttnArgs& a, int num_sms, cudaStream_t s) {
  CUtensorMap unused;  // the 4-bit path moves pages with 1-D bulk copies
  memset(&unused, 0, sizeof unused);
  if (a.G == 1) {  // one query head per kv head: the single-head layout
    if (d == 128)
      return sparse ? launch_attn_t<128, true, true, true, true>(a, unused, unused, num_sms, s)
                    : launch_attn_t<128, true, false, true, true>(a, unused, unused, num_sms, s);
    return sparse ? launch_attn_t<64, true, true, true, true>(a, unused, unused, num_sms, s)
                  : launch_attn_t<64, true, false, true, true>(a, unused, unused, num_sms, s);
  }
  if (d == 128)
    return sparse ? launch_attn_t<128, true, true, true>(a, unused, unused, num_sms, s)
                  : launch_attn_t<128, true, false, true>(a, unused, unused, num_sms, s);
  return sparse ? launch_attn_t<64, true, true, true>(a, unused, unused, num_sms, s)
                : launch_attn_t<64, true, false, true>(a, unused, unused, num_sms, s);
}

cudaError_t attn_ctas_per_sm(int d, bool f16, bool sparse, bool q4, int* out) {
  if (q4) {
    if (d == 128) return sparse ? attn_ctas_per_sm_t<128, true, true, true>(out)
                                : attn_ctas_per_sm_t<128, true, false, true>(out);
    return sparse ? attn_ctas_per_sm_t<64, true, true, true>(out)
                  : attn_ctas_per_sm_t<64, true, false, true>(out);
  }
  if (d == 128) {
    if (f16) return sparse ? attn_ctas_per_sm_t<128, true, true, false>(out)
                           : attn_ctas_per_sm_t<128, true, false, false>(out);
    return sparse ? attn_ctas_per_sm_t<128, false, true, false>(out)
                  : attn_ctas_per_sm_t<128, false, false, false>(out);
  }
  if (f16) return sparse ? attn_ctas_per_sm_t<64, true, true, false>(out)
                         : attn_ctas_per_sm_t<64, true, false, false>(out);
  return sparse ? attn_ctas_per_sm_t<64, false, true, false>(out)
                : attn_ctas_per_sm_t<64, false, false, false>(out);
}

cudaError_t launch_merge(int d, const MergeArgs& m, int rows, cudaStream_t s) {
  if (m.n_chunks <= kSmallMergeChunks) {
    const dim3 grid(static_cast<unsigned>(ceil_div(rows, kSmallMergeThreads / d)));
    return d == 128 ? launch_pdl(merge_small_kernel<128>, grid, dim3(kSmallMergeThreads), 0, s, m,
                                 rows)
                    : launch_pdl(merge_small_kernel<64>, grid, dim3(kSmallMergeThreads), 0, s, m,
                                 rows);
  }
  const int slices = static_cast<int>(ceil_div(m.n_chunks, 32));
  const dim3 grid(rows), block(d * slices);
  return d == 128 ? launch_pdl(merge_kernel<128>, grid, block, 0, s, m)
                  : launch_pdl(merge_kernel<64>, grid, block, 0, s, m);
}

}  // namespace dkv

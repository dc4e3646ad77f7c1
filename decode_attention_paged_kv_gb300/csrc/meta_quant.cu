// meta_quant.cu -- page metadata build and the 4-bit KV format.
//
// Page metadata ("TinyServe: Query-Aware Cache Selection for Efficient LLM
// Serving", 结构化内存布局 / 相关性函数实例化): for every page of S tokens, m_j
// and M_j are the channel-wise min / max of the page's keys.  One thread owns
// 8 channels of one page (of a 16-token cache page for S = 4 and 8): it
// streams the rows as 16-byte vectors -- a warp covers whole contiguous
// 256-byte key rows -- and reduces on order-preserving 16-bit keys with
// per-halfword integer min / max, so the result is exactly one of the stored
// values (-0 below +0).  A 4-bit cache is dequantised in registers first (its
// own kernel, meta_q4_kernel); its metadata describes the fp16 keys that
// attention actually uses.  The 8-bit metadata of the same pages (a byte grid
// per page, rounded outward) is built from the 16-bit one (meta8_kernel).
//
// 4-bit format ("FlexGen: High-Throughput Generative Inference of Large
// Language Models with a Single GPU" 解读, 4-bit 近似方法): groups of 64
// channels of one (token, head) row; per-group min / max in fp16; 16 levels
// mn + c * s with the step s rounded down from (max - min) / 15 (an fp16 step,
// or an fp32 one for groups narrower than 451 * 2^-24); codes are the nearest
// level; values are dequantised back to fp16 by rounding the exact level once.

#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {
namespace {

constexpr int kMetaThreads = 256;

// Two fp32 values in one 64-bit register pair, and the packed fp32 pair
// arithmetic of sm_100 and later (each lane rounded as the scalar operation
// with the same rounding mode; subnormals kept).
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// rounded down: an exact zero difference is -0 (IEEE 754, rounding toward
// negative), so the sign bit of a - b is set exactly when a <= b
__device__ __forceinline__ uint64_t f2_sub_down(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rm.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add_down(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rm.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add_up(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rp.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint32_t lo32(uint64_t v) { return static_cast<uint32_t>(v); }
__device__ __forceinline__ uint32_t hi32(uint64_t v) { return static_cast<uint32_t>(v >> 32); }


__global__ void __launch_bounds__(kMetaThreads, 2) meta_kernel(const MetaArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  const int vpr = a.d / 8;  // 16-byte vectors per row
  // every page, or (last_only) one page per (batch, kv head)
  const int pages = a.last_only ? 1 : a.P;
  const int64_t total = static_cast<int64_t>(a.B) * a.Hkv * pages * vpr;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(idx % vpr);
    const int64_t bh = idx / vpr / pages;
    const int h = static_cast<int>(bh % a.Hkv);
    const int b = static_cast<int>(bh / a.Hkv);
    const int Nb = seq_len_of(a.lens, b, a.N);
    // the page holding the sequence's newest token, or page idx / vpr % P
    const int page = a.last_only ? (Nb - 1) / a.S : static_cast<int>(idx / vpr % a.P);
    const int64_t pg = bh * a.P + page;  // (b * Hkv + h) * P + page
    const int t0 = page * a.S;  // a metadata page of S tokens
    if (t0 >= Nb) continue;  // past a shorter sequence: not written
    const int nt = min(a.S, Nb - t0);
    uint32_t kmin[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
    uint32_t kmax[4] = {0u, 0u, 0u, 0u};
    // the metadata page's 16-token cache pages, one at a time
#pragma unroll 1
    for (int c0 = 0; c0 < nt; c0 += kPage) {
      const int cp = (t0 + c0) / kPage;  // cache page
      const int ntc = min(kPage, nt - c0);
      // a paged cache: the cache page's pool block (clamped), token 0 of it
      // (a page of 4 or 8 tokens starts inside its block)
      const int64_t base = a.bt != nullptr
                               ? static_cast<int64_t>(min(max(a.bt[b * a.bts + cp], 0),
                                                          a.nblocks - 1)) * a.sb +
                                     static_cast<int64_t>((t0 + c0) % kPage) * a.d
                               : b * a.sb + static_cast<int64_t>(t0 + c0) * a.d;
      const uint16_t* src = static_cast<const uint16_t*>(a.data) + base + h * a.sh + 8 * v;
      uint4 x[kPage];
#pragma unroll
      for (int t = 0; t < kPage; ++t)
        if (t < ntc)
          x[t] = __ldcs(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(t) * a.d));
#pragma unroll
      for (int t = 0; t < kPage; ++t) {
        if (t < ntc) {
          const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t k = to_key2(w[u]);
            kmin[u] = __vminu2(kmin[u], k);
            kmax[u] = __vmaxu2(kmax[u], k);
          }
        }
      }
    }
    uint4 omin, omax;
    omin.x = from_key2(kmin[0]);
    omin.y = from_key2(kmin[1]);
    omin.z = from_key2(kmin[2]);
    omin.w = from_key2(kmin[3]);
    omax.x = from_key2(kmax[0]);
    omax.y = from_key2(kmax[1]);
    omax.z = from_key2(kmax[2]);
    omax.w = from_key2(kmax[3]);
    const int64_t o = pg * a.d + 8 * v;
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.meta_min) + o) = omin;
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.meta_max) + o) = omax;
  }
}

// Pages of S = 16 / SUBS tokens (8 or 4) over a 16-bit cache: one thread owns 8
// channels of a whole 16-token cache page (its 16 rows in flight, as for
// S = 16) and writes the page's SUBS metadata pages, each from its own S rows
// -- rather than a thread per S-token page with S rows in flight.
template <int SUBS>
__global__ void __launch_bounds__(kMetaThreads, 2) meta_sub_kernel(const MetaArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  constexpr int S = kPage / SUBS;
  const int vpr = a.d / 8;  // 16-byte vectors per row
  const int P16 = static_cast<int>(ceil_div(a.N, kPage));
  const int64_t total = static_cast<int64_t>(a.B) * a.Hkv * P16 * vpr;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(idx % vpr);
    const int cp = static_cast<int>(idx / vpr % P16);  // cache page
    const int64_t bh = idx / vpr / P16;
    const int h = static_cast<int>(bh % a.Hkv);
    const int b = static_cast<int>(bh / a.Hkv);
    const int Nb = seq_len_of(a.lens, b, a.N);
    const int t0 = cp * kPage;
    if (t0 >= Nb) continue;  // past a shorter sequence: not written
    const int nt = min(kPage, Nb - t0);
    // a paged cache: the cache page's pool block (clamped)
    const int64_t base = a.bt != nullptr
                             ? static_cast<int64_t>(min(max(a.bt[b * a.bts + cp], 0),
                                                        a.nblocks - 1)) * a.sb
                             : b * a.sb + static_cast<int64_t>(t0) * a.d;
    const uint16_t* src = static_cast<const uint16_t*>(a.data) + base + h * a.sh + 8 * v;
    uint4 x[kPage];
#pragma unroll
    for (int t = 0; t < kPage; ++t)
      if (t < nt) x[t] = __ldcs(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(t) * a.d));
#pragma unroll
    for (int sp = 0; sp < SUBS; ++sp) {
      if (sp * S >= nt) break;  // past the sequence: not written
      uint32_t kmin[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      uint32_t kmax[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int t = sp * S; t < sp * S + S; ++t) {
        if (t < nt) {
          const uint32_t w[4] = {x[t].x, x[t].y, x[t].z, x[t].w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t k = to_key2(w[u]);
            kmin[u] = __vminu2(kmin[u], k);
            kmax[u] = __vmaxu2(kmax[u], k);
          }
        }
      }
      const int64_t o = (bh * a.P + static_cast<int64_t>(cp) * SUBS + sp) * a.d + 8 * v;
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.meta_min) + o) =
          make_uint4(from_key2(kmin[0]), from_key2(kmin[1]), from_key2(kmin[2]), from_key2(kmin[3]));
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.meta_max) + o) =
          make_uint4(from_key2(kmax[0]), from_key2(kmax[1]), from_key2(kmax[2]), from_key2(kmax[3]));
    }
  }
}

// A 4-bit cache: D/16 lanes per page, lane u owning channels 16u .. 16u + 15
// (two code words of a token row, one 8-byte load).  One row of blocks per
// (batch, kv head) (grid y), a warp over 32/(D/16) consecutive pages of it, so
// every lane of a warp runs the same chunks of 8 tokens (those of the warp's
// first page; a shorter page's extra tokens are skipped) and full-warp
// shuffles and votes are safe.  The four lanes of a group share its steps: per
// chunk each computes two and the others take them by shuffle.  A normal
// group's levels fl16(c * step + mn) are multiples of 2^-24, so they are never
// -0 and fp16 min / max (two lanes at a time) is exact on them; the nibble
// pairs (c, c + 4) of a code word are dequantised together and the order
// restored once per page.  When a chunk of the warp holds a narrow group (the
// fp32 step), its pages are taken again from their first token, token by
// token, on order-preserving keys (-0 below +0).
// One token's 16 channels into the running fp16 min / max.  Nibble pairs
// (c, c + 4) of a code word become exact fp16 codes by the exponent trick:
// bits 0-3 under 1024.0 (ulp 1) and bits 4-7 under 64.0 (ulp 1/16) give
// 1024 + c and 64 + c, so one shift of the word by 8 and four masks reach all
// four pairs; then c = that - 1024 (or - 64) and fl16(c step + mn), one fused
// rounding as the format defines.  All on packed registers.
__device__ __forceinline__ uint32_t h2_level(uint32_t bits, uint32_t bias, uint32_t st2,
                                            uint32_t mn2) {
  uint32_t c, x;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(c) : "r"(bits), "r"(bias));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(x) : "r"(c), "r"(st2), "r"(mn2));
  return x;
}
__device__ __forceinline__ void h2_minmax(uint32_t& lo, uint32_t& hi, uint32_t x) {
  asm("min.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(x));
  asm("max.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(x));
}
__device__ __forceinline__ void q4_minmax_token(uint2 cw, uint32_t ms, uint32_t (&hmin)[8],
                                                uint32_t (&hmax)[8]) {
  const uint32_t mn2 = __byte_perm(ms, 0u, 0x1010u), st2 = __byte_perm(ms, 0u, 0x3232u);
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t w = j ? cw.y : cw.x, w8 = w >> 8;
    h2_minmax(hmin[4 * j], hmax[4 * j],
              h2_level((w & 0x000f000fu) | 0x64006400u, 0x64006400u, st2, mn2));
    h2_minmax(hmin[4 * j + 1], hmax[4 * j + 1],
              h2_level((w & 0x00f000f0u) | 0x54005400u, 0x54005400u, st2, mn2));
    h2_minmax(hmin[4 * j + 2], hmax[4 * j + 2],
              h2_level((w8 & 0x000f000fu) | 0x64006400u, 0x64006400u, st2, mn2));
    h2_minmax(hmin[4 * j + 3], hmax[4 * j + 3],
              h2_level((w8 & 0x00f000f0u) | 0x54005400u, 0x54005400u, st2, mn2));
  }
}

template <int D>
__global__ void __launch_bounds__(kMetaThreads, 4) meta_q4_kernel(const MetaArgs a) {
  griddep_launch_dependents();
  griddep_wait();
  constexpr int LPP = D / 16;  // lanes per page
  constexpr int NG = D / 64;   // groups per token row
  constexpr unsigned kFull = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int u = lane % LPP, g = u >> 2;
  const int lin = blockIdx.x * blockDim.x + threadIdx.x;
  const int wpage = (lin - lane) / LPP;  // the warp's first page slot
  for (int bh = blockIdx.y; bh < a.B * a.Hkv; bh += gridDim.y) {
    const int h = bh % a.Hkv, b = bh / a.Hkv;
    const int Nb = seq_len_of(a.lens, b, a.N);
    // page slot -> page: every page, or (last_only) slot 0 is the newest token's page
    const int slot = lin / LPP;
    const int last = (Nb - 1) / a.S;
    const bool live = a.last_only ? slot == 0 : slot < a.P;
    const int page = a.last_only ? last : slot;
    const int nt = live ? max(0, min(a.S, Nb - page * a.S)) : 0;
    // tokens of the warp's first and last pages (pages are consecutive)
    const int wfirst = a.last_only ? (wpage == 0 ? last : a.P) : wpage;
    const int wlast = a.last_only ? wfirst : wpage + 32 / LPP - 1;
    const int nt_first = wfirst < a.P ? max(0, min(a.S, Nb - wfirst * a.S)) : 0;
    const int nt_last = wlast < a.P ? max(0, min(a.S, Nb - wlast * a.S)) : 0;
    const int t0 = page * a.S;
    const uint8_t* src = static_cast<const uint8_t*>(a.data) + b * a.sb + h * a.sh +
                         static_cast<int64_t>(t0) * (D / 2) + 8 * u;
    const int64_t goff = b * a.gsb + h * a.gsh + static_cast<int64_t>(t0) * NG + g;
    const __half* gmn = static_cast<const __half*>(a.gmin) + goff;
    const __half* gmx = static_cast<const __half*>(a.gmax) + goff;
    uint32_t omin[8], omax[8];
    bool narrow_page = false;
    {
      uint32_t hmin[8], hmax[8];  // fp16 pairs (c, c + 4) of each code word
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        hmin[i] = 0x7c007c00u;  // +inf
        hmax[i] = 0xfc00fc00u;  // -inf
      }
#pragma unroll 1
      for (int c0 = 0; c0 < nt_first; c0 += 8) {
        const bool full = c0 + 8 <= nt_last;  // every page of the warp: a whole chunk
        uint2 cw[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (full || c0 + k < nt)
            cw[k] = __ldcs(reinterpret_cast<const uint2*>(src + static_cast<int64_t>(c0 + k) *
                                                                    (D / 2)));
        uint32_t own[2];  // (mn, step) of tokens c0 + 2 (u & 3) + e, as a half pair
        bool narrow = false;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = c0 + 2 * (u & 3) + e;
          own[e] = 0u;
          if (t < nt) {
            const __half mn = gmn[static_cast<int64_t>(t) * NG];
            const __half mx = gmx[static_cast<int64_t>(t) * NG];
            const float range = q4_range(mn, mx);
            narrow |= range < kQ4TinyRange;
            own[e] = static_cast<uint32_t>(__half_as_ushort(mn)) |
                     (static_cast<uint32_t>(
                          __half_as_ushort(q4_step16(fmaxf(range, kQ4TinyRange))))
                      << 16);
          }
        }
        if (__any_sync(kFull, narrow)) {
          narrow_page = true;
          break;
        }
        uint32_t ms[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ms[k] = __shfl_sync(kFull, own[k & 1], k >> 1, 4);
        if (full) {
#pragma unroll
          for (int k = 0; k < 8; ++k) q4_minmax_token(cw[k], ms[k], hmin, hmax);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (c0 + k < nt) q4_minmax_token(cw[k], ms[k], hmin, hmax);
        }
      }
      // pairs (c0, c4) (c1, c5) (c2, c6) (c3, c7) -> (c0, c1) (c2, c3) (c4, c5) (c6, c7)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t* pn = hmin + 4 * j;
        const uint32_t* px = hmax + 4 * j;
        omin[4 * j] = __byte_perm(pn[0], pn[1], 0x5410u);
        omin[4 * j + 1] = __byte_perm(pn[2], pn[3], 0x5410u);
        omin[4 * j + 2] = __byte_perm(pn[0], pn[1], 0x7632u);
        omin[4 * j + 3] = __byte_perm(pn[2], pn[3], 0x7632u);
        omax[4 * j] = __byte_perm(px[0], px[1], 0x5410u);
        omax[4 * j + 1] = __byte_perm(px[2], px[3], 0x5410u);
        omax[4 * j + 2] = __byte_perm(px[0], px[1], 0x7632u);
        omax[4 * j + 3] = __byte_perm(px[2], px[3], 0x7632u);
      }
    }
    if (nt == 0) continue;  // no page here (after the warp's shuffles and votes)
    if (narrow_page) {
      // the whole page again, token by token, on order-preserving keys
      uint32_t kmin[8], kmax[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        kmin[i] = 0xffffffffu;
        kmax[i] = 0u;
      }
      for (int t = 0; t < nt; ++t) {
        const uint2 c =
            __ldcs(reinterpret_cast<const uint2*>(src + static_cast<int64_t>(t) * (D / 2)));
        const __half mn = gmn[static_cast<int64_t>(t) * NG];
        const __half mx = gmx[static_cast<int64_t>(t) * NG];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t w[4];
          q4_dequant8(j ? c.y : c.x, mn, mx, w);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t k = to_key2(w[i]);
            kmin[4 * j + i] = __vminu2(kmin[4 * j + i], k);
            kmax[4 * j + i] = __vmaxu2(kmax[4 * j + i], k);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        omin[i] = from_key2(kmin[i]);
        omax[i] = from_key2(kmax[i]);
      }
    }
    const int64_t pg = static_cast<int64_t>(bh) * a.P + page;
    uint4* dmin = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.meta_min) + pg * D + 16 * u);
    uint4* dmax = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.meta_max) + pg * D + 16 * u);
    dmin[0] = make_uint4(omin[0], omin[1], omin[2], omin[3]);
    dmin[1] = make_uint4(omin[4], omin[5], omin[6], omin[7]);
    dmax[0] = make_uint4(omax[0], omax[1], omax[2], omax[3]);
    dmax[1] = make_uint4(omax[4], omax[5], omax[6], omax[7]);
  }
}

// One predicated 16-bit store (no branch when the lanes differ on c).
__device__ __forceinline__ void st_global_u16_if(void* p, unsigned short v, bool c) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.global.u16 [%0], %1;\n\t}"
               :
               : "l"(p), "h"(v), "r"(static_cast<uint32_t>(c))
               : "memory");
}

constexpr float kRint23 = 8388608.0f;      // 2^23: x + 2^23 holds rint(x) in its low bits
constexpr uint32_t kRint23Bits = 0x4b000000u;  // the float bits of 2^23

// One thread's 16 channels of group t / 4 (every lane of the warp calls it:
// the group's min / max go round its 4 lanes).
__device__ __forceinline__ void quant4_part(const uint4 (&xv)[2], int64_t t, bool valid,
                                            uint8_t* codes, __half* gmin, __half* gmax) {
  const int64_t grp = t >> 2;
  const int quarter = static_cast<int>(t & 3);
  const uint32_t w[8] = {xv[0].x, xv[0].y, xv[0].z, xv[0].w, xv[1].x, xv[1].y, xv[1].z, xv[1].w};
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint32_t k = to_key2(w[u]);
    kmin = __vminu2(kmin, k);
    kmax = __vmaxu2(kmax, k);
  }
  // fold the two halfwords, then the 4 lanes of the group
  kmin = min(kmin & 0xffffu, kmin >> 16);
  kmax = max(kmax & 0xffffu, kmax >> 16);
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
  }
  if (!valid) return;
  const __half mn = __ushort_as_half(static_cast<unsigned short>(from_key2(kmin) & 0xffffu));
  const __half mx = __ushort_as_half(static_cast<unsigned short>(from_key2(kmax) & 0xffffu));
  const float fstep = q4_step_f32(mn, mx);
  const float fmn = __half2float(mn);
  // q4_code's decisions two values at a time: the same q, rint(q) as 2^23 + q
  // rounded to nearest (ties to even, 0 <= q < 17), the same test for q near
  // a half-integer (|q - rint(q)| <= 1/2, so | |d| - 1/2 | < 2^-16 is
  // |d| > 1/2 - 2^-16); each such value takes q4_code's exact decision.  A
  // zero step (every value equal to mn) gives q = 0 through a zero
  // reciprocal: codes 0.
  const float inv = fstep != 0.f ? __frcp_rn(fstep) : 0.f;
  const uint64_t MN = f2(fmn, fmn), INV = f2(inv, inv);
  const uint64_t K23 = f2(kRint23, kRint23);
  uint32_t packed[2] = {0u, 0u};
  uint32_t near = 0u;  // bit e: value e's quotient is near a half-integer
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float2 xf = __half22float2(*reinterpret_cast<const __half2*>(&w[u]));
    const uint64_t q = f2_mul(f2_sub(f2(xf.x, xf.y), MN), INV);
    const uint64_t tq = f2_add(q, K23);               // 2^23 + rint(q)
    const uint64_t dq = f2_sub(q, f2_sub(tq, K23));   // q - rint(q), exact
    near |= (fabsf(__uint_as_float(lo32(dq))) > 0.5f - 0x1p-16f ? 1u : 0u) << (2 * u);
    near |= (fabsf(__uint_as_float(hi32(dq))) > 0.5f - 0x1p-16f ? 2u : 0u) << (2 * u);
    const uint32_t c0 = min(lo32(tq) - kRint23Bits, 15u), c1 = min(hi32(tq) - kRint23Bits, 15u);
    packed[u >> 2] |= (c0 | (c1 << 4)) << (8 * (u & 3));
  }
  // those values (a few in ten thousand) take q4_code's exact decision
  while (near != 0u) {
    const int e = __ffs(near) - 1;
    near &= near - 1u;
    const uint32_t hv = (w[e >> 1] >> (16 * (e & 1))) & 0xffffu;
    const float xf = __half2float(__ushort_as_half(static_cast<unsigned short>(hv)));
    const int sh = 4 * (e & 7);
    packed[e >> 3] = (packed[e >> 3] & ~(0xfu << sh)) | (q4_code(xf, fmn, fstep, inv) << sh);
  }
  *reinterpret_cast<uint2*>(codes + grp * 32 + quarter * 8) = make_uint2(packed[0], packed[1]);
  st_global_u16_if(gmin + grp, __half_as_ushort(mn), quarter == 0);
  st_global_u16_if(gmax + grp, __half_as_ushort(mx), quarter == 0);
}

// 4 threads per group of 64 channels, 16 channels (32 bytes) per thread; two
// iterations' loads go out before either is used.  The loop advances whole
// blocks, so the 4 lanes of a group always shuffle together.
__global__ void __launch_bounds__(256) quant4_kernel(int64_t groups, const __half* x,
                                                     uint8_t* codes, __half* gmin, __half* gmax) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t total = groups * 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; t0 < total; t0 += 2 * stride) {
    const int64_t ta = t0 + threadIdx.x, tb = ta + stride;
    const bool va = (ta >> 2) < groups, vb = (tb >> 2) < groups;
    uint4 xa[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    uint4 xb[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    const uint4* pa = reinterpret_cast<const uint4*>(x + (ta >> 2) * 64 + (ta & 3) * 16);
    const uint4* pb = reinterpret_cast<const uint4*>(x + (tb >> 2) * 64 + (tb & 3) * 16);
    if (va) {
      xa[0] = __ldcs(pa);
      xa[1] = __ldcs(pa + 1);
    }
    if (vb) {
      xb[0] = __ldcs(pb);
      xb[1] = __ldcs(pb + 1);
    }
    quant4_part(xa, ta, va, codes, gmin, gmax);
    quant4_part(xb, tb, vb, codes, gmin, gmax);
  }
}

__global__ void __launch_bounds__(256) dequant4_kernel(int64_t groups, const uint8_t* codes,
                                                       const __half* gmin, const __half* gmax,
                                                       __half* x) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t total = groups * 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += stride) {
    const int64_t grp = t >> 3;
    const int sub = static_cast<int>(t & 7);
    const __half mn = gmin[grp], mx = gmax[grp];
    const uint32_t c4 = __ldcs(reinterpret_cast<const uint32_t*>(codes + grp * 32 + sub * 4));
    uint32_t w[4];
    q4_dequant8(c4, mn, mx, w);
    *reinterpret_cast<uint4*>(x + grp * 64 + sub * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------- 8-bit
// 8-bit page metadata: the bound of "TinyServe" (相关性函数实例化) needs only
// m_j <= k <= M_j channel by channel, so the metadata can be stored on a
// per-page grid dec(c) = fma(c, step, lo) with m rounded down and M rounded up
// (one byte each instead of two):
//   lo = min_i m_i, hi = max_i M_i (a zero as +0);
//   step = fp32(fp32(hi - lo) / 255), raised one ulp at a time until
//          dec(255) >= hi (0 when hi == lo);
//   code_min_i = the largest c with dec(c) <= m_i,
//   code_max_i = the smallest c with dec(c) >= M_i.
// The codes are defined by those extremes, so the first guess (a product
// with the step's reciprocal) only sets where the exact search starts.  Pages
// past a shorter sequence are not written.
__device__ __forceinline__ float value16f(uint32_t h, bool f16) {
  return f16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(h)))
             : __uint_as_float(h << 16);
}
template <bool F16>
__device__ __forceinline__ uint32_t min16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (F16) {
    const __half2 v = __hmin2(*reinterpret_cast<const __half2*>(&a),
                              *reinterpret_cast<const __half2*>(&b));
    r = *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __nv_bfloat162 v = __hmin2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                     *reinterpret_cast<const __nv_bfloat162*>(&b));
    r = *reinterpret_cast<const uint32_t*>(&v);
  }
  return r;
}
template <bool F16>
__device__ __forceinline__ uint32_t max16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (F16) {
    const __half2 v = __hmax2(*reinterpret_cast<const __half2*>(&a),
                              *reinterpret_cast<const __half2*>(&b));
    r = *reinterpret_cast<const uint32_t*>(&v);
  } else {
    const __nv_bfloat162 v = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                                     *reinterpret_cast<const __nv_bfloat162*>(&b));
    r = *reinterpret_cast<const uint32_t*>(&v);
  }
  return r;
}
__device__ __forceinline__ float dec8(int c, float step, float lo) {
  return __fmaf_rn(static_cast<float>(c), step, lo);
}
// 3 2^22: for 0 <= x < 2^22, x + K - 1 lies where floats are spaced by one,
// so its rounding down / up is K - 1 + floor(x) / ceil(x), held in the low
// bits (the float bits of K + j are those of K plus j)
constexpr float kMagic = 12582912.0f;

// the low bytes of four words, in order, as one word
__device__ __forceinline__ uint32_t low_bytes4(const uint32_t (&c)[4]) {
  return __byte_perm(__byte_perm(c[0], c[1], 0x0040u), __byte_perm(c[2], c[3], 0x0040u),
                     0x5410u);
}

// One page per 8 lanes (four pages a warp); lane u of a page owns channels
// D/8 u .. D/8 u + D/8 - 1 (two or four 16-byte loads of m and M).  The
// page's lo / hi by three shuffles within the 8 lanes; the step by the
// definition (an IEEE division, then one-ulp raises).  Each code without a
// search: with t = (m - lo) / step exactly and em = fl(fl(m - lo) fl(1/step)),
// |em - t| <= 256 * 3 * 2^-24; and a 16-bit page's range is at least one
// 16-bit ulp of its values (2^13 fp32 ulps for fp16, 2^16 for bf16), so the
// step is at least 16 fp32 ulps of any value in it and the largest c with
// dec(c) <= m is floor(t) or floor(t) + 1.  Hence code_min is within one of
// fm = floor(em), and
//   code_min = fm - 1 + [dec(fm) <= m] + [dec(fm + 1) <= m];
// likewise code_max = gM + 1 - [dec(gM) >= M] - [dec(gM - 1) >= M] with
// gM = ceil(eM).  floor / ceil as em + 3 2^22 - 1 rounded down / up, whose
// low byte plus the two comparison bits is the code.  This needs 1 / step
// finite and normal: steps below 2^-100 (bf16 pages below about 2^-92
// throughout) and infinite ones (a bf16 range above the largest float) take
// bounded walks from a clamped guess instead.
template <int D, bool F16>
__global__ void __launch_bounds__(kMetaThreads, D == 128 ? 5 : 0) meta8_kernel(const Meta8Args a) {
  griddep_launch_dependents();
  griddep_wait();
  constexpr int CPL = D / 8;  // channels per lane
  const int lane = threadIdx.x & 31, u = lane & 7;
  const unsigned gmask = 0xffu << (lane & 24);
  // one row of blocks per (batch, kv head) (grid y), 8 lanes a page along it
  const int j = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 3);
  for (int bh = blockIdx.y; bh < a.B * a.Hkv; bh += gridDim.y) {
    const int b = bh / a.Hkv;
    if (j >= a.P || static_cast<int64_t>(j) * a.S >= seq_len_of(a.lens, b, a.N))
      continue;  // the 8 lanes alike
    const int64_t pg = static_cast<int64_t>(bh) * a.P + j;
    const int64_t off = pg * D + CPL * u;
    uint32_t wm[CPL / 2], wM[CPL / 2];
#pragma unroll
    for (int v = 0; v < CPL / 8; ++v) {
      const uint4 x = __ldcs(reinterpret_cast<const uint4*>(a.meta_min + off) + v);
      const uint4 y = __ldcs(reinterpret_cast<const uint4*>(a.meta_max + off) + v);
      wm[4 * v] = x.x; wm[4 * v + 1] = x.y; wm[4 * v + 2] = x.z; wm[4 * v + 3] = x.w;
      wM[4 * v] = y.x; wM[4 * v + 1] = y.y; wM[4 * v + 2] = y.z; wM[4 * v + 3] = y.w;
    }
    float m[CPL], M[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      m[i] = value16f((wm[i / 2] >> (16 * (i & 1))) & 0xffffu, F16);
      M[i] = value16f((wM[i / 2] >> (16 * (i & 1))) & 0xffffu, F16);
    }
    uint32_t wlo = wm[0], whi = wM[0];  // two 16-bit lanes at a time
#pragma unroll
    for (int i = 1; i < CPL / 2; ++i) {
      wlo = min16x2<F16>(wlo, wm[i]);
      whi = max16x2<F16>(whi, wM[i]);
    }
    float lo = fminf(value16f(wlo & 0xffffu, F16), value16f(wlo >> 16, F16));
    float hi = fmaxf(value16f(whi & 0xffffu, F16), value16f(whi >> 16, F16));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(gmask, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(gmask, hi, o));
    }
    if (lo == 0.f) lo = 0.f;  // +0
    if (hi == 0.f) hi = 0.f;
    float step = 0.f;
    if (hi > lo) {
      step = __fdiv_rn(__fsub_rn(hi, lo), 255.f);
      while (dec8(255, step, lo) < hi) step = __int_as_float(__float_as_int(step) + 1);
    }
    uint32_t cmw[CPL / 4], cMw[CPL / 4];
#pragma unroll
    for (int i = 0; i < CPL / 4; ++i) cmw[i] = cMw[i] = 0u;
    if (step >= 0x1p-100f && step < INFINITY) {
      // the guess and the two comparisons that settle the code, two channels
      // per packed operation, each comparison the sign bit of a difference
      const float inv = __frcp_rn(step);
      const uint64_t LO = f2(lo, lo), INV = f2(inv, inv), STEP = f2(step, step);
      const uint64_t K1 = f2(kMagic - 1.f, kMagic - 1.f), K2 = f2(kMagic - 2.f, kMagic - 2.f);
      const uint64_t K0 = f2(kMagic, kMagic);
#pragma unroll
      for (int w = 0; w < CPL / 4; ++w) {
        uint32_t cm[4], cM[4];
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int i = 4 * w + e;
          const uint64_t mm = f2(m[i], m[i + 1]), MM = f2(M[i], M[i + 1]);
          // code_min = (floor - 1) + [dec(floor) <= m] + [dec(floor + 1) <= m]
          const uint64_t tm = f2_add_down(f2_mul(f2_sub(mm, LO), INV), K1);  // K - 1 + floor
          const uint64_t sm0 = f2_sub_down(f2_fma(f2_sub(tm, K1), STEP, LO), mm);
          const uint64_t sm1 = f2_sub_down(f2_fma(f2_sub(tm, K2), STEP, LO), mm);
          cm[e] = lo32(tm) + (lo32(sm0) >> 31) + (lo32(sm1) >> 31);
          cm[e + 1] = hi32(tm) + (hi32(sm0) >> 31) + (hi32(sm1) >> 31);
          // code_max = (ceil - 1) + [dec(ceil) < M] + [dec(ceil - 1) < M]
          const uint64_t tM = f2_add_up(f2_mul(f2_sub(MM, LO), INV), K1);  // K - 1 + ceil
          const uint64_t sM0 = f2_sub(f2_fma(f2_sub(tM, K1), STEP, LO), MM);
          const uint64_t sM1 = f2_sub(f2_fma(f2_sub(tM, K0), STEP, LO), MM);
          cM[e] = lo32(tM) + (lo32(sM0) >> 31) + (lo32(sM1) >> 31);
          cM[e + 1] = hi32(tM) + (hi32(sM0) >> 31) + (hi32(sM1) >> 31);
        }
        cmw[w] = low_bytes4(cm);
        cMw[w] = low_bytes4(cM);
      }
    } else if (step > 0.f) {
      // a step below 2^-100 (1 / step may overflow) or an infinite one: the
      // clamped guess and bounded walks to the defining extremes
      const float inv = __frcp_rn(step);
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const float em = __fmul_rn(__fsub_rn(m[i], lo), inv);
        const float eM = __fmul_rn(__fsub_rn(M[i], lo), inv);
        int cm = static_cast<int>(fminf(fmaxf(floorf(em), 0.f), 255.f));
        int cM = static_cast<int>(fminf(fmaxf(ceilf(eM), 0.f), 255.f));
        for (int t = 0; t < 256 && cm < 255 && dec8(cm + 1, step, lo) <= m[i]; ++t) ++cm;
        for (int t = 0; t < 256 && cm > 0 && dec8(cm, step, lo) > m[i]; ++t) --cm;
        for (int t = 0; t < 256 && cM > 0 && dec8(cM - 1, step, lo) >= M[i]; ++t) --cM;
        for (int t = 0; t < 256 && cM < 255 && dec8(cM, step, lo) < M[i]; ++t) ++cM;
        cmw[i / 4] |= static_cast<uint32_t>(cm) << (8 * (i & 3));
        cMw[i / 4] |= static_cast<uint32_t>(cM) << (8 * (i & 3));
      }
    }
    if constexpr (CPL == 16) {
      *reinterpret_cast<uint4*>(a.code_min + off) = make_uint4(cmw[0], cmw[1], cmw[2], cmw[3]);
      *reinterpret_cast<uint4*>(a.code_max + off) = make_uint4(cMw[0], cMw[1], cMw[2], cMw[3]);
    } else {
      *reinterpret_cast<uint2*>(a.code_min + off) = make_uint2(cmw[0], cmw[1]);
      *reinterpret_cast<uint2*>(a.code_max + off) = make_uint2(cMw[0], cMw[1]);
    }
    if (u == 0) {
      a.lo[pg] = lo;
      a.step[pg] = step;
    }
  }
}

int grid_for(int64_t threads, int block) {
  const int64_t blocks = ceil_div(threads, block);
  return static_cast<int>(blocks < 152 * 64 ? blocks : 152 * 64);
}

}  // namespace

cudaError_t launch_meta(bool q4, bool f16, const MetaArgs& a, cudaStream_t s) {
  (void)f16;  // min / max on order-preserving keys: identical code for bf16 and fp16
  const int64_t work =
      static_cast<int64_t>(a.B) * a.Hkv * (a.last_only ? 1 : a.P) * (a.d / 8);
  const dim3 grid(grid_for(work, kMetaThreads)), block(kMetaThreads);
  if (!q4 && !a.last_only && (a.S == 4 || a.S == 8)) {
    // a thread per 16-token cache page and 8 channels
    const int64_t sub_work =
        static_cast<int64_t>(a.B) * a.Hkv * ceil_div(a.N, kPage) * (a.d / 8);
    const dim3 sgrid(grid_for(sub_work, kMetaThreads));
    return a.S == 8 ? launch_pdl(meta_sub_kernel<2>, sgrid, block, 0, s, a)
                    : launch_pdl(meta_sub_kernel<4>, sgrid, block, 0, s, a);
  }
  if (!q4) return launch_pdl(meta_kernel, grid, block, 0, s, a);
  // one row of blocks per (batch, kv head): the row's pages, d/16 lanes each
  const int64_t row = static_cast<int64_t>(a.last_only ? 1 : a.P) * (a.d / 16);
  const int64_t rows = static_cast<int64_t>(a.B) * a.Hkv;
  const dim3 grid4(static_cast<unsigned>(ceil_div(row, kMetaThreads)),
                   static_cast<unsigned>(rows < 65535 ? rows : 65535));
  return a.d == 128 ? launch_pdl(meta_q4_kernel<128>, grid4, block, 0, s, a)
                    : launch_pdl(meta_q4_kernel<64>, grid4, block, 0, s, a);
}

cudaError_t launch_meta8(bool f16, const Meta8Args& a, cudaStream_t s) {
  // one row of blocks per (batch, kv head): its pages, 8 threads each
  const int64_t rows = static_cast<int64_t>(a.B) * a.Hkv;
  const dim3 grid(static_cast<unsigned>(ceil_div(static_cast<int64_t>(a.P) * 8, kMetaThreads)),
                  static_cast<unsigned>(rows < 65535 ? rows : 65535));
  const dim3 block(kMetaThreads);
  if (a.d == 128)
    return f16 ? launch_pdl(meta8_kernel<128, true>, grid, block, 0, s, a)
               : launch_pdl(meta8_kernel<128, false>, grid, block, 0, s, a);
  return f16 ? launch_pdl(meta8_kernel<64, true>, grid, block, 0, s, a)
             : launch_pdl(meta8_kernel<64, false>, grid, block, 0, s, a);
}

cudaError_t launch_quant4(int64_t rows, int d, const void* x, void* codes, void* gmin,
                          void* gmax, cudaStream_t s) {
  const int64_t groups = rows * (d / 64);
  return launch_pdl(quant4_kernel, dim3(grid_for(groups * 4, 256)), dim3(256), 0, s, groups,
                    static_cast<const __half*>(x), static_cast<uint8_t*>(codes),
                    static_cast<__half*>(gmin), static_cast<__half*>(gmax));
}

cudaError_t launch_dequant4(int64_t rows, int d, const void* codes, const void* gmin,
                            const void* gmax, void* x, cudaStream_t s) {
  const int64_t groups = rows * (d / 64);
  return launch_pdl(dequant4_kernel, dim3(grid_for(groups * 8, 256)), dim3(256), 0, s, groups,
                    static_cast<const uint8_t*>(codes), static_cast<const __half*>(gmin),
                    static_cast<const __half*>(gmax), static_cast<__half*>(x));
}

}  // namespace dkv

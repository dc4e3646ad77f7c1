// dkv_device.cuh -- device helpers for the sm_103a kernels of libdkv:
// mbarrier / TMA / ldmatrix / mma.sync wrappers in inline PTX, bounded waits
// that report through the status word, 16-bit float key transforms and the
// in-register 4-bit dequantisation.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace dkv {

// Device status codes (mirror dkv_status in include/dkv.h).
constexpr uint32_t kStatusTimeout = 8;
constexpr uint32_t kStatusCheck = 9;

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t code) {
  if (status != nullptr) atomicCAS(status, 0u, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- launch order
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialisation attribute may start while its predecessor in the stream
// finishes; griddep_wait() blocks until the predecessor has completed and its
// memory is visible, so it goes before the first read of anything a previous
// kernel may have written.  griddep_launch_dependents() lets the next kernel's
// CTAs be scheduled as this grid's last CTAs drain.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with `parity` of `bar` has completed.  Gives up (returns
// false) after `limit_ns` of wall time, or at once when limit_ns == 0 (the
// forced-timeout test hook), or when *abort becomes non-zero.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns,
                                                  const volatile int* abort_flag) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// A flag one kernel publishes for another running alongside it: a release
// store after the data it guards, an acquire load before reading that data.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Wait until *flag is non-zero.  Gives up (returns false) like
// mbar_wait_bounded: after `limit_ns`, at once when limit_ns == 0, or when
// *abort becomes non-zero.
__device__ __forceinline__ bool flag_wait_bounded(const uint32_t* flag, uint64_t limit_ns,
                                                  const volatile int* abort_flag) {
  if (limit_ns == 0) return false;
  if (ld_acquire_gpu(flag) != 0u) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(100);
    if (ld_acquire_gpu(flag) != 0u) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------- TMA
// Tiled tensor copy global -> shared, 5-D coordinates, completion counted in
// bytes on `bar`.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(c4)
      : "memory");
}

// Same, with an L2 eviction-priority hint (streamed-once data).
__device__ __forceinline__ void tma_load_5d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int c0, int c1, int c2, int c3,
                                                 int c4, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(c4), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Lines loaded under this policy are the last the L2 evicts (data the next
// call will read again).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Untiled bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- ldmatrix / mma
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D[16x8] += A[16x16] * B[16x8], fp32 accumulate.  F16 selects fp16 operands
// (otherwise bf16).
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Round two floats to a packed pair of 16-bit floats (round to nearest even);
// `lo` lands in the low half.
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Value of the low / high 16-bit float of a packed pair.
template <bool F16>
__device__ __forceinline__ float lo16(uint32_t w) {
  if constexpr (F16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
  } else {
    return __uint_as_float(w << 16);
  }
}
template <bool F16>
__device__ __forceinline__ float hi16(uint32_t w) {
  if constexpr (F16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
  } else {
    return __uint_as_float(w & 0xffff0000u);
  }
}

// Split p into hi + lo, each a 16-bit float pair, so that the tensor-core PV
// product keeps ~16 significant bits of the softmax weights.
template <bool F16>
__device__ __forceinline__ void split_pair(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  hi = pack2<F16>(p0, p1);
  lo = pack2<F16>(p0 - lo16<F16>(hi), p1 - hi16<F16>(hi));
}

// ---------------------------------------------------------------- 16-bit keys
// Order-preserving map of two packed 16-bit floats to unsigned 16-bit keys
// (numeric order, -0 below +0), and its inverse.
__device__ __forceinline__ uint32_t to_key2(uint32_t x) {
  const uint32_t s = (x >> 15) & 0x00010001u;
  return x ^ ((s * 0xffffu) | 0x80008000u);
}
__device__ __forceinline__ uint32_t from_key2(uint32_t k) {
  const uint32_t t = (~k >> 15) & 0x00010001u;
  return k ^ ((t * 0x7fffu) | 0x80008000u);
}

// ---------------------------------------------------------------- 4-bit format
// A group's 16 levels are mn + c * s, c = 0 .. 15, with the step s rounded
// down from (mx - mn) / 15 so that no level passes the group max, and the
// dequantised value is the level rounded once to fp16:
//   range = fp32_down(mx - mn)
//   normal groups (range >= 451 * 2^-24): s = fp16_down(fp32_down(range / 15)),
//     and x = fp16(c * s + mn) is one fused fp16 multiply-add;
//   tiny groups: s = floor(range / (15 g)) * g, g = 2^(floor(log2 max(|mn|,
//     |mx|)) - 22), an fp32 value; every value of such a group lies below 2^-5
//     and mn + c * s is a multiple of g, so it is exact in fp32 and
//     x = fp16(fp32 fma(c, s, mn)).
// (fp32_down / fp16_down: the largest binary32 / binary16 at or below.)  With
// codes chosen as the nearest level, |x - x_in| <= (mx - mn)/30 plus half an
// fp16 ulp of x for every finite group.
constexpr float kQ4TinyRange = 451.0f * 0x1p-24f;

__device__ __forceinline__ float q4_range(__half mn, __half mx) {
  return __fsub_rd(__half2float(mx), __half2float(mn));
}

// fp16_down(fp32_down(range / 15)) for a normal group's range.  fl(range / 15)
// by the FMA method for division by a constant (q = fl(range * fl(1/15)),
// corrected once with the exact remainder), then one ulp down when the exact
// remainder range - 15 q is negative; both steps are checked for every
// binary32 below 2^18 on the host.
__device__ __forceinline__ __half q4_step16(float range) {
  constexpr float kInv15 = 1.0f / 15.0f;
  const float q0 = __fmul_rn(range, kInv15);
  const float r0 = __fmaf_rn(-q0, 15.0f, range);
  const float q = __fmaf_rn(r0, kInv15, q0);  // the IEEE quotient
  const float r = __fmaf_rn(-q, 15.0f, range);  // exact
  const float qd = r < 0.f ? __int_as_float(__float_as_int(q) - 1) : q;
  return __float2half_rd(qd);
}

// The fp32 step of a tiny group (range < kQ4TinyRange).
__device__ __forceinline__ float q4_step32(float range, __half mn, __half mx) {
  if (range == 0.f) return 0.f;
  const float a = fmaxf(fabsf(__half2float(mn)), fabsf(__half2float(mx)));
  const int ea = (__float_as_int(a) >> 23) - 127;  // floor(log2 a), a a normal binary32
  const float up = __int_as_float((127 + 22 - ea) << 23);  // 1 / g
  const float g = __int_as_float((127 - 22 + ea) << 23);
  const uint32_t r = static_cast<uint32_t>(__fmul_rn(range, up));  // exact, below 2^24
  return __fmul_rn(static_cast<float>(r / 15u), g);  // exact
}

// The step of any group as an fp32 value (a normal group's fp16 step widened).
__device__ __forceinline__ float q4_step_f32(__half mn, __half mx) {
  const float range = q4_range(mn, mx);
  return range >= kQ4TinyRange ? __half2float(q4_step16(range)) : q4_step32(range, mn, mx);
}

// The code of x: the c in [0, 15] nearest to (x - mn) / s, ties to the even
// c.  q = fl(fl(x - mn) * fl(1/s)) is within 2^-18 of (x - mn) / s while it is
// below 16 (three roundings of 2^-24 relative); so rint(q) is the code unless
// q lies within 2^-16 of a half-integer, and only then is the choice made
// exactly: 2 (x - mn) against (2 floor(q) + 1) s in double (both exact).
__device__ __forceinline__ uint32_t q4_code(float x, float mn, float s, float inv) {
  const float q = __fmul_rn(__fsub_rn(x, mn), inv);
  float c = rintf(q);
  if (fabsf(fabsf(q - c) - 0.5f) < 0x1p-16f) {
    const double lo = floor(static_cast<double>(q));
    const double r = 2.0 * (static_cast<double>(x) - static_cast<double>(mn)) -
                     (2.0 * lo + 1.0) * static_cast<double>(s);
    c = static_cast<float>(r > 0.0 || (r == 0.0 && fmod(lo, 2.0) != 0.0) ? lo + 1.0 : lo);
  }
  return static_cast<uint32_t>(fminf(15.f, fmaxf(0.f, c)));
}

// One code of a tiny group: fp16(fp32 fma(c, s, mn)), exact before the rounding.
__device__ __forceinline__ __half q4_level32(uint32_t code, float s, float mn) {
  return __float2half_rn(__fmaf_rn(static_cast<float>(code), s, mn));
}

// Dequantise the 8 codes of one 32-bit word (byte i: channel 2i low nibble,
// 2i+1 high nibble) of the group (mn, mx).  Output: 4 packed half pairs,
// channels in order.  Normal groups: a nibble masked into the mantissa of
// 1024 is 1024 + code exactly; subtracting 1024 leaves the code, then one
// HFMA2 per pair.
__device__ __forceinline__ void q4_dequant8(uint32_t c4, __half mn, __half mx, uint32_t (&out)[4]) {
  const float range = q4_range(mn, mx);
  if (range >= kQ4TinyRange) {
    const __half2 step2 = __half2half2(q4_step16(range)), mn2 = __half2half2(mn);
    const __half2 k1024 = __half2half2(__ushort_as_half(0x6400));  // 1024.0
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t byte = (c4 >> (8 * i)) & 0xffu;
      const uint32_t bits = (byte & 0x0fu) | ((byte & 0xf0u) << 12) | 0x64006400u;
      const __half2 code = __hsub2(*reinterpret_cast<const __half2*>(&bits), k1024);
      const __half2 x = __hfma2(code, step2, mn2);
      out[i] = *reinterpret_cast<const uint32_t*>(&x);
    }
  } else {
    const float s = q4_step32(range, mn, mx), m = __half2float(mn);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t byte = (c4 >> (8 * i)) & 0xffu;
      const __half lo = q4_level32(byte & 0x0fu, s, m), hi = q4_level32(byte >> 4, s, m);
      out[i] = static_cast<uint32_t>(__half_as_ushort(lo)) |
               (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
    }
  }
}

// ---------------------------------------------------------------- selection
// Keep the halves of two packed 16-bit floats that belong to q+ (negative_part
// false: +0, -0 and positive values) or to q- (negative values); zero the rest.
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

// Order-preserving key of an fp32 score (-0 taken as +0).
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The score a key stands for (inverse of score_key).
__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

}  // namespace dkv

// attn.cu -- decode attention over pages of a KV cache (exact and page-sparse),
// with the split-K merge done inside the same kernel.
//
// What it computes (per query head h of batch b, kv head h / G):
//   out = sum_t softmax_t(scale * q . k_t) v_t
// over all N tokens ("论文阅读：HeadInfer", 核心 idea; "TinyServe: Query-Aware
// Cache Selection for Efficient LLM Serving", 标准Transformer解码层的注意力计算)
// or over the tokens of the pages selected for h (TinyServe, 问题公式化定义,
// Algorithm 1 steps 3-4: gather the selected pages, then softmax-weighted sum).
//
// Structure (one CTA = one chunk of pages of one (batch, kv head)):
//   * warp 4 (producer): one lane streams whole pages of K and V into a ring of
//     shared-memory stages with TMA tensor copies (cp.async.bulk.tensor, 128B
//     swizzle), each stage guarded by a full / empty mbarrier pair.  In the
//     sparse path the warp first turns the per-head selection bitmaps into the
//     CTA's page list (union over the G query heads of the group).
//   * warps 0-3 (consumers): page i goes to warp i % 4.  A warp computes the
//     16-token page for all G <= 8 query heads of the group at once on tensor
//     cores: S[8 heads x 16 tokens] = Q K^T with mma.sync m16n8k16 (heads on the
//     M side, rows 8-15 unused), an online softmax in fp32 (log2 domain), then
//     O += P V with P split into a high and a low 16-bit half (rows 0-7 / 8-15
//     of the A operand) so the weights keep ~16 significant bits.
//   * the four warps' (max, sum, o) states are merged in shared memory into the
//     chunk's partial.  The last CTA to finish among a group of kGroup chunks
//     (an atomic ticket) merges the group; the last group merges the groups
//     and writes out.  Merges run in ascending order, so results are
//     deterministic, and chunking depends only on (P, d), so one kv head at a
//     time gives bitwise the all-heads result.  Tickets return to zero at the
//     end of every call.
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the status word, stops issuing, drains the copies it issued and still takes
// its tickets (so the counters stay consistent), leaving garbage output.

#include <math.h>

#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {
namespace {

constexpr uint64_t kDrainLimitNs = 200000000ull;  // 200 ms for the whole drain

template <int D>
struct AttnCfg {
  static constexpr int kPageBytes = kPage * D * 2;  // one tensor's page
  static constexpr int kStageBytes = 2 * kPageBytes;
  static constexpr int kStages = attn_stages(D);
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kMiscOffset = kBarOffset + 2 * kStages * 8;
  // misc: abort, n_pages, last-flag | list[256] | mask[256] | merge scratch
  static constexpr int kListOffset = kMiscOffset + 16;
  static constexpr int kMaskOffset = kListOffset + 4 * kMaxSelectList;
  static constexpr int kScratchOffset = kMaskOffset + 4 * kMaxSelectList;
  static constexpr int kScratchBytes = 4 * (2 * 8 * kGroup + 2 * 8);
  static constexpr int kSmemBytes = 1024 + kScratchOffset + kScratchBytes;
  static_assert(kPageBytes % 1024 == 0, "stages must stay 1024-byte aligned");
  static_assert(kConsumerWarps * 8 * (D + 2) * 4 <= kBarOffset, "merge area fits");
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

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
}

// Sparse path: the pages of the union of the group's selections whose rank (in
// ascending page order) falls in [chunk * ppc, (chunk + 1) * ppc), with a
// bit per query head that selected each page.  Run by one full warp.
__device__ void build_sparse_list(const AttnArgs& a, int b, int kvh, int chunk, int* s_list,
                                  uint32_t* s_mask, int* s_npages, int lane) {
  const int lo = chunk * a.pages_per_chunk, hi = lo + a.pages_per_chunk;
  const uint32_t* bm = a.bitmaps + (static_cast<int64_t>(b) * a.Hq + kvh * a.G) * a.W32;
  int count = 0;
  for (int w0 = 0; w0 < a.W32 && count < hi; w0 += 32) {
    const int wi = w0 + lane;
    uint32_t words[8];
    uint32_t uni = 0;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      words[g] = (g < a.G && wi < a.W32) ? bm[static_cast<int64_t>(g) * a.W32 + wi] : 0u;
      uni |= words[g];
    }
    const int c = __popc(uni);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    int r = count + incl - c;
    if (r < hi && r + c > lo) {
      uint32_t bits = uni;
      while (bits) {
        const int j = __ffs(bits) - 1;
        bits &= bits - 1;
        if (r >= lo && r < hi) {
          uint32_t m = 0;
#pragma unroll
          for (int g = 0; g < 8; ++g) m |= ((words[g] >> j) & 1u) << g;
          s_list[r - lo] = wi * 32 + j;
          s_mask[r - lo] = m;
        }
        ++r;
      }
    }
    count += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) *s_npages = max(0, min(count, hi) - lo);
}

__device__ __forceinline__ void store_out(const AttnArgs& a, int b, int h, int c, float v) {
  const int64_t off = b * a.o_sb + h * a.o_sh + c;
  if (a.out_dtype == 2) {
    static_cast<float*>(a.out)[off] = v;
  } else if (a.out_dtype == 1) {
    static_cast<__half*>(a.out)[off] = __float2half_rn(v);
  } else {
    static_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(v);
  }
}

// Merge `count` (<= kGroup) consecutive partials [first, first + count) of the
// G rows (b, kvh*G + h): weights w_i = 2^(m_i - max m), in ascending order.
// Writes one merged partial (item `out_item` of rows with `n_out` items) or,
// when final, out = sum w_i o_i / sum w_i l_i.  All threads of the CTA call it.
template <int D>
__device__ void merge_partials(const AttnArgs& a, int b, int kvh, const float* ml_in,
                               const float* o_in, int n_in, int first, int count, bool final,
                               float* ml_out, float* o_out, int n_out, int out_item,
                               float* scratch) {
  float* s_w = scratch;                 // [8][kGroup] m_i, then weights
  float* s_l = scratch + 8 * kGroup;    // [8][kGroup]
  float* s_M = scratch + 16 * kGroup;   // [8]
  float* s_L = s_M + 8;                 // [8]
  const int64_t row0 = static_cast<int64_t>(b) * a.Hq + kvh * a.G;
  for (int t = threadIdx.x; t < a.G * count; t += blockDim.x) {
    const int h = t / count, i = t % count;
    const int64_t item = (row0 + h) * n_in + first + i;
    s_w[h * kGroup + i] = __ldcg(ml_in + 2 * item);
    s_l[h * kGroup + i] = __ldcg(ml_in + 2 * item + 1);
  }
  __syncthreads();
  if (threadIdx.x < a.G) {
    const int h = threadIdx.x;
    float M = -INFINITY;
    for (int i = 0; i < count; ++i) M = fmaxf(M, s_w[h * kGroup + i]);
    float L = 0.f;
    for (int i = 0; i < count; ++i) {
      const float m = s_w[h * kGroup + i];
      const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
      L += w * s_l[h * kGroup + i];
      s_w[h * kGroup + i] = w;
    }
    s_M[h] = M;
    s_L[h] = L;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < a.G * D; idx += blockDim.x) {
    const int h = idx / D, c = idx % D;
    const float* src = o_in + ((row0 + h) * n_in + first) * D + c;
    float x[kGroup];
#pragma unroll
    for (int i = 0; i < kGroup; ++i) x[i] = (i < count) ? __ldcg(src + i * D) : 0.f;
    float O = 0.f;
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      const float w = (i < count) ? s_w[h * kGroup + i] : 0.f;
      O += (w != 0.f) ? w * x[i] : 0.f;  // empty partials hold no o values
    }
    if (final) {
      store_out(a, b, kvh * a.G + h, c, O / s_L[h]);
    } else {
      const int64_t item = (row0 + h) * n_out + out_item;
      o_out[item * D + c] = O;
      if (c == 0) {
        ml_out[2 * item] = s_M[h];
        ml_out[2 * item + 1] = s_L[h];
      }
    }
  }
}

template <int D, bool F16, bool SPARSE>
__global__ void __launch_bounds__(kAttnThreads)
    attn_pages_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv) {
  using C = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t full0 = sbase + C::kBarOffset;
  const uint32_t empty0 = full0 + 8 * C::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOffset);
  int* s_npages = reinterpret_cast<int*>(smem + C::kMiscOffset + 4);
  volatile int* s_last = reinterpret_cast<volatile int*>(smem + C::kMiscOffset + 8);
  int* s_list = reinterpret_cast<int*>(smem + C::kListOffset);
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(smem + C::kMaskOffset);
  float* scratch = reinterpret_cast<float*>(smem + C::kScratchOffset);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tensormap(&mk);
    prefetch_tensormap(&mv);
  }
  griddep_launch_dependents();
  griddep_wait();  // q, K, V, bitmaps and the workspace may come from earlier kernels
  int first_page = 0, n_pages = 0;
  if constexpr (SPARSE) {
    if (warp == kConsumerWarps) build_sparse_list(a, b, kvh, chunk, s_list, s_mask, s_npages, lane);
  } else {
    first_page = chunk * a.pages_per_chunk;
    n_pages = max(0, min(a.P - first_page, a.pages_per_chunk));
  }
  __syncthreads();
  if constexpr (SPARSE) n_pages = *s_npages;

  const int64_t row0 = static_cast<int64_t>(b) * a.Hq + kvh * a.G;
  if (n_pages <= 0) {
    // Nothing to attend in this chunk: an empty partial (no o values).
    if (threadIdx.x < a.G) {
      const int64_t item = (row0 + threadIdx.x) * a.n_chunks + chunk;
      a.part_ml[2 * item] = -INFINITY;
      a.part_ml[2 * item + 1] = 0.f;
    }
  } else if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (int i = 0; i < n_pages; ++i) {
        const int s = i % C::kStages, k = i / C::kStages;
        if (i >= C::kStages &&
            !mbar_wait_bounded(empty0 + 8 * s, (k - 1) & 1, a.wait_limit_ns, abort_flag)) {
          if (!*abort_flag) {
            set_status(a.status, kStatusTimeout);
            *abort_flag = 1;
          }
          break;
        }
        if (*abort_flag) break;
        const int page = SPARSE ? s_list[i] : first_page + i;
        const uint32_t dst = sbase + s * C::kStageBytes;
        mbar_arrive_expect_tx(full0 + 8 * s, C::kStageBytes);
        tma_load_5d_hint(dst, &mk, full0 + 8 * s, 0, page * kPage, 0, kvh, b, pol);
        tma_load_5d_hint(dst + C::kPageBytes, &mv, full0 + 8 * s, 0, page * kPage, 0, kvh, b,
                         pol);
        ++issued;
      }
      if (*abort_flag) {  // let every copy this CTA issued land before it exits
        const uint64_t deadline = globaltimer_ns() + kDrainLimitNs;
        for (int i = max(0, issued - C::kStages); i < issued; ++i) {
          const uint64_t now = globaltimer_ns();
          if (now >= deadline) break;
          mbar_wait_bounded(full0 + 8 * (i % C::kStages), (i / C::kStages) & 1, deadline - now,
                            nullptr);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t4 = lane & 3;
    const bool head_ok = g < a.G;
    uint32_t qa[D / 16][2];
    {
      const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + b * a.q_sb +
                             static_cast<int64_t>(kvh * a.G + (head_ok ? g : 0)) * a.q_sh;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qa[ks][0] = head_ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t4) : 0u;
        qa[ks][1] =
            head_ok ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t4 + 8) : 0u;
      }
    }
    float m_run = -INFINITY, l_run = 0.f;
    float acc[D / 8][4];
#pragma unroll
    for (int cn = 0; cn < D / 8; ++cn) acc[cn][0] = acc[cn][1] = acc[cn][2] = acc[cn][3] = 0.f;

    bool aborted = false;
    const int mtx = lane >> 3, mrow = lane & 7;
    for (int i = warp; i < n_pages; i += kConsumerWarps) {
      const int s = i % C::kStages, k = i / C::kStages;
      const bool ok = mbar_wait_bounded(full0 + 8 * s, k & 1, a.wait_limit_ns, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          set_status(a.status, kStatusTimeout);
          *abort_flag = 1;
        }
        aborted = true;
        break;
      }
      const uint32_t kb = sbase + s * C::kStageBytes, vb = kb + C::kPageBytes;
      const int page = SPARSE ? s_list[i] : first_page + i;
      const uint32_t hmask = SPARSE ? s_mask[i] : 0xffu;

      // S = Q K^T for the page: sc[nt][e] = score of head g, token 8 nt + 2 t4 + e.
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(tile_addr(kb, 8 * (mtx >> 1) + mrow, 16 * ks + 8 * (mtx & 1)), r0, r1, r2, r3);
        mma16816<F16>(sc[0], qa[ks][0], 0u, qa[ks][1], 0u, r0, r1);
        mma16816<F16>(sc[1], qa[ks][0], 0u, qa[ks][1], 0u, r2, r3);
      }

      // Online softmax (log2 domain) for head g over its 4 tokens of this page.
      const bool head_on = head_ok && ((hmask >> g) & 1u);
      float sv[4];
      float pmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int tok = page * kPage + 8 * (j >> 1) + 2 * t4 + (j & 1);
        sv[j] = (head_on && tok < a.N) ? sc[j >> 1][j & 1] * a.scale_log2 : -INFINITY;
        pmax = fmaxf(pmax, sv[j]);
      }
      pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, 1));
      pmax = fmaxf(pmax, __shfl_xor_sync(0xffffffffu, pmax, 2));
      const float m_new = fmaxf(m_run, pmax);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(m_run - m_use);
      float p[4];
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        p[j] = exp2f(sv[j] - m_use);
        psum += p[j];
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

    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);

    // Merge the consumer warps' states into the chunk's partial (the stage ring
    // is free once every warp is past its loop: all issued copies were consumed).
    if (!consumers_any(aborted)) {
      float* mrg = reinterpret_cast<float*>(smem);
      {
        float* r = mrg + (warp * 8 + g) * (D + 2);
        if (t4 == 0) {
          r[D] = m_run;
          r[D + 1] = l_run;
        }
#pragma unroll
        for (int cn = 0; cn < D / 8; ++cn) {
          r[8 * cn + 2 * t4] = acc[cn][0] + acc[cn][2];
          r[8 * cn + 2 * t4 + 1] = acc[cn][1] + acc[cn][3];
        }
      }
      consumers_sync();
      for (int idx = threadIdx.x; idx < a.G * D; idx += kConsumerWarps * 32) {
        const int h = idx / D, c = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mrg[(w * 8 + h) * (D + 2) + D]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float* r = mrg + (w * 8 + h) * (D + 2);
            if (r[D] == -INFINITY) continue;
            const float f = exp2f(r[D] - M);
            L += f * r[D + 1];
            O += f * r[c];
          }
        }
        const int64_t item = (row0 + h) * a.n_chunks + chunk;
        a.part_o[item * D + c] = O;
        if (c == 0) {
          a.part_ml[2 * item] = M;
          a.part_ml[2 * item + 1] = L;
        }
      }
    }
  }

  // ---------------------------------------------------------- split-K merge
  __syncthreads();
  const int64_t unit = static_cast<int64_t>(b) * a.Hkv + kvh;
  const int grp = chunk / kGroup;
  const int gsize = min(kGroup, a.n_chunks - grp * kGroup);
  if (threadIdx.x == 0) {
    __threadfence();
    uint32_t* t = a.tickets + unit * a.n_groups + grp;
    const bool last = atomicAdd(t, 1u) == static_cast<uint32_t>(gsize - 1);
    if (last) atomicExch(t, 0u);  // every CTA of the group has arrived: reset
    *s_last = last;
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  const bool skip = *abort_flag != 0;  // this CTA's copies may still be landing
  if (!skip)
    merge_partials<D>(a, b, kvh, a.part_ml, a.part_o, a.n_chunks, grp * kGroup, gsize,
                      a.n_groups == 1, a.part2_ml, a.part2_o, a.n_groups, grp, scratch);
  if (a.n_groups == 1) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    uint32_t* t = a.tickets + static_cast<int64_t>(a.B) * a.Hkv * a.n_groups + unit;
    const bool last = atomicAdd(t, 1u) == static_cast<uint32_t>(a.n_groups - 1);
    if (last) atomicExch(t, 0u);
    *s_last = last;
  }
  __syncthreads();
  if (!*s_last) return;
  __threadfence();
  if (!skip)
    merge_partials<D>(a, b, kvh, a.part2_ml, a.part2_o, a.n_groups, 0, a.n_groups, true,
                      nullptr, nullptr, 0, 0, scratch);
}

template <int D, bool F16, bool SPARSE>
cudaError_t launch_attn_t(const AttnArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                          dim3 grid, cudaStream_t s) {
  using C = AttnCfg<D>;
  auto kern = attn_pages_kernel<D, F16, SPARSE>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(kAttnThreads), C::kSmemBytes, s, a, mk, mv);
}

}  // namespace

cudaError_t launch_attn(int d, bool f16, bool sparse, const AttnArgs& a, const CUtensorMap& mk,
                        const CUtensorMap& mv, dim3 grid, cudaStream_t s) {
  if (d == 128) {
    if (f16) return sparse ? launch_attn_t<128, true, true>(a, mk, mv, grid, s)
                           : launch_attn_t<128, true, false>(a, mk, mv, grid, s);
    return sparse ? launch_attn_t<128, false, true>(a, mk, mv, grid, s)
                  : launch_attn_t<128, false, false>(a, mk, mv, grid, s);
  }
  if (f16) return sparse ? launch_attn_t<64, true, true>(a, mk, mv, grid, s)
                         : launch_attn_t<64, true, false>(a, mk, mv, grid, s);
  return sparse ? launch_attn_t<64, false, true>(a, mk, mv, grid, s)
                : launch_attn_t<64, false, false>(a, mk, mv, grid, s);
}

}  // namespace dkv

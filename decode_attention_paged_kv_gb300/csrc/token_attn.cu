// token_attn.cu -- attention over each query head's top-K tokens.
//
// Token-level sparse attention ("FlexGen: High-Throughput Generative Inference
// of Large Language Models with a Single GPU" 解读, its sparse attention: each
// query keeps the top 10% of the K cache's indices and loads only that subset
// of V).  The exact scores s_t = q . k_t of all tokens come from the score pass
// (the bound-score kernel with single-token pages, where m = M = k makes the
// bound the dot product itself) and the top-K tokens from the radix top-K.
// This kernel does the rest for one (b, q-head) row per CTA:
//   M = max of the selected scores; p_t = 2^((s_t - M) * scale * log2 e);
//   out = (sum p_t v_t) / (sum p_t) over the selected tokens.
// Warp w takes the w-th contiguous slice of the ascending token list, so its
// V rows come in ascending order; lane l owns channels [c l, c (l + 1)),
// c = d / 32, so a warp reads whole 2d-byte V rows.  Sixteen tokens' loads are
// in flight per warp.  The warps' sums are combined in warp order:
// deterministic.  Bytes per row: kk V rows (d * 2 each) + kk indices and
// scores + out.

#include <math.h>

#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {
namespace {

constexpr int kTokWarps = 8;
constexpr int kTokUnroll = 16;

template <int D, bool F16>
__device__ __forceinline__ void load_v(const uint16_t* v, float (&x)[D / 32]) {
  if constexpr (D == 128) {
    const uint2 w = __ldcs(reinterpret_cast<const uint2*>(v));
    x[0] = lo16<F16>(w.x);
    x[1] = hi16<F16>(w.x);
    x[2] = lo16<F16>(w.y);
    x[3] = hi16<F16>(w.y);
  } else {
    const uint32_t w = __ldcs(reinterpret_cast<const uint32_t*>(v));
    x[0] = lo16<F16>(w);
    x[1] = hi16<F16>(w);
  }
}

template <int D, bool F16>
__global__ void __launch_bounds__(kTokWarps * 32) token_attn_kernel(const TokenAttnArgs a) {
  __shared__ float s_red[kTokWarps];
  __shared__ float s_o[kTokWarps][D];
  __shared__ float s_l[kTokWarps];
  griddep_launch_dependents();
  griddep_wait();  // scores and the selection come from the previous kernels
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x;
  const int b = row / a.Hq, h = row % a.Hq, kvh = h / a.G;
  const int32_t* sel = a.selected + static_cast<int64_t>(row) * a.kk;
  const float* sc = a.scores + static_cast<int64_t>(row) * a.N;

  // M: the largest selected score
  float m = -INFINITY;
  for (int i = threadIdx.x; i < a.kk; i += kTokWarps * 32) m = fmaxf(m, __ldcg(sc + __ldcg(sel + i)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) s_red[warp] = m;
  __syncthreads();
  float M = s_red[0];
#pragma unroll
  for (int w = 1; w < kTokWarps; ++w) M = fmaxf(M, s_red[w]);

  // this warp's contiguous slice of the ascending token list
  const int per = static_cast<int>(ceil_div(a.kk, kTokWarps));
  const int i0 = warp * per, i1 = min(a.kk, i0 + per);
  const uint16_t* vbase = static_cast<const uint16_t*>(a.v) + b * a.v_sb + kvh * a.v_sh +
                          (D / 32) * lane;
  float acc[D / 32];
#pragma unroll
  for (int c = 0; c < D / 32; ++c) acc[c] = 0.f;
  float l = 0.f;
  for (int i = i0; i < i1; i += kTokUnroll) {
    int t[kTokUnroll];
    float s[kTokUnroll];
#pragma unroll
    for (int u = 0; u < kTokUnroll; ++u) t[u] = i + u < i1 ? __ldcg(sel + i + u) : -1;
#pragma unroll
    for (int u = 0; u < kTokUnroll; ++u) s[u] = t[u] >= 0 ? __ldcg(sc + t[u]) : -INFINITY;
    float x[kTokUnroll][D / 32];
#pragma unroll
    for (int u = 0; u < kTokUnroll; ++u) {
      if (t[u] >= 0) {
        load_v<D, F16>(vbase + static_cast<int64_t>(t[u]) * a.v_st, x[u]);
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) x[u][c] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < kTokUnroll; ++u) {
      const float p = t[u] >= 0 ? exp2f((s[u] - M) * a.scale_log2) : 0.f;
      l += p;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) acc[c] = fmaf(p, x[u][c], acc[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < D / 32; ++c) s_o[warp][(D / 32) * lane + c] = acc[c];
  if (lane == 0) s_l[warp] = l;
  __syncthreads();
  if (threadIdx.x < D) {
    float o = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < kTokWarps; ++w) {
      o += s_o[w][threadIdx.x];
      L += s_l[w];
    }
    const float v = o / L;
    const int64_t off = b * a.o_sb + h * a.o_sh + threadIdx.x;
    if (a.out_dtype == 2) {
      static_cast<float*>(a.out)[off] = v;
    } else if (a.out_dtype == 1) {
      static_cast<__half*>(a.out)[off] = __float2half_rn(v);
    } else {
      static_cast<__nv_bfloat16*>(a.out)[off] = __float2bfloat16_rn(v);
    }
  }
}

}  // namespace

cudaError_t launch_token_attn(int d, bool f16, const TokenAttnArgs& a, int rows, cudaStream_t s) {
  const dim3 grid(rows), block(kTokWarps * 32);
  if (d == 128)
    return f16 ? launch_pdl(token_attn_kernel<128, true>, grid, block, 0, s, a)
               : launch_pdl(token_attn_kernel<128, false>, grid, block, 0, s, a);
  return f16 ? launch_pdl(token_attn_kernel<64, true>, grid, block, 0, s, a)
             : launch_pdl(token_attn_kernel<64, false>, grid, block, 0, s, a);
}

}  // namespace dkv

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
// The selected list is taken kTokChunk tokens at a time: its indices and
// scores are staged in shared memory, the running maximum M updated (the sums
// so far rescaled by 2^((M_old - M) * scale * log2 e)), and the scores turned
// into weights p_t there.  Warp w takes the w-th contiguous slice of the chunk,
// so its V rows come in ascending order; lane l owns channels [c l, c (l + 1)),
// c = d / 32, so a warp reads whole 2d-byte V rows, kTokBatch of them in
// flight while it accumulates the previous kTokBatch.  The warps' sums are
// combined in warp order: deterministic.  Bytes per row: kk V rows (d * 2
// each) + kk indices and scores + out.

#include <math.h>

#include <type_traits>

#include "dkv_device.cuh"
#include "dkv_kernels.h"

namespace dkv {
namespace {

constexpr int kTokWarps = 8;
constexpr int kTokBatch = 8;     // V rows a warp loads at a time
constexpr int kTokChunk = 4096;  // selected tokens staged at a time (32 KiB)

template <int D>
struct VRaw {  // one lane's share of a V row: D / 32 16-bit values
  using T = typename std::conditional<D == 128, uint2, uint32_t>::type;
};

template <int D>
__device__ __forceinline__ typename VRaw<D>::T load_v(const uint16_t* v) {
  return __ldcs(reinterpret_cast<const typename VRaw<D>::T*>(v));
}

template <int D, bool F16>
__device__ __forceinline__ void acc_v(float p, const typename VRaw<D>::T& w, float (&acc)[D / 32]) {
  if constexpr (D == 128) {
    acc[0] = fmaf(p, lo16<F16>(w.x), acc[0]);
    acc[1] = fmaf(p, hi16<F16>(w.x), acc[1]);
    acc[2] = fmaf(p, lo16<F16>(w.y), acc[2]);
    acc[3] = fmaf(p, hi16<F16>(w.y), acc[3]);
  } else {
    acc[0] = fmaf(p, lo16<F16>(w), acc[0]);
    acc[1] = fmaf(p, hi16<F16>(w), acc[1]);
  }
}

template <int D, bool F16>
__global__ void __launch_bounds__(kTokWarps * 32, 4) token_attn_kernel(const TokenAttnArgs a) {
  using Raw = typename VRaw<D>::T;
  __shared__ int s_idx[kTokChunk];
  __shared__ float s_p[kTokChunk];
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
  const uint16_t* vbase = static_cast<const uint16_t*>(a.v) + b * a.v_sb + kvh * a.v_sh +
                          (D / 32) * lane;
  float acc[D / 32];
#pragma unroll
  for (int c = 0; c < D / 32; ++c) acc[c] = 0.f;
  float l = 0.f, M = -INFINITY;
  for (int c0 = 0; c0 < a.kk; c0 += kTokChunk) {
    const int n = min(kTokChunk, a.kk - c0);
    // stage the chunk's indices and scores; its maximum
    float m = -INFINITY;
    for (int i = threadIdx.x; i < n; i += kTokWarps * 32) {
      const int t = __ldcg(sel + c0 + i);
      const float x = __ldcg(sc + t);
      s_idx[i] = t;
      s_p[i] = x;
      m = fmaxf(m, x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float Mc = s_red[0];
#pragma unroll
    for (int w = 1; w < kTokWarps; ++w) Mc = fmaxf(Mc, s_red[w]);
    if (Mc > M) {  // a new maximum: rescale what this warp has summed
      const float f = exp2f((M - Mc) * a.scale_log2);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) acc[c] *= f;
      l *= f;
      M = Mc;
    }
    // weights p_t = 2^((s_t - M) * scale * log2 e)
    for (int i = threadIdx.x; i < n; i += kTokWarps * 32) s_p[i] = exp2f((s_p[i] - M) * a.scale_log2);
    __syncthreads();
    // this warp's contiguous slice, kTokBatch rows in flight while the
    // previous kTokBatch are accumulated
    const int per = static_cast<int>(ceil_div(n, kTokWarps));
    const int i0 = warp * per, i1 = min(n, i0 + per);
    Raw xa[kTokBatch], xb[kTokBatch];
    auto load = [&](int i, Raw (&x)[kTokBatch]) {
#pragma unroll
      for (int u = 0; u < kTokBatch; ++u) {
        if (i + u < i1) x[u] = load_v<D>(vbase + static_cast<int64_t>(s_idx[i + u]) * a.v_st);
      }
    };
    auto consume = [&](int i, const Raw (&x)[kTokBatch]) {
#pragma unroll
      for (int u = 0; u < kTokBatch; ++u) {
        if (i + u < i1) {
          const float p = s_p[i + u];
          l += p;
          acc_v<D, F16>(p, x[u], acc);
        }
      }
    };
    int i = i0;
    if (i < i1) load(i, xa);
    while (i < i1) {
      if (i + kTokBatch < i1) load(i + kTokBatch, xb);
      consume(i, xa);
      i += kTokBatch;
      if (i >= i1) break;
      if (i + kTokBatch < i1) load(i + kTokBatch, xa);
      consume(i, xb);
      i += kTokBatch;
    }
    __syncthreads();  // the chunk's staging may be overwritten
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

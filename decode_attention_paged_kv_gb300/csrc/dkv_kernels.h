// dkv_kernels.h -- internal interface between the C ABI (api.cu) and the
// kernel translation units: argument structs, tiling constants and launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dkv {

constexpr int kPage = 16;             // tokens per page (S)
constexpr int kConsumerWarps = 4;     // attention: warps that compute
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;  // + one producer warp

// Pages one attention CTA streams in the exact path.  Depends only on d, so the
// sequence chunking (and hence every result bit) is the same whether the call
// covers all kv heads or one.  512 KiB of K+V per CTA.
constexpr int full_pages_per_chunk(int d) { return d == 128 ? 64 : 128; }
// Selected pages one attention CTA gathers in the sparse path (128 KiB K+V).
constexpr int select_pages_per_chunk(int d) { return d == 128 ? 16 : 32; }
// Pipeline depth: pages of K+V in flight per CTA (96 KiB of shared memory).
constexpr int attn_stages(int d) { return d == 128 ? 12 : 24; }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct AttnArgs {
  const void* q;
  int64_t q_sb, q_sh;          // elements
  int B, Hq, Hkv, G, N, P;
  float scale_log2;            // softmax scale * log2(e)
  int pages_per_chunk;
  int n_chunks;
  float* part_ml;              // [B, Hq, n_chunks, 2]  (running max in log2 units, sum)
  float* part_o;               // [B, Hq, n_chunks, d]  unnormalised
  const uint32_t* bitmaps;     // sparse path: [B, Hq, W32] selected-page bits
  int W32;
  uint32_t* status;
  uint64_t wait_limit_ns;
};

struct CombineArgs {
  const float* part_ml;
  const float* part_o;
  int n_chunks;
  int Hq;
  void* out;
  int out_dtype;               // 0 bf16, 1 fp16, 2 fp32
  int64_t o_sb, o_sh;
};

struct ScoreArgs {
  const void* q;
  int64_t q_sb, q_sh;
  const void* meta_min;
  const void* meta_max;
  int B, Hq, Hkv, G, P;
  float* scores;               // [B, Hq, P]
};

struct TopkArgs {
  const float* scores;         // [rows, P]
  int rows, P, kk;
  int32_t* selected;           // [rows, kk]
  uint32_t* bitmaps;           // [rows, W32]
  int W32;
};

struct MetaArgs {
  const void* data;            // dense K or Q4 codes
  const void* gmin;
  const void* gmax;
  int64_t sb, sh, gsb, gsh;
  int B, Hkv, N, P, d;
  void* meta_min;
  void* meta_max;
};

// Launchers: return the launch's cudaError_t.
cudaError_t launch_attn(int d, bool f16, bool sparse, const AttnArgs& a, const CUtensorMap& mk,
                        const CUtensorMap& mv, dim3 grid, cudaStream_t s);
cudaError_t launch_combine(int d, const CombineArgs& a, int rows, cudaStream_t s);
cudaError_t launch_score(int d, bool f16, const ScoreArgs& a, cudaStream_t s);
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s);
cudaError_t launch_meta(bool q4, bool f16, const MetaArgs& a, cudaStream_t s);
cudaError_t launch_quant4(int64_t rows, int d, const void* x, void* codes, void* gmin,
                          void* gmax, cudaStream_t s);
cudaError_t launch_dequant4(int64_t rows, int d, const void* codes, const void* gmin,
                            const void* gmax, void* x, cudaStream_t s);

}  // namespace dkv

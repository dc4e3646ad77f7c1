// dkv_kernels.h -- internal interface between the C ABI (api.cu) and the
// kernel translation units: argument structs, tiling constants and launchers.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace dkv {

constexpr int kPage = 16;             // tokens per page (S)
constexpr int kConsumerWarps = 4;     // attention: warps that compute
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;  // + one producer warp

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tokens batch entry b attends: lens[b] clamped into [1, N], or N without lens.
__device__ __forceinline__ int seq_len_of(const int32_t* lens, int b, int N) {
  return lens != nullptr ? min(max(lens[b], 1), N) : N;
}

// Selection pages of S tokens (S a multiple of the cache's 16-token pages):
// the cache pages inside selection page j of a sequence of n tokens.  Every
// page but the sequence's last holds S / 16 of them.
__device__ __forceinline__ int cache_pages_in(int j, int S, int n) {
  return min(S / kPage, static_cast<int>(ceil_div(n, kPage)) - j * (S / kPage));
}

// Split-K: a (batch, kv head) is cut into at most kMaxChunks chunks of pages;
// each chunk's partial (max, sum, o) is merged by merge_kernel.
constexpr int kMaxChunks = 256;

// Pages one attention work item streams in the exact path: 512 KiB of K+V at
// least, more for long contexts so a (batch, kv head) never has more than
// kMaxChunks chunks.  Depends only on (P, d) -- not on the batch or the number
// of kv heads in the call -- so one kv head at a time gives bitwise the
// all-heads result.
inline int full_pages_per_chunk(int64_t P, int d) {
  const int64_t base = d == 128 ? 64 : 128;
  const int64_t need = ceil_div(P, kMaxChunks);
  return static_cast<int>(need > base ? ceil_div(need, 16) * 16 : base);
}
// Selected pages one sparse work item gathers (256 KiB of K+V at least), from a
// union of at most `union_max` pages per (batch, kv head).
constexpr int kMaxSelectList = 256;  // shared-memory page list capacity
inline int select_pages_per_chunk(int64_t union_max, int d) {
  const int64_t base = d == 128 ? 32 : 64;
  const int64_t need = ceil_div(union_max, kMaxChunks);
  return static_cast<int>(need > base ? need : base);
}
// The per-(batch, kv head) selection kernel holds a head's P scores in a
// warp's registers, 64 a lane at most; longer contexts take the separate
// score / top-K / union kernels.
constexpr int kUnitMaxP = 64 * 32;  // 2048 pages (32K tokens)
// Pipeline depth: pages of K+V in flight per CTA (96 KiB of shared memory), as
// one sub-ring per consumer warp (a multiple of kConsumerWarps).
constexpr int attn_stages(int d) { return d == 128 ? 12 : 24; }
// Resident attention CTAs per SM (the persistent grid is this times the SMs).
constexpr int kAttnCtasPerSm = 2;
// Two resident CTAs need at most 168 registers a thread: an SM's registers are
// split over its four sub-partitions (16384 each) and warps are placed on them
// by index, so two CTAs of five warps put three warps on one sub-partition
// (3 x 32 x 168 <= 16384).  The launch sizes the persistent grid from the
// occupancy the compiled kernel actually gets.

// One K or V cache in the 4-bit group-of-64 format (device pointers).
struct Q4View {
  const uint8_t* codes;        // [B, Hkv, N, d/2]
  const __half* gmin;          // [B, Hkv, N, d/64]
  const __half* gmax;
  int64_t sb, sh;              // codes strides, bytes
  int64_t gsb, gsh;            // gmin / gmax strides, elements
};

struct AttnArgs {
  const void* q;
  int64_t q_sb, q_sh;          // elements
  int B, Hq, Hkv, G, N, P;
  float scale_log2;            // softmax scale * log2(e)
  int pages_per_chunk;
  int n_chunks;                // per (batch, kv head), <= kMaxChunks
  int n_items;                 // B * Hkv * n_chunks work items
  float* part_ml;              // [B, Hq, n_chunks, 2]  (max in log2 units, sum)
  float* part_o;               // [B, Hq, n_chunks, d]  unnormalised
  // sparse 4-bit path with n_chunks == 1: each item is its rows' whole result,
  // written normalised to out (strides in elements), no partials, no merge
  void* out;
  int out_dtype;               // 0 bf16, 1 fp16, 2 fp32
  int64_t o_sb, o_sh;
  uint32_t* work_counter;      // next work item; zero between calls
  uint32_t* exit_counter;      // CTAs done fetching; zero between calls
  // sparse path: per (batch, kv head) the ascending union of the group's
  // selected pages, as (page, bit per query head that chose it)
  const int2* union_list;      // [B * Hkv, union_stride]
  const int* union_count;      // [B * Hkv]
  int union_stride;
  // Selection pages of 16 >> sub_log2 tokens (sub_log2 = 1, 2: 8 or 4 tokens,
  // 2 or 4 to a cache page): a union entry's mask then holds 1 << sub_log2
  // bits per query head, one per sub-page (bit (h << sub_log2) + sub-page);
  // 0 otherwise (one bit per head).
  int sub_log2;
  // Per (batch, kv head): non-zero once the selection kernel has written that
  // unit's union.  When set, the kernel starts alongside the selection grid
  // and waits unit by unit; nullptr: it waits for the whole previous grid.
  const uint32_t* unit_ready;  // [B * Hkv] or nullptr
  Q4View k4, v4;               // 4-bit caches (the dense path uses the tensor maps)
  // paged caches: page j of batch entry b is pool block bt[b * bts + j] (the
  // tensor maps then view the pool); nullptr for a [B, Hkv, N, d] cache
  const int32_t* bt;
  int64_t bts;
  int nblocks;
  const int32_t* lens;         // per-sequence lengths [B] or nullptr (all N)
  uint32_t* status;
  uint64_t wait_limit_ns;
  // Cross-step page reuse (sparse path, 16-bit caches; nullptr when unused):
  // per (batch, kv head) and cache page, the step that last gathered the page
  // (0: never), and counters of pages gathered and of those gathered at
  // hot_step - 1 too.  The pages of units (b * Hkv + kv head) below
  // hot_keep_units -- as many as half the L2 holds -- are loaded with an L2
  // evict-last policy, so the next step finds the ones it selects again;
  // every other page streams through with evict-first.
  uint32_t* hot_stamp;         // [B * Hkv, hot_pages]
  int hot_pages;               // cache pages per (batch, kv head)
  uint32_t hot_step;           // this call's step, >= 1
  int hot_keep_units;
  unsigned long long* hot_stats;  // [0] pages gathered, [1] of them gathered at hot_step - 1
};

struct MergeArgs {
  const float* part_ml;
  const float* part_o;
  int n_chunks;
  int Hq;
  // sparse path: only the chunks that hold pages, ceil(count / ppc) per unit
  const int* union_count;      // [B * Hkv] or nullptr (every chunk is valid)
  int pages_per_chunk, G, Hkv;
  void* out;
  int out_dtype;               // 0 bf16, 1 fp16, 2 fp32
  int64_t o_sb, o_sh;
  // exact path with per-sequence lengths: ceil(ceil(N_b / 16) / ppc) chunks per row
  const int32_t* lens;
  int N;
};

struct ScoreArgs {
  const void* q;
  int64_t q_sb, q_sh;
  const void* meta_min;
  const void* meta_max;
  int B, Hq, Hkv, G, P;
  float* scores;               // [B, Hq, P]
  int exact;                   // 1: meta_max holds single keys (m = M): score q . k once
};

// 8-bit page metadata: per page a grid dec(c) = fma(c, step, lo) and, per
// channel, the codes of m rounded down and of M rounded up on it.
struct Meta8Args {
  const uint16_t* meta_min;    // [B, Hkv, P, d] bf16 / fp16 bits
  const uint16_t* meta_max;
  uint8_t* code_min;           // [B, Hkv, P, d]
  uint8_t* code_max;
  float* lo;                   // [B, Hkv, P]
  float* step;
  int B, Hkv, P, d, S, N;
  const int32_t* lens;         // per-sequence lengths [B] or nullptr
};

// Bound scores over 8-bit metadata into [B, Hq, P] (same layout as ScoreArgs).
struct Score8Args {
  const void* q;
  int64_t q_sb, q_sh;
  const uint8_t* code_min;
  const uint8_t* code_max;
  const float* lo;
  const float* step;
  int B, Hq, Hkv, G, P;
  float* scores;
};

struct TopkArgs {
  const float* scores;         // [rows, P]
  int rows, P, kk;
  int Hq;                      // rows are (b, h): b * Hq + h
  int group;                   // heads whose scores a row sums (1, or G for one selection per group)
  const int32_t* lens;         // per-sequence lengths [B] or nullptr; N = the longest
  int N;
  int S;                       // tokens per selection page
  int32_t* selected;           // [rows, kk]
  uint32_t* bitmaps;           // [rows, W32]
  int W32;
  // One query head per kv head at 16-token pages: the units' union lists,
  // written here from the rows (nullptr: the union kernel builds them)
  int2* union_list;            // [rows, union_stride]
  int* union_count;            // [rows]
  int union_stride;
};

struct UnionArgs {
  const uint32_t* bitmaps;     // [B, Hq, W32] over selection pages
  int Hq, Hkv, G, P, W32;
  int2* union_list;            // cache pages (16 tokens), each selection page expanded
  int* union_count;
  int union_stride;
  const int32_t* lens;         // per-sequence lengths [B] or nullptr; N = the longest
  int N;
  int S;                       // tokens per selection page (16, 32 or 64)
};

// Per (batch, kv head) unit: bound scores, per-head top-K and union; a
// persistent grid of at most num_sms CTAs takes the units in turn.
struct UnitSelectArgs {
  const void* q;
  int64_t q_sb, q_sh;
  const void* meta_min;        // [B, Hkv, P, d]
  const void* meta_max;
  // 8-bit metadata (the M8 kernel; the codes come through the tensor maps):
  // r = lo * sum_i q_i + step * (q+ . code_max + q- . code_min), lo / step [B, Hkv, P]
  const float* lo;
  const float* step;
  int B, Hq, Hkv, G, P, kk;
  int32_t* selected;           // [B, Hq, kk]
  int2* union_list;            // [B * Hkv, union_stride]
  int* union_count;            // [B * Hkv]
  int union_stride;
  uint32_t* unit_ready;        // [B * Hkv] or nullptr: set once a unit's union is written
  int group;                   // 1: one selection per kv head group (summed scores)
  const int32_t* lens;         // per-sequence lengths [B] or nullptr; N = the longest
  int N;
  int S;                       // tokens per selection page (16, 32 or 64); the union
                               // list holds 16-token cache pages
  uint32_t* status;
  uint64_t wait_limit_ns;
  int num_sms;                 // multiprocessors of the device (grid bound)
};

// Attention over each (b, q-head)'s top-K tokens (token-level sparse attention).
struct TokenAttnArgs {
  const float* scores;         // [B * Hq, N] exact q . k_t
  const int32_t* selected;     // [B * Hq, kk] ascending token indices
  int kk, N, Hq, G;
  const void* v;               // V [B, Hkv, N, d]
  int64_t v_sb, v_sh, v_st;    // elements
  float scale_log2;            // softmax scale * log2(e)
  void* out;
  int out_dtype;               // 0 bf16, 1 fp16, 2 fp32
  int64_t o_sb, o_sh;
};

struct MetaArgs {
  const void* data;            // dense K or Q4 codes
  const void* gmin;
  const void* gmax;
  int64_t sb, sh, gsb, gsh;
  int B, Hkv, N, P, d;
  void* meta_min;
  void* meta_max;
  const int32_t* bt;           // paged cache: block table [B, P] (row stride bts), else nullptr
  int64_t bts;
  int nblocks;
  const int32_t* lens;         // per-sequence lengths [B] or nullptr (all N)
  int S;                       // tokens per metadata page (16, 32 or 64); P = ceil(N / S)
  int last_only;               // 1: only the page holding each sequence's last token
};

// Launch `kern` with programmatic stream serialisation, so it may begin while
// the previous kernel in the stream drains (every kernel here calls
// griddep_wait() before touching data a predecessor could have written).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Launchers: return the launch's cudaError_t.
cudaError_t launch_attn(int d, bool f16, bool sparse, const AttnArgs& a, const CUtensorMap& mk,
                        const CUtensorMap& mv, int num_sms, cudaStream_t s);
cudaError_t launch_attn_q4(int d, bool sparse, const AttnArgs& a, int num_sms, cudaStream_t s);
// Resident attention CTAs per SM for one instantiation (1 .. kAttnCtasPerSm).
cudaError_t attn_ctas_per_sm(int d, bool f16, bool sparse, bool q4, int* out);
cudaError_t launch_merge(int d, const MergeArgs& m, int rows, cudaStream_t s);
cudaError_t launch_token_attn(int d, bool f16, const TokenAttnArgs& a, int rows, cudaStream_t s);
cudaError_t launch_score(int d, bool f16, const ScoreArgs& a, cudaStream_t s);
cudaError_t launch_score8(int d, bool f16, const Score8Args& a, cudaStream_t s);
cudaError_t launch_meta8(bool f16, const Meta8Args& a, cudaStream_t s);
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s);
cudaError_t launch_union(const UnionArgs& a, int units, cudaStream_t s);
// Shared memory of unit_select_kernel for G heads of P pages (P <= kUnitMaxP).
size_t unit_select_smem(int d, bool m8, int G, int P);
// mmx / mmn: maps over meta_max / meta_min, box {64, 64 pages, d/64, 1, 1}; with
// m8, over code_max / code_min, box {d bytes, 64 pages, 1, 1, 1}.
cudaError_t launch_unit_select(int d, bool f16, bool m8, const UnitSelectArgs& a,
                               const CUtensorMap& mmx, const CUtensorMap& mmn, cudaStream_t s);

cudaError_t launch_meta(bool q4, bool f16, const MetaArgs& a, cudaStream_t s);
cudaError_t launch_quant4(int64_t rows, int d, const void* x, void* codes, void* gmin,
                          void* gmax, cudaStream_t s);
cudaError_t launch_dequant4(int64_t rows, int d, const void* codes, const void* gmin,
                            const void* gmax, void* x, cudaStream_t s);

}  // namespace dkv

/*
 * dkv.h -- C ABI of libdkv: single-token decode attention over a paged KV cache
 * on NVIDIA GB300 (sm_103a).
 *
 * The operations and where they are defined:
 *
 *   dkv_kv_meta_build       page metadata phi(K_j) = (m_j, M_j), the channel-wise
 *                           min / max of each page of S keys.
 *                           "TinyServe: Query-Aware Cache Selection for Efficient
 *                           LLM Serving", 方法细节: 结构化内存布局 and
 *                           相关性函数实例化.
 *   dkv_decode_attn_full    exact decode attention Softmax(q K^T * scale) V per
 *                           query head, with grouped kv heads (GQA).
 *                           "论文阅读：HeadInfer", 核心 idea (the A^(h) equation);
 *                           TinyServe, 标准Transformer解码层的注意力计算.
 *   dkv_decode_attn_select  query-aware page-sparse attention: bound score
 *                           r(q, phi_j) = sum_i (q_i >= 0 ? q_i M_ji : q_i m_ji),
 *                           top-K pages, attention over the selected pages only.
 *                           TinyServe, 相关性函数实例化, 问题公式化定义 and
 *                           Algorithm 1 (Fused Query-Aware Sparse Attention
 *                           Kernel), steps 1-4.
 *   dkv_kv_meta8_build /    the same metadata in one byte per channel: a
 *   dkv_decode_attn_select_ per-page grid with m rounded down and M rounded up,
 *   meta8                   so r stays an upper bound (TinyServe,
 *                           相关性函数实例化; the byte form is not on the pages).
 *   dkv_kv_quant4 /         4-bit KV format: groups of 64 channels along the head
 *   dkv_kv_dequant4         dimension, per-group min / max, 4-bit codes,
 *                           dequantised to fp16 before use.
 *                           "FlexGen: High-Throughput Generative Inference of
 *                           Large Language Models with a Single GPU" (解读),
 *                           4-bit 近似方法.
 *
 * Conventions shared by every entry point:
 *   - Every data pointer is a DEVICE pointer owned by the caller, 16-byte
 *     aligned.  The library allocates no device memory and keeps no per-call
 *     state.  Scratch space is a caller-owned `workspace` of
 *     dkv_workspace_bytes() bytes, zero-filled once before its first use; each
 *     call that completes returns the workspace's counters to zero, so it can
 *     be reused by any later call (of any shape that fits).  The counters
 *     live in the first DKV_WORKSPACE_HEADER_BYTES bytes, which no call uses
 *     for anything else; the rest is scratch whose contents never matter.
 *     After a device error (dkv_read_device_status) zero-fill the header (or
 *     the whole workspace) again.  One workspace serves one call at a time:
 *     calls that may overlap on the GPU need separate ones.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every call is asynchronous on that stream; only
 *     dkv_read_device_status synchronises.
 *   - Layouts are row-major with the innermost (channel) stride 1:
 *       q        [B, Hq, d]        strides q_stride_b, q_stride_h (elements)
 *       out      [B, Hq, d]        strides o_stride_b, o_stride_h (elements)
 *       K, V     [B, Hkv, N, d]    token stride d; batch / head strides in dkv_kv
 *       meta     [B, Hkv, P, d]    contiguous, P = ceil(N / S)
 *       selected [B, Hq, kk]       contiguous int32, kk = min(top_k, P)
 *     Query head h reads kv head h / (Hq / Hkv).
 *   - Argument errors are returned before anything is launched.  Launch
 *     failures return DKV_ERR_CUDA.  Errors found on the device (a bounded
 *     wait that expired, an in-kernel check) are written to a status word at
 *     the start of the workspace and read back with dkv_read_device_status.
 *     No call aborts the process.
 *   - Supported: d in {64, 128}; S in {4, 8, 16, 32, 64} (the page of the metadata
 *     and of selection; the cache itself is read in pages of 16 tokens, and a
 *     paged cache's blocks hold 16 tokens); Hq % Hkv == 0 and Hq / Hkv <= 8;
 *     1 <= N < 2^31; bf16 or fp16 dense caches (q in the same dtype), or the
 *     4-bit format with fp16 q.  A ragged last page is masked.
 */
#ifndef DKV_H_
#define DKV_H_

#include <stddef.h>
#include <stdint.h>

/* Workspace header: the status word and the work counters. */
#define DKV_WORKSPACE_HEADER_BYTES ((size_t)256)

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dkv_status {
  DKV_OK = 0,
  DKV_ERR_NULL = 1,           /* a required pointer is NULL */
  DKV_ERR_SHAPE = 2,          /* a size or stride is out of range */
  DKV_ERR_ALIGN = 3,          /* a pointer or stride is not 16-byte aligned */
  DKV_ERR_DTYPE = 4,          /* unsupported dtype / format combination */
  DKV_ERR_UNSUPPORTED = 5,    /* d, S or Hq/Hkv outside what the kernels cover */
  DKV_ERR_WORKSPACE = 6,      /* workspace NULL or smaller than required */
  DKV_ERR_CUDA = 7,           /* a CUDA runtime call or kernel launch failed */
  DKV_ERR_DEVICE_TIMEOUT = 8, /* device status: a bounded wait expired */
  DKV_ERR_DEVICE_CHECK = 9    /* device status: an in-kernel check failed */
} dkv_status;

typedef enum dkv_dtype { DKV_BF16 = 0, DKV_FP16 = 1, DKV_FP32 = 2 } dkv_dtype;

typedef enum dkv_kv_format {
  DKV_KV_DENSE = 0, /* data: [B, Hkv, N, d] elements of `dtype` (bf16 or fp16) */
  DKV_KV_Q4G64 = 1, /* data: codes [B, Hkv, N, d/2] bytes, channel 2i in the low
                       nibble of byte i; gmin / gmax: [B, Hkv, N, d/64] fp16 */
  DKV_KV_PAGED = 2  /* a pool of pages (blocks) of S = 16 tokens, `dtype` bf16 or
                       fp16: block n of kv head h starts at data + n * stride_b +
                       h * stride_h (elements), token stride d.  block_table
                       [B, P] int32 (row stride block_table_stride, at least
                       P = ceil(N / 16) when B > 1) maps page j
                       of batch entry b to its block; entries outside
                       [0, num_blocks) are clamped into it (nothing outside
                       the pool is read) and the attention calls then record
                       DKV_ERR_DEVICE_CHECK in the workspace status word
                       (dkv_kv_meta_build, which has no workspace, only
                       clamps).  A sequence's ragged
                       last page may hold anything past N: it is never used.
                       K and V of one call share the table.  ("TinyServe"
                       结构化内存布局: the cache as pages of S tokens.) */
} dkv_kv_format;

/* One K or V cache. */
typedef struct dkv_kv {
  int32_t format;           /* dkv_kv_format */
  int32_t dtype;            /* DENSE: DKV_BF16 | DKV_FP16.  Q4G64: DKV_FP16 */
  const void* data;         /* device pointer, see dkv_kv_format */
  const void* gmin;         /* Q4G64 only (else NULL) */
  const void* gmax;         /* Q4G64 only (else NULL) */
  int64_t stride_b;         /* of data: elements (DENSE) or bytes (Q4G64 codes) */
  int64_t stride_h;         /*   token stride is d (DENSE) or d/2 (codes) */
  int64_t gstride_b;        /* of gmin / gmax, in fp16 elements; Q4G64 only, */
  int64_t gstride_h;        /*   multiples of 8 (16 bytes: contiguous bounds need
                               N * d / 64 % 8 == 0); token stride is d/64 */
  const int32_t* block_table;   /* PAGED only (else NULL): [B, P] block indices */
  int64_t block_table_stride;   /* PAGED only: elements from one batch row to the next */
  int32_t num_blocks;           /* PAGED only: blocks in the pool */
} dkv_kv;

/* Problem description shared by the attention and metadata calls. */
typedef struct dkv_params {
  int32_t batch;            /* B  >= 1 */
  int32_t num_q_heads;      /* Hq >= 1 */
  int32_t num_kv_heads;     /* Hkv >= 1, Hq % Hkv == 0, Hq / Hkv <= 8 */
  int32_t head_dim;         /* d in {64, 128} */
  int32_t seq_len;          /* N >= 1 context tokens, all attended */
  int32_t page_size;        /* S in {4, 8, 16, 32, 64}: tokens per metadata /
                               selection page ("TinyServe" 结构化内存布局 and its
                               page-size study); P = ceil(N / S).  Pages of 4
                               or 8 tokens are gathered as the 16-token cache
                               page that holds them, with the tokens of
                               unselected pages masked out.  The exact path
                               does not depend on it. */
  int64_t q_stride_b, q_stride_h;   /* q, in elements */
  int64_t o_stride_b, o_stride_h;   /* out, in elements */
  float scale;              /* softmax scale, usually 1/sqrt(d) */
  uint32_t flags;           /* DKV_FLAG_* ; 0 for normal use */
  const int32_t* seq_lens;  /* NULL, or a DEVICE array [B]: batch entry b attends
                               its first N_b tokens (clamped into [1, seq_len]);
                               seq_len is then the longest and sizes P, the
                               workspace and the block table.  Tokens past N_b
                               in the cache may hold anything.  Metadata rows
                               of pages past ceil(N_b / S) are not written;
                               selection keeps min(top_k, ceil(N_b / S)) pages
                               and pads `selected` rows with -1.  Dense and
                               paged caches only (not Q4G64). */
} dkv_params;

/* Test hook: every bounded device wait gives up at once, so the timeout path
   (status word set, in-flight copies drained, clean exit) runs without a hang. */
#define DKV_FLAG_FORCE_TIMEOUT 0x1u
/* dkv_decode_attn_select only: one selection per kv head group (GQA).  Page
   j's score is the sum of the group's bound scores, sum_h r(q_h, phi_j) (the
   sum over heads h = 0 .. G-1 in that order, in fp32); the group keeps its
   top_k pages and every head of the group attends them, so the `selected`
   rows of a group are identical.  The sum stays an upper bound:
   sum_h r(q_h, phi_j) >= max over the page's keys k of sum_h q_h . k.
   ("TinyServe: Query-Aware Cache Selection for Efficient LLM Serving",
   相关性函数实例化, defines r for one query vector; summing over a group is a
   reading for grouped heads.) */
#define DKV_FLAG_GROUP_SELECT 0x2u

/* Bytes of workspace the attention calls need for `p` (top_k = 0: the exact
   path; top_k >= 1: the sparse path).  0 if `p` is invalid.  Host only. */
size_t dkv_workspace_bytes(const dkv_params* p, int32_t top_k);

/* Page metadata.  meta_min / meta_max: [B, Hkv, P, d] contiguous, in K's dtype
   (fp16 for a Q4G64 cache, built from the dequantised fp16 keys).  m_j / M_j
   are exact: minimum and maximum of the stored values (total order, -0 < +0).
   Uses p->batch, num_kv_heads, head_dim, seq_len, page_size. */
dkv_status dkv_kv_meta_build(const dkv_params* p, const dkv_kv* K, void* meta_min,
                             void* meta_max, void* stream);

/* Page metadata after a decode step appended tokens: rebuilds, for every
   (batch entry b, kv head), only the page holding the sequence's last token
   N_b - 1 (N_b from seq_lens, else seq_len), the one page an appended token
   changes; every other page's (m_j, M_j) is left as it is.  Same arguments
   and layout as dkv_kv_meta_build, whose result it reproduces bit for bit
   when the other pages are already built.  ("TinyServe: Query-Aware Cache
   Selection for Efficient LLM Serving", 结构化内存布局 and 系统实现意义: the
   page metadata is kept alongside the cache as it grows.) */
dkv_status dkv_kv_meta_append(const dkv_params* p, const dkv_kv* K, void* meta_min,
                              void* meta_max, void* stream);

/* Exact decode attention.  out [B, Hq, d] in out_dtype (DKV_FP32 | DKV_BF16 |
   DKV_FP16).  Splits the sequence into fixed chunks whose length depends only
   on d, so evaluating one kv head at a time (a view with Hkv = 1) gives results
   bitwise identical to the all-heads call. */
dkv_status dkv_decode_attn_full(const dkv_params* p, const void* q, const dkv_kv* K,
                                const dkv_kv* V, void* out, int32_t out_dtype,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Query-aware page-sparse decode attention.  For each (b, q-head): bound
   scores of all P pages from meta_min / meta_max, the top_k best pages (ties
   to the lower page index; top_k clamped to P), attention over those pages'
   tokens only (softmax normalised over them).  `selected` (nullable) receives
   the chosen pages [B, Hq, min(top_k, P)] in ascending order. */
dkv_status dkv_decode_attn_select(const dkv_params* p, const void* q, const dkv_kv* K,
                                  const dkv_kv* V, const void* meta_min,
                                  const void* meta_max, int32_t top_k, void* out,
                                  int32_t out_dtype, int32_t* selected, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* dkv_decode_attn_select as one step of a decode loop that keeps hot pages
   resident across steps ("TinyServe: Query-Aware Cache Selection for
   Efficient LLM Serving", 内存效率量化模型构建 / 单步解码内存移动公式: a
   step moves the metadata of all pages plus only the rho K pages not already
   held; 系统实现意义: hot pages stay resident).  The cache is HBM-resident,
   so "resident" here means the L2: the pages of the first (batch entry, kv
   head) units, as many as half the L2 holds at the selection's largest
   union, are loaded with an L2 evict-last policy and stay there for the
   next step, which finds those it selects again; every other page streams
   through with evict-first.  Results are exactly those
   of dkv_decode_attn_select on the same arguments; only the cache policy and
   the counters below differ.
   - hot_state: caller-owned DEVICE buffer of dkv_hot_state_bytes(p) bytes
     (16-byte aligned), zero-filled once before the first step of a decode
     sequence and then passed, unchanged, to every step of it.  It holds a
     256-byte header -- u64 at offset 0: cache pages gathered so far, u64 at
     offset 8: how many of them the step before had gathered too, both
     summed over calls (rho of a run = 1 - [8] / [0]; the caller may zero
     them between reads) -- and one u32 stamp per (batch entry, kv head,
     16-token cache page): the last step that gathered it.
   - step: 1 for the first step, +1 for each step after (a page counts as
     held when its stamp is step - 1).
   - 16-bit caches only (DKV_KV_DENSE or DKV_KV_PAGED; DKV_ERR_UNSUPPORTED for
     DKV_KV_Q4G64).  One hot_state serves one call at a time. */
size_t dkv_hot_state_bytes(const dkv_params* p);
dkv_status dkv_decode_attn_select_hot(const dkv_params* p, const void* q, const dkv_kv* K,
                                      const dkv_kv* V, const void* meta_min,
                                      const void* meta_max, int32_t top_k, void* out,
                                      int32_t out_dtype, int32_t* selected, void* hot_state,
                                      size_t hot_state_bytes, int32_t step, void* workspace,
                                      size_t workspace_bytes, void* stream);

/* 8-bit page metadata from (meta_min, meta_max) [B, Hkv, P, d] of dtype
   meta_dtype (DKV_BF16 | DKV_FP16).  TinyServe's bound (相关性函数实例化) needs
   only m_j <= k <= M_j channel by channel; this stores that interval on a
   per-page grid at one byte per channel instead of two.  No page defines this
   form; it is the plainest that keeps r an upper bound.  Per page:
     lo = min_i m_i, hi = max_i M_i (a zero stored as +0), written to lo [B, Hkv, P]
     step = fp32(fp32(hi - lo) / 255), raised one ulp at a time until
            dec(255) >= hi, where dec(c) = fmaf(c, step, lo); 0 when hi == lo;
            written to step [B, Hkv, P] (fp32)
     code_min [B, Hkv, P, d] u8 = the largest c with dec(c) <= m_i
     code_max [B, Hkv, P, d] u8 = the smallest c with dec(c) >= M_i.
   Uses p->batch, num_kv_heads, head_dim, seq_len, page_size and seq_lens
   (pages past a shorter sequence are not written).  Metadata must be finite.
   code_min / code_max / meta 16-byte aligned, lo / step 4-byte aligned. */
dkv_status dkv_kv_meta8_build(const dkv_params* p, const void* meta_min, const void* meta_max,
                              int32_t meta_dtype, void* code_min, void* code_max, void* lo,
                              void* step, void* stream);

/* dkv_decode_attn_select over 8-bit metadata (dkv_kv_meta8_build): the bound
   score of page j is r = sum_i q_i * dec(q_i >= 0 ? code_max_i : code_min_i),
   an upper bound of max q.k over the page's keys, then top-K, union and
   attention exactly as in dkv_decode_attn_select.  Same workspace
   (dkv_workspace_bytes(p, top_k)), flags, page sizes, cache formats and
   per-sequence lengths. */
dkv_status dkv_decode_attn_select_meta8(const dkv_params* p, const void* q, const dkv_kv* K,
                                        const dkv_kv* V, const void* code_min,
                                        const void* code_max, const void* lo, const void* step,
                                        int32_t top_k, void* out, int32_t out_dtype,
                                        int32_t* selected, void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Token-level sparse decode attention ("FlexGen: High-Throughput Generative
   Inference of Large Language Models with a Single GPU" (解读), its sparse
   attention: each query keeps the top 10% of the K cache's indices and loads
   only that subset of V).  For each (b, q-head): the exact scores q . k_t of
   all N tokens, the top_k highest (ties to the lower token index; top_k
   clamped to N), softmax over those tokens' scaled scores, and the weighted
   sum of their V rows.  K and V dense bf16 / fp16 (q in the same dtype); K
   contiguous [B, Hkv, N, d] (the score pass reads it as one row per token);
   no per-sequence lengths.  `selected` (nullable) receives the tokens
   [B, Hq, min(top_k, N)], ascending.  The workspace needs
   dkv_workspace_bytes_tokens(p, top_k) bytes; page_size is not used. */
dkv_status dkv_decode_attn_topk_tokens(const dkv_params* p, const void* q, const dkv_kv* K,
                                       const dkv_kv* V, int32_t top_k, void* out,
                                       int32_t out_dtype, int32_t* selected, void* workspace,
                                       size_t workspace_bytes, void* stream);
size_t dkv_workspace_bytes_tokens(const dkv_params* p, int32_t top_k);

/* 4-bit group-of-64 quantisation of `rows` fp16 rows of d channels (d % 64 == 0).
   Per group of 64 channels: mn, mx = group min / max (written to gmin / gmax);
   16 levels mn + c * s, c = 0 .. 15, with the step s rounded down from
   (mx - mn) / 15 so that no level passes mx:
     range = fp32_down(mx - mn)
     range >= 451 * 2^-24:  s = fp16_down(fp32_down(range / 15))
     range <  451 * 2^-24:  s = floor(range / (15 g)) * g,
                            g = 2^(floor(log2 max(|mn|, |mx|)) - 22)
     code = 0 if s == 0, else the c nearest to (x - mn) / s (ties to even c)
   (fp32_down / fp16_down: the largest binary32 / binary16 at or below).
   Dequantised values are within (mx - mn)/30 plus half an fp16 ulp of the
   input, for every finite group.  codes [rows, d/2] (channel 2i in the low
   nibble), gmin / gmax [rows, d/64]. */
dkv_status dkv_kv_quant4(int64_t rows, int32_t d, const void* x, void* codes, void* gmin,
                         void* gmax, void* stream);

/* Inverse: x = fp16(mn + code * s), the exact level rounded once to fp16
   (always inside [mn, mx]).  Inputs are finite fp16 values. */
dkv_status dkv_kv_dequant4(int64_t rows, int32_t d, const void* codes, const void* gmin,
                           const void* gmax, void* x, void* stream);

/* Exact decode attention with no workspace argument and no allocation.  The
   pages have no counterpart: this serves callers that cannot allocate device
   memory for the library (a host whose allocator owns the device budget, or a
   loop that must never call cudaMalloc).  Same arguments, layouts and results
   as dkv_decode_attn_full, whose kernels it runs; the scratch is a fixed
   array of DKV_NOALLOC_SCRATCH_BYTES inside the library, held by every GPU that
   loads it until exit.
   - Returns DKV_ERR_WORKSPACE when the problem needs more scratch than that
     (dkv_workspace_bytes(p, 0) > DKV_NOALLOC_SCRATCH_BYTES).
   - The first call on a device looks up the array's address (with that device
     current); make that first call before any stream capture.  The address is
     kept per device and context: a call under another context (after a device
     reset, or with a context of the caller's own current) looks it up again.
   - Every call shares the array: calls that may overlap on the GPU race and
     must be serialised by the caller.
   - A device-side error (an expired bounded wait) cannot be read back with
     dkv_read_device_status; instead every element of that call's `out` is
     set to NaN.  The next call starts clean. */
#define DKV_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
dkv_status dkv_decode_attn_full_noalloc(const dkv_params* p, const void* q, const dkv_kv* K,
                                        const dkv_kv* V, void* out, int32_t out_dtype,
                                        void* stream);

/* Synchronises `stream`, returns the device status word held at the start of
   `workspace` (DKV_OK, DKV_ERR_DEVICE_TIMEOUT or DKV_ERR_DEVICE_CHECK) and
   resets it to DKV_OK.  Returns DKV_ERR_CUDA if the copy itself fails. */
dkv_status dkv_read_device_status(void* workspace, void* stream);

/* Diagnostic with no counterpart in the pages: how many CTAs of the persistent
   attention kernel for (head_dim, dtype, format, sparse != 0) stay resident on
   one multiprocessor of the current device (the grid is this times the SM
   count; the kernels are built for two).  Writes it to *ctas_per_sm.  Returns
   DKV_ERR_UNSUPPORTED for a head_dim / dtype / format the kernels do not
   cover, DKV_ERR_CUDA if the query fails. */
dkv_status dkv_attn_ctas_per_sm(int32_t head_dim, int32_t dtype, int32_t format, int32_t sparse,
                                int32_t* ctas_per_sm);

/* Static description of a status code. */
const char* dkv_status_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* DKV_H_ */

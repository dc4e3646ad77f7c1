// api.cu -- the extern "C" boundary of libdkv (declared in include/dkv.h):
// argument validation, workspace layout, TMA tensor-map encoding and kernel
// launches.  Every argument error is returned before anything is launched.

#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/dkv.h"
#include "dkv_kernels.h"

namespace {

using dkv::ceil_div;

constexpr uint64_t kWaitLimitNs = 200000000ull;  // 200 ms per bounded device wait
constexpr size_t kAlign = 256;
static_assert(DKV_WORKSPACE_HEADER_BYTES == kAlign, "status word and counters");
// Shared memory the per-unit selection kernel may take (one CTA per SM), and
// the shortest context (pages) it is used for.
constexpr size_t kUnitSelectSmemLimit = 227 * 1024;
constexpr int kUnitSelectMinP = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte offsets of the regions inside a caller-provided workspace.
struct WsLayout {
  size_t status = 0;     // u32 device status word (first 256 bytes)
  size_t counter = 0;    // u32 attention work counter, zero between calls
  size_t exit_counter = 0;  // u32 CTAs done fetching, zero between calls
  size_t part_ml = 0;    // [B, Hq, n_chunks, 2] fp32
  size_t part_o = 0;     // [B, Hq, n_chunks, d] fp32
  size_t scores = 0;     // sparse: [B, Hq, P] fp32 (fallback selection only)
  size_t selected = 0;   // sparse: [B, Hq, kk] int32 (used when the caller passes none)
  size_t bitmaps = 0;    // sparse: [B, Hq, W32] u32 (fallback selection only)
  size_t union_list = 0; // sparse: [B * Hkv, union_stride] (page, head mask)
  size_t union_count = 0;  // sparse: [B * Hkv] int32
  size_t unit_ready = 0;   // sparse: [B * Hkv] u32 (per-unit selection only)
  size_t total = 0;
  int n_chunks = 0, pages_per_chunk = 0, kk = 0, W32 = 0, union_stride = 0;
  int64_t n_items = 0;
  bool ok = true;        // false: the sizes exceed what the kernels cover
};

WsLayout layout_for(const dkv_params& p, int top_k) {
  WsLayout L;
  const int d = p.head_dim;
  const int64_t P = ceil_div(p.seq_len, p.page_size);   // selection (metadata) pages
  const int64_t P16 = ceil_div(p.seq_len, dkv::kPage);  // cache pages
  const int64_t rows = static_cast<int64_t>(p.batch) * p.num_q_heads;
  const int64_t units = static_cast<int64_t>(p.batch) * p.num_kv_heads;
  if (top_k <= 0) {
    L.pages_per_chunk = dkv::full_pages_per_chunk(P16, d);
    L.n_chunks = static_cast<int>(ceil_div(P16, L.pages_per_chunk));
  } else {
    const int G = p.num_q_heads / p.num_kv_heads;
    L.kk = static_cast<int>(top_k < P ? top_k : P);
    L.W32 = static_cast<int>(ceil_div(P, 32));
    // the union list holds cache pages: a selection page is S / 16 of them
    const int64_t union_sel = (static_cast<int64_t>(G) * L.kk < P) ? G * L.kk : P;
    // (pages below 16 tokens: each selected page lies in one cache page)
    const int64_t union_max =
        std::min(p.page_size < dkv::kPage ? union_sel : union_sel * (p.page_size / dkv::kPage),
                 P16);
    L.union_stride = static_cast<int>(union_max);
    L.pages_per_chunk = dkv::select_pages_per_chunk(union_max, d);
    if (L.pages_per_chunk > dkv::kMaxSelectList) L.ok = false;
    L.n_chunks = static_cast<int>(ceil_div(union_max, L.pages_per_chunk));
  }
  if (L.n_chunks > dkv::kMaxChunks) L.ok = false;
  L.n_items = units * L.n_chunks;
  if (L.n_items >= (static_cast<int64_t>(1) << 31)) L.ok = false;
  L.status = 0;
  L.counter = 4;
  L.exit_counter = 8;
  size_t off = DKV_WORKSPACE_HEADER_BYTES;
  if (top_k > 0) {
    L.scores = off;
    off = align_up(off + sizeof(float) * rows * P);
    L.selected = off;
    off = align_up(off + sizeof(int32_t) * rows * L.kk);
    L.bitmaps = off;
    off = align_up(off + sizeof(uint32_t) * rows * L.W32);
    L.union_list = off;
    off = align_up(off + 8 * static_cast<size_t>(units) * L.union_stride);
    L.union_count = off;
    off = align_up(off + sizeof(int32_t) * units);
    L.unit_ready = off;
    off = align_up(off + sizeof(uint32_t) * units);
  }
  L.part_ml = off;
  off = align_up(off + sizeof(float) * 2 * rows * L.n_chunks);
  L.part_o = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(d) * rows * L.n_chunks);
  L.total = off;
  return L;
}

// Multiprocessor count of the current device (the persistent attention grid).
int current_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

dkv_status check_params(const dkv_params* p) {
  if (p == nullptr) return DKV_ERR_NULL;
  if (p->batch < 1 || p->num_q_heads < 1 || p->num_kv_heads < 1 || p->seq_len < 1 ||
      p->page_size < 1 || p->head_dim < 1)
    return DKV_ERR_SHAPE;
  if (p->num_q_heads % p->num_kv_heads != 0) return DKV_ERR_SHAPE;
  if (p->head_dim != 64 && p->head_dim != 128) return DKV_ERR_UNSUPPORTED;
  // metadata / selection pages of 4, 8, 16, 32 or 64 tokens (the cache's pages
  // are 16: a smaller selection page is a quarter or half of one)
  if (p->page_size != 4 && p->page_size != 8 && p->page_size != dkv::kPage &&
      p->page_size != 2 * dkv::kPage && p->page_size != 4 * dkv::kPage)
    return DKV_ERR_UNSUPPORTED;
  if (p->num_q_heads / p->num_kv_heads > 8) return DKV_ERR_UNSUPPORTED;
  if (p->batch > 65535 || p->num_kv_heads > 65535) return DKV_ERR_SHAPE;  // grid limits
  if (reinterpret_cast<uintptr_t>(p->seq_lens) & 3u) return DKV_ERR_ALIGN;
  return DKV_OK;
}

dkv_status check_query_out(const dkv_params* p, const void* q, const void* out) {
  if (q == nullptr || out == nullptr) return DKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(out)) return DKV_ERR_ALIGN;
  if (p->q_stride_b % 8 || p->q_stride_h % 8 || p->o_stride_b % 8 || p->o_stride_h % 8)
    return DKV_ERR_ALIGN;
  if (p->q_stride_b < 0 || p->q_stride_h < 0 || p->o_stride_b < 0 || p->o_stride_h < 0)
    return DKV_ERR_SHAPE;
  if (!(p->scale > 0.f) || !isfinite(p->scale)) return DKV_ERR_SHAPE;
  return DKV_OK;
}

dkv_status check_kv(const dkv_params* p, const dkv_kv* kv) {
  if (kv == nullptr || kv->data == nullptr) return DKV_ERR_NULL;
  if (!aligned16(kv->data)) return DKV_ERR_ALIGN;
  if (kv->stride_b < 0 || kv->stride_h < 0) return DKV_ERR_SHAPE;
  if (kv->format == DKV_KV_DENSE) {
    if (kv->dtype != DKV_BF16 && kv->dtype != DKV_FP16) return DKV_ERR_DTYPE;
    if (kv->stride_b % 8 || kv->stride_h % 8) return DKV_ERR_ALIGN;
    return DKV_OK;
  }
  if (kv->format == DKV_KV_PAGED) {
    if (kv->dtype != DKV_BF16 && kv->dtype != DKV_FP16) return DKV_ERR_DTYPE;
    if (kv->stride_b % 8 || kv->stride_h % 8) return DKV_ERR_ALIGN;
    if (kv->block_table == nullptr) return DKV_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(kv->block_table) & 3u) return DKV_ERR_ALIGN;
    if (kv->num_blocks < 1 || kv->block_table_stride < 0) return DKV_ERR_SHAPE;
    // the [B, P] table's rows may not overlap (P = ceil(N / 16) cache pages)
    if (p->batch > 1 && kv->block_table_stride < ceil_div(p->seq_len, dkv::kPage))
      return DKV_ERR_SHAPE;
    return DKV_OK;
  }
  if (kv->format == DKV_KV_Q4G64) {
    if (kv->dtype != DKV_FP16) return DKV_ERR_DTYPE;
    if (kv->gmin == nullptr || kv->gmax == nullptr) return DKV_ERR_NULL;
    if (!aligned16(kv->gmin) || !aligned16(kv->gmax)) return DKV_ERR_ALIGN;
    if (kv->stride_b % 16 || kv->stride_h % 16) return DKV_ERR_ALIGN;
    if (kv->gstride_b < 0 || kv->gstride_h < 0) return DKV_ERR_SHAPE;
    if (kv->gstride_b % 8 || kv->gstride_h % 8) return DKV_ERR_ALIGN;
    return DKV_OK;
  }
  return DKV_ERR_DTYPE;
}

// ------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Map over one dense K or V cache [B, Hkv, N, d] viewed as 5-D
// {64 channels, N tokens, d/64 halves, Hkv, B} with a box of one page
// {64, 16, d/64, 1, 1} and 128-byte swizzle.
// Map over a cache [B, Hkv, N, d] viewed as {64 channels, N, d/64 halves, Hkv,
// B}, or over a pool of blocks as {64 channels, 16 tokens, d/64 halves, Hkv,
// blocks}; box {64, 16, d/64, 1, 1} (one page of one kv head), 128-byte swizzle.
bool encode_page_map(CUtensorMap* map, const dkv_params* p, const dkv_kv* kv) {
  if (!get_encode()) return false;
  const int d = p->head_dim;
  const bool paged = kv->format == DKV_KV_PAGED;
  const cuuint64_t dims[5] = {64,
                              static_cast<cuuint64_t>(paged ? dkv::kPage : p->seq_len),
                              static_cast<cuuint64_t>(d / 64),
                              static_cast<cuuint64_t>(p->num_kv_heads),
                              static_cast<cuuint64_t>(paged ? kv->num_blocks : p->batch)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(d) * 2, 128,
                                 static_cast<cuuint64_t>(kv->stride_h) * 2,
                                 static_cast<cuuint64_t>(kv->stride_b) * 2};
  const cuuint32_t box[5] = {64, static_cast<cuuint32_t>(dkv::kPage),
                             static_cast<cuuint32_t>(d / 64), 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUtensorMapDataType dt = kv->dtype == DKV_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // A size-1 dimension's stride still has to be a valid (16-byte multiple) value.
  cuuint64_t st[4] = {strides[0], strides[1], strides[2], strides[3]};
  if (p->num_kv_heads == 1 && st[2] == 0) st[2] = 16;
  if (dims[4] == 1 && st[3] == 0) st[3] = 16;
  const CUresult r = g_encode(map, dt, 5, const_cast<void*>(kv->data), dims, st, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Map over page metadata [B, Hkv, P, d] (contiguous) viewed like a cache:
// {64 channels, P pages, d/64 halves, Hkv, B}, box {64, box_pages, d/64, 1, 1},
// 128-byte swizzle.
bool encode_meta_map(CUtensorMap* map, const dkv_params* p, const void* meta, bool f16,
                     int box_pages) {
  if (!get_encode()) return false;
  const int d = p->head_dim;
  const uint64_t P = static_cast<uint64_t>(ceil_div(p->seq_len, p->page_size));
  const cuuint64_t dims[5] = {64, P, static_cast<cuuint64_t>(d / 64),
                              static_cast<cuuint64_t>(p->num_kv_heads),
                              static_cast<cuuint64_t>(p->batch)};
  const cuuint64_t st[4] = {static_cast<cuuint64_t>(d) * 2, 128, P * d * 2,
                            P * d * 2 * static_cast<cuuint64_t>(p->num_kv_heads)};
  const cuuint32_t box[5] = {64, static_cast<cuuint32_t>(box_pages),
                             static_cast<cuuint32_t>(d / 64), 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              5, const_cast<void*>(meta), dims, st, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Map over 8-bit metadata codes [B, Hkv, P, d] (u8) for the per-unit selection
// kernel: {d bytes, P pages, 1, Hkv, B}, box {d, box_pages, 1, 1, 1}, with a
// d-byte swizzle (128 or 64 bytes).
bool encode_code_map(CUtensorMap* map, const dkv_params* p, const void* codes, int box_pages) {
  if (!get_encode()) return false;
  const uint64_t d = static_cast<uint64_t>(p->head_dim);
  const uint64_t P = static_cast<uint64_t>(ceil_div(p->seq_len, p->page_size));
  const cuuint64_t dims[5] = {d, P, 1, static_cast<cuuint64_t>(p->num_kv_heads),
                              static_cast<cuuint64_t>(p->batch)};
  const cuuint64_t st[4] = {d, P * d, P * d, P * d * static_cast<cuuint64_t>(p->num_kv_heads)};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(d), static_cast<cuuint32_t>(box_pages), 1, 1,
                             1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(codes),
                              dims, st, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int out_code(int32_t out_dtype) {
  return out_dtype == DKV_FP32 ? 2 : (out_dtype == DKV_FP16 ? 1 : 0);
}

dkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DKV_OK : DKV_ERR_CUDA; }

}  // namespace

extern "C" {

size_t dkv_workspace_bytes(const dkv_params* p, int32_t top_k) {
  if (check_params(p) != DKV_OK || top_k < 0) return 0;
  const WsLayout L = layout_for(*p, top_k);
  return L.ok ? L.total : 0;
}

static dkv_status meta_impl(const dkv_params* p, const dkv_kv* K, void* meta_min,
                            void* meta_max, bool last_only, void* stream) {
  dkv_status st = check_params(p);
  if (st != DKV_OK) return st;
  if ((st = check_kv(p, K)) != DKV_OK) return st;
  if (meta_min == nullptr || meta_max == nullptr) return DKV_ERR_NULL;
  if (!aligned16(meta_min) || !aligned16(meta_max)) return DKV_ERR_ALIGN;
  dkv::MetaArgs a{};
  a.data = K->data;
  a.gmin = K->gmin;
  a.gmax = K->gmax;
  a.sb = K->stride_b;
  a.sh = K->stride_h;
  a.gsb = K->gstride_b;
  a.gsh = K->gstride_h;
  a.B = p->batch;
  a.Hkv = p->num_kv_heads;
  a.N = p->seq_len;
  a.P = static_cast<int>(ceil_div(p->seq_len, p->page_size));
  a.S = p->page_size;
  a.d = p->head_dim;
  a.meta_min = meta_min;
  a.meta_max = meta_max;
  a.lens = p->seq_lens;
  a.last_only = last_only ? 1 : 0;
  if (K->format == DKV_KV_PAGED) {
    a.bt = K->block_table;
    a.bts = K->block_table_stride;
    a.nblocks = K->num_blocks;
  }
  return cuda_status(dkv::launch_meta(K->format == DKV_KV_Q4G64, K->dtype == DKV_FP16, a,
                                      static_cast<cudaStream_t>(stream)));
}

dkv_status dkv_kv_meta_build(const dkv_params* p, const dkv_kv* K, void* meta_min,
                             void* meta_max, void* stream) {
  return meta_impl(p, K, meta_min, meta_max, false, stream);
}

dkv_status dkv_kv_meta_append(const dkv_params* p, const dkv_kv* K, void* meta_min,
                              void* meta_max, void* stream) {
  return meta_impl(p, K, meta_min, meta_max, true, stream);
}

static dkv_status attn_common(const dkv_params* p, const void* q, const dkv_kv* K,
                              const dkv_kv* V, void* out, int32_t out_dtype, void* workspace,
                              size_t workspace_bytes, int top_k, const WsLayout& L) {
  dkv_status st = check_params(p);
  if (st != DKV_OK) return st;
  if ((st = check_query_out(p, q, out)) != DKV_OK) return st;
  if ((st = check_kv(p, K)) != DKV_OK) return st;
  if ((st = check_kv(p, V)) != DKV_OK) return st;
  if (K->format != V->format || K->dtype != V->dtype) return DKV_ERR_DTYPE;
  if (p->seq_lens != nullptr && K->format == DKV_KV_Q4G64) return DKV_ERR_UNSUPPORTED;
  if (K->format == DKV_KV_PAGED) {
    // K and V share one block table; an item's blocks fit the page list
    if (K->block_table != V->block_table || K->block_table_stride != V->block_table_stride ||
        K->num_blocks != V->num_blocks)
      return DKV_ERR_SHAPE;
    if (L.pages_per_chunk > dkv::kMaxSelectList) return DKV_ERR_UNSUPPORTED;
  }
  if (out_dtype != DKV_FP32 && out_dtype != DKV_BF16 && out_dtype != DKV_FP16)
    return DKV_ERR_DTYPE;
  if (!L.ok) return DKV_ERR_UNSUPPORTED;
  if (workspace == nullptr) return DKV_ERR_WORKSPACE;
  if (!aligned16(workspace)) return DKV_ERR_ALIGN;
  if (workspace_bytes < L.total) return DKV_ERR_WORKSPACE;
  (void)top_k;
  return DKV_OK;
}

static dkv::Q4View q4_view(const dkv_kv* kv) {
  dkv::Q4View v{};
  v.codes = static_cast<const uint8_t*>(kv->data);
  v.gmin = static_cast<const __half*>(kv->gmin);
  v.gmax = static_cast<const __half*>(kv->gmax);
  v.sb = kv->stride_b;
  v.sh = kv->stride_h;
  v.gsb = kv->gstride_b;
  v.gsh = kv->gstride_h;
  return v;
}

// Tensor maps for a dense cache; a 4-bit cache is described by Q4 views instead.
static bool cache_views(const dkv_params* p, const dkv_kv* K, const dkv_kv* V, CUtensorMap* mk,
                        CUtensorMap* mv, dkv::AttnArgs* a) {
  if (K->format == DKV_KV_Q4G64) {
    memset(mk, 0, sizeof *mk);
    memset(mv, 0, sizeof *mv);
    a->k4 = q4_view(K);
    a->v4 = q4_view(V);
    return true;
  }
  if (K->format == DKV_KV_PAGED) {
    a->bt = K->block_table;
    a->bts = K->block_table_stride;
    a->nblocks = K->num_blocks;
  }
  return encode_page_map(mk, p, K) && encode_page_map(mv, p, V);
}

static dkv::AttnArgs attn_args(const dkv_params* p, const void* q, const WsLayout& L,
                               uint8_t* ws) {
  dkv::AttnArgs a{};
  a.q = q;
  a.q_sb = p->q_stride_b;
  a.q_sh = p->q_stride_h;
  a.B = p->batch;
  a.Hq = p->num_q_heads;
  a.Hkv = p->num_kv_heads;
  a.G = p->num_q_heads / p->num_kv_heads;
  a.N = p->seq_len;
  a.P = static_cast<int>(ceil_div(p->seq_len, dkv::kPage));  // cache pages
  a.scale_log2 = p->scale * 1.4426950408889634f;
  a.pages_per_chunk = L.pages_per_chunk;
  a.n_chunks = L.n_chunks;
  a.n_items = static_cast<int>(L.n_items);
  a.part_ml = reinterpret_cast<float*>(ws + L.part_ml);
  a.part_o = reinterpret_cast<float*>(ws + L.part_o);
  a.work_counter = reinterpret_cast<uint32_t*>(ws + L.counter);
  a.exit_counter = reinterpret_cast<uint32_t*>(ws + L.exit_counter);
  a.status = reinterpret_cast<uint32_t*>(ws + L.status);
  a.wait_limit_ns = (p->flags & DKV_FLAG_FORCE_TIMEOUT) ? 0 : kWaitLimitNs;
  a.lens = p->seq_lens;
  return a;
}

// Persistent attention over all work items, then the split-K merge into out.
static dkv_status run_attention(const dkv_params* p, const dkv::AttnArgs& a, bool sparse,
                                bool f16, const CUtensorMap& mk, const CUtensorMap& mv,
                                void* out, int32_t out_dtype, cudaStream_t s) {
  // (sparse: a.union_count tells the merge how many chunks of a unit hold pages)
  const int sms = current_sm_count();
  if (sms <= 0) return DKV_ERR_CUDA;
  const bool q4 = a.k4.codes != nullptr;
  dkv::AttnArgs ao = a;
  ao.out = out;
  ao.out_dtype = out_code(out_dtype);
  ao.o_sb = p->o_stride_b;
  ao.o_sh = p->o_stride_h;
  dkv_status st = cuda_status(
      q4 ? dkv::launch_attn_q4(p->head_dim, sparse, ao, sms, s)
         : dkv::launch_attn(p->head_dim, f16, sparse, ao, mk, mv, sms, s));
  if (st != DKV_OK) return st;
  if (q4 && sparse && a.n_chunks == 1) return DKV_OK;  // the attention wrote out itself
  dkv::MergeArgs m{};
  m.part_ml = a.part_ml;
  m.part_o = a.part_o;
  m.n_chunks = a.n_chunks;
  m.Hq = p->num_q_heads;
  m.out = out;
  m.out_dtype = out_code(out_dtype);
  m.o_sb = p->o_stride_b;
  m.o_sh = p->o_stride_h;
  m.union_count = sparse ? a.union_count : nullptr;
  m.pages_per_chunk = a.pages_per_chunk;
  m.G = a.G;
  m.Hkv = a.Hkv;
  m.lens = a.lens;
  m.N = a.N;
  return cuda_status(dkv::launch_merge(p->head_dim, m, p->batch * p->num_q_heads, s));
}

dkv_status dkv_decode_attn_full(const dkv_params* p, const void* q, const dkv_kv* K,
                                const dkv_kv* V, void* out, int32_t out_dtype,
                                void* workspace, size_t workspace_bytes, void* stream) {
  dkv_status st = check_params(p);
  if (st != DKV_OK) return st;
  const WsLayout L = layout_for(*p, 0);
  if ((st = attn_common(p, q, K, V, out, out_dtype, workspace, workspace_bytes, 0, L)) != DKV_OK)
    return st;
  CUtensorMap mk, mv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  dkv::AttnArgs a = attn_args(p, q, L, ws);
  if (!cache_views(p, K, V, &mk, &mv, &a)) return DKV_ERR_CUDA;
  return run_attention(p, a, false, K->dtype == DKV_FP16, mk, mv, out, out_dtype, s);
}

// 8-bit page metadata (device pointers), for the select path that scores it.
struct Meta8Ptrs {
  const uint8_t* code_min;
  const uint8_t* code_max;
  const float* lo;
  const float* step;
};

// Cross-step reuse state of dkv_decode_attn_select_hot: a 256-byte header
// (u64 pages gathered, u64 of them gathered at the previous step) and the
// per-page stamps [B, Hkv, ceil(N / 16)] u32.
struct HotArgs {
  void* state;
  size_t bytes;
  int32_t step;
};

static size_t hot_stamp_pages(const dkv_params& p) {
  return static_cast<size_t>(ceil_div(p.seq_len, dkv::kPage));
}

static size_t hot_bytes(const dkv_params& p) {
  return kAlign + align_up(sizeof(uint32_t) * static_cast<size_t>(p.batch) * p.num_kv_heads *
                           hot_stamp_pages(p));
}

// The page-sparse call over 16-bit metadata (m8 == nullptr) or 8-bit metadata,
// with cross-step reuse when hot != nullptr.
static dkv_status select_impl(const dkv_params* p, const void* q, const dkv_kv* K,
                              const dkv_kv* V, const void* meta_min, const void* meta_max,
                              const Meta8Ptrs* m8, int32_t top_k, void* out, int32_t out_dtype,
                              int32_t* selected, void* workspace, size_t workspace_bytes,
                              void* stream, const HotArgs* hot = nullptr) {
  dkv_status st = check_params(p);
  if (st != DKV_OK) return st;
  if (top_k < 1) return DKV_ERR_SHAPE;
  const WsLayout L = layout_for(*p, top_k);
  if ((st = attn_common(p, q, K, V, out, out_dtype, workspace, workspace_bytes, top_k, L)) !=
      DKV_OK)
    return st;
  if (hot != nullptr) {
    if (K->format == DKV_KV_Q4G64) return DKV_ERR_UNSUPPORTED;
    if (hot->state == nullptr) return DKV_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(hot->state) & 15u) return DKV_ERR_ALIGN;
    if (hot->bytes < hot_bytes(*p)) return DKV_ERR_WORKSPACE;
    if (hot->step < 1) return DKV_ERR_SHAPE;
  }
  if (m8 == nullptr) {
    if (meta_min == nullptr || meta_max == nullptr) return DKV_ERR_NULL;
    if (!aligned16(meta_min) || !aligned16(meta_max)) return DKV_ERR_ALIGN;
  } else {
    if (m8->code_min == nullptr || m8->code_max == nullptr || m8->lo == nullptr ||
        m8->step == nullptr)
      return DKV_ERR_NULL;
    if (!aligned16(m8->code_min) || !aligned16(m8->code_max) ||
        (reinterpret_cast<uintptr_t>(m8->lo) & 3u) || (reinterpret_cast<uintptr_t>(m8->step) & 3u))
      return DKV_ERR_ALIGN;
  }
  if (selected != nullptr && (reinterpret_cast<uintptr_t>(selected) & 3u)) return DKV_ERR_ALIGN;
  CUtensorMap mk, mv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int P = static_cast<int>(ceil_div(p->seq_len, p->page_size));
  const int G = p->num_q_heads / p->num_kv_heads;
  const bool f16 = K->dtype == DKV_FP16;
  const bool group = (p->flags & DKV_FLAG_GROUP_SELECT) != 0;

  int32_t* sel = selected != nullptr ? selected : reinterpret_cast<int32_t*>(ws + L.selected);
  int2* ulist = reinterpret_cast<int2*>(ws + L.union_list);
  int* ucount = reinterpret_cast<int*>(ws + L.union_count);

  dkv::AttnArgs a = attn_args(p, q, L, ws);
  if (!cache_views(p, K, V, &mk, &mv, &a)) return DKV_ERR_CUDA;
  a.sub_log2 = p->page_size == 4 ? 2 : (p->page_size == 8 ? 1 : 0);
  if (hot != nullptr) {
    uint8_t* hs = static_cast<uint8_t*>(hot->state);
    a.hot_stats = reinterpret_cast<unsigned long long*>(hs);
    a.hot_stamp = reinterpret_cast<uint32_t*>(hs + kAlign);
    a.hot_pages = static_cast<int>(hot_stamp_pages(*p));
    a.hot_step = static_cast<uint32_t>(hot->step);
    // Keep as many units' pages as half the L2 holds, at the union's upper
    // bound: G * kk selection pages, each S / 16 cache pages (or one), per unit.
    int dev = 0, l2 = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return DKV_ERR_CUDA;
    const int64_t sel_pages = static_cast<int64_t>(G) * L.kk *
                              (p->page_size > dkv::kPage ? p->page_size / dkv::kPage : 1);
    const int64_t pages = std::min<int64_t>(sel_pages, hot_stamp_pages(*p));
    const int64_t unit_bytes = pages * 2 * dkv::kPage * p->head_dim * 2;
    a.hot_keep_units = static_cast<int>(std::min<int64_t>(
        static_cast<int64_t>(p->batch) * p->num_kv_heads, (l2 / 2) / std::max<int64_t>(unit_bytes, 1)));
  }
  a.union_list = ulist;
  a.union_count = ucount;
  a.union_stride = L.union_stride;

  if (p->page_size >= dkv::kPage && P >= kUnitSelectMinP && P <= dkv::kUnitMaxP &&
      dkv::unit_select_smem(p->head_dim, m8 != nullptr, G, P) <=
          static_cast<size_t>(kUnitSelectSmemLimit)) {
    // Contexts of 256 pages and more: a persistent grid of selection CTAs
    // takes the (batch, kv head) units in turn; each unit's metadata (16-bit,
    // or 8-bit codes) is scored, each head's top-K selected and the union
    // list built in one CTA.  (Shorter contexts have too little metadata per
    // CTA to hide the selection's latency; the three kernels below spread the
    // same work wider.)
    dkv::UnitSelectArgs ua{};
    ua.q = q;
    ua.q_sb = p->q_stride_b;
    ua.q_sh = p->q_stride_h;
    ua.meta_min = meta_min;
    ua.meta_max = meta_max;
    if (m8 != nullptr) {
      ua.lo = m8->lo;
      ua.step = m8->step;
    }
    ua.B = p->batch;
    ua.Hq = p->num_q_heads;
    ua.Hkv = p->num_kv_heads;
    ua.G = G;
    ua.P = P;
    ua.kk = L.kk;
    ua.selected = sel;
    ua.union_list = ulist;
    ua.union_count = ucount;
    ua.union_stride = L.union_stride;
    ua.group = group ? 1 : 0;
    ua.lens = p->seq_lens;
    ua.N = p->seq_len;
    ua.S = p->page_size;
    ua.status = a.status;
    ua.wait_limit_ns = a.wait_limit_ns;
    ua.num_sms = current_sm_count();
    // the attention takes each unit's items once its union is written
    ua.unit_ready = reinterpret_cast<uint32_t*>(ws + L.unit_ready);
    a.unit_ready = ua.unit_ready;
    CUtensorMap mmx, mmn;
    const bool maps_ok =
        m8 != nullptr
            ? encode_code_map(&mmx, p, m8->code_max, 64) && encode_code_map(&mmn, p, m8->code_min, 64)
            : encode_meta_map(&mmx, p, meta_max, f16, 64) && encode_meta_map(&mmn, p, meta_min, f16, 64);
    if (!maps_ok) return DKV_ERR_CUDA;
    if ((st = cuda_status(dkv::launch_unit_select(p->head_dim, f16, m8 != nullptr, ua, mmx, mmn,
                                                  s))) != DKV_OK)
      return st;
    return run_attention(p, a, true, f16, mk, mv, out, out_dtype, s);
  }

  // Otherwise: bound scores, per-head top-K and the group's page union as
  // three kernels.
  {
    dkv::ScoreArgs sa{};
    sa.q = q;
    sa.q_sb = p->q_stride_b;
    sa.q_sh = p->q_stride_h;
    sa.meta_min = meta_min;
    sa.meta_max = meta_max;
    sa.B = p->batch;
    sa.Hq = p->num_q_heads;
    sa.Hkv = p->num_kv_heads;
    sa.G = G;
    sa.P = P;
    sa.scores = reinterpret_cast<float*>(ws + L.scores);
    if (m8 == nullptr) {
      if ((st = cuda_status(dkv::launch_score(p->head_dim, f16, sa, s))) != DKV_OK) return st;
    } else {
      dkv::Score8Args s8{};
      s8.q = q;
      s8.q_sb = p->q_stride_b;
      s8.q_sh = p->q_stride_h;
      s8.code_min = m8->code_min;
      s8.code_max = m8->code_max;
      s8.lo = m8->lo;
      s8.step = m8->step;
      s8.B = p->batch;
      s8.Hq = p->num_q_heads;
      s8.Hkv = p->num_kv_heads;
      s8.G = G;
      s8.P = P;
      s8.scores = sa.scores;
      if ((st = cuda_status(dkv::launch_score8(p->head_dim, f16, s8, s))) != DKV_OK) return st;
    }
    dkv::TopkArgs ta{};
    ta.scores = sa.scores;
    ta.rows = p->batch * p->num_q_heads;
    ta.P = P;
    ta.kk = L.kk;
    ta.selected = sel;
    ta.bitmaps = reinterpret_cast<uint32_t*>(ws + L.bitmaps);
    ta.W32 = L.W32;
    ta.Hq = p->num_q_heads;
    ta.group = group ? G : 1;
    ta.lens = p->seq_lens;
    ta.N = p->seq_len;
    ta.S = p->page_size;
    // one query head per kv head at 16-token pages: the rows are the unions
    const bool row_unions = G == 1 && p->page_size == dkv::kPage;
    if (row_unions) {
      ta.union_list = ulist;
      ta.union_count = ucount;
      ta.union_stride = L.union_stride;
    }
    if ((st = cuda_status(dkv::launch_topk(ta, s))) != DKV_OK) return st;
    if (row_unions) return run_attention(p, a, true, f16, mk, mv, out, out_dtype, s);
    dkv::UnionArgs ua{};
    ua.bitmaps = ta.bitmaps;
    ua.Hq = p->num_q_heads;
    ua.Hkv = p->num_kv_heads;
    ua.G = G;
    ua.P = P;
    ua.W32 = L.W32;
    ua.union_list = ulist;
    ua.union_count = ucount;
    ua.union_stride = L.union_stride;
    ua.lens = p->seq_lens;
    ua.N = p->seq_len;
    ua.S = p->page_size;
    if ((st = cuda_status(dkv::launch_union(ua, p->batch * p->num_kv_heads, s))) != DKV_OK)
      return st;
  }

  return run_attention(p, a, true, f16, mk, mv, out, out_dtype, s);
}

size_t dkv_hot_state_bytes(const dkv_params* p) {
  if (check_params(p) != DKV_OK) return 0;
  return hot_bytes(*p);
}

dkv_status dkv_decode_attn_select_hot(const dkv_params* p, const void* q, const dkv_kv* K,
                                      const dkv_kv* V, const void* meta_min,
                                      const void* meta_max, int32_t top_k, void* out,
                                      int32_t out_dtype, int32_t* selected, void* hot_state,
                                      size_t hot_state_bytes, int32_t step, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  const HotArgs hot{hot_state, hot_state_bytes, step};
  return select_impl(p, q, K, V, meta_min, meta_max, nullptr, top_k, out, out_dtype, selected,
                     workspace, workspace_bytes, stream, &hot);
}

dkv_status dkv_decode_attn_select(const dkv_params* p, const void* q, const dkv_kv* K,
                                  const dkv_kv* V, const void* meta_min,
                                  const void* meta_max, int32_t top_k, void* out,
                                  int32_t out_dtype, int32_t* selected, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return select_impl(p, q, K, V, meta_min, meta_max, nullptr, top_k, out, out_dtype, selected,
                     workspace, workspace_bytes, stream);
}

dkv_status dkv_decode_attn_select_meta8(const dkv_params* p, const void* q, const dkv_kv* K,
                                        const dkv_kv* V, const void* code_min,
                                        const void* code_max, const void* lo, const void* step,
                                        int32_t top_k, void* out, int32_t out_dtype,
                                        int32_t* selected, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  const Meta8Ptrs m8{static_cast<const uint8_t*>(code_min), static_cast<const uint8_t*>(code_max),
                     static_cast<const float*>(lo), static_cast<const float*>(step)};
  return select_impl(p, q, K, V, nullptr, nullptr, &m8, top_k, out, out_dtype, selected,
                     workspace, workspace_bytes, stream);
}

dkv_status dkv_kv_meta8_build(const dkv_params* p, const void* meta_min, const void* meta_max,
                              int32_t meta_dtype, void* code_min, void* code_max, void* lo,
                              void* step, void* stream) {
  dkv_status st = check_params(p);
  if (st != DKV_OK) return st;
  if (meta_dtype != DKV_BF16 && meta_dtype != DKV_FP16) return DKV_ERR_DTYPE;
  if (meta_min == nullptr || meta_max == nullptr || code_min == nullptr || code_max == nullptr ||
      lo == nullptr || step == nullptr)
    return DKV_ERR_NULL;
  if (!aligned16(meta_min) || !aligned16(meta_max) || !aligned16(code_min) ||
      !aligned16(code_max) || (reinterpret_cast<uintptr_t>(lo) & 3u) ||
      (reinterpret_cast<uintptr_t>(step) & 3u))
    return DKV_ERR_ALIGN;
  const int64_t pages =
      static_cast<int64_t>(p->batch) * p->num_kv_heads * ceil_div(p->seq_len, p->page_size);
  if (pages >= (static_cast<int64_t>(1) << 31)) return DKV_ERR_UNSUPPORTED;
  dkv::Meta8Args a{};
  a.meta_min = static_cast<const uint16_t*>(meta_min);
  a.meta_max = static_cast<const uint16_t*>(meta_max);
  a.code_min = static_cast<uint8_t*>(code_min);
  a.code_max = static_cast<uint8_t*>(code_max);
  a.lo = static_cast<float*>(lo);
  a.step = static_cast<float*>(step);
  a.B = p->batch;
  a.Hkv = p->num_kv_heads;
  a.P = static_cast<int>(ceil_div(p->seq_len, p->page_size));
  a.d = p->head_dim;
  a.S = p->page_size;
  a.N = p->seq_len;
  a.lens = p->seq_lens;
  return cuda_status(
      dkv::launch_meta8(meta_dtype == DKV_FP16, a, static_cast<cudaStream_t>(stream)));
}

dkv_status dkv_kv_quant4(int64_t rows, int32_t d, const void* x, void* codes, void* gmin,
                         void* gmax, void* stream) {
  if (x == nullptr || codes == nullptr || gmin == nullptr || gmax == nullptr) return DKV_ERR_NULL;
  if (rows < 0 || d < 64 || d % 64 != 0) return DKV_ERR_SHAPE;
  if (rows * (d / 64) * 8 > (static_cast<int64_t>(1) << 40)) return DKV_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(gmin) & 1u) ||
      (reinterpret_cast<uintptr_t>(gmax) & 1u))
    return DKV_ERR_ALIGN;
  if (rows == 0) return DKV_OK;
  return cuda_status(
      dkv::launch_quant4(rows, d, x, codes, gmin, gmax, static_cast<cudaStream_t>(stream)));
}

dkv_status dkv_kv_dequant4(int64_t rows, int32_t d, const void* codes, const void* gmin,
                           const void* gmax, void* x, void* stream) {
  if (x == nullptr || codes == nullptr || gmin == nullptr || gmax == nullptr) return DKV_ERR_NULL;
  if (rows < 0 || d < 64 || d % 64 != 0) return DKV_ERR_SHAPE;
  if (rows * (d / 64) * 8 > (static_cast<int64_t>(1) << 40)) return DKV_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(gmin) & 1u) ||
      (reinterpret_cast<uintptr_t>(gmax) & 1u))
    return DKV_ERR_ALIGN;
  if (rows == 0) return DKV_OK;
  return cuda_status(
      dkv::launch_dequant4(rows, d, codes, gmin, gmax, x, static_cast<cudaStream_t>(stream)));
}

// Token-level top-K workspace: header | scores [rows, N] fp32 | selected
// [rows, kk] int32 | the top-K's bitmaps [rows, ceil(N / 32)] u32.
static size_t token_layout(const dkv_params* p, int top_k, size_t* scores, size_t* sel,
                           size_t* bits) {
  const int64_t rows = static_cast<int64_t>(p->batch) * p->num_q_heads;
  const int64_t N = p->seq_len;
  const int64_t kk = top_k < N ? top_k : N;
  size_t off = DKV_WORKSPACE_HEADER_BYTES;
  *scores = off;
  off = align_up(off + sizeof(float) * rows * N);
  *sel = off;
  off = align_up(off + sizeof(int32_t) * rows * kk);
  *bits = off;
  off = align_up(off + sizeof(uint32_t) * rows * ceil_div(N, 32));
  return off;
}

size_t dkv_workspace_bytes_tokens(const dkv_params* p, int32_t top_k) {
  if (check_params(p) != DKV_OK || top_k < 1) return 0;
  size_t a, b, c;
  return token_layout(p, top_k, &a, &b, &c);
}

dkv_status dkv_decode_attn_topk_tokens(const dkv_params* p, const void* q, const dkv_kv* K,
                                       const dkv_kv* V, int32_t top_k, void* out,
                                       int32_t out_dtype, int32_t* selected, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  dkv_status st = check_params(p);
  if (st != DKV_OK) return st;
  if (top_k < 1) return DKV_ERR_SHAPE;
  if ((st = check_query_out(p, q, out)) != DKV_OK) return st;
  if ((st = check_kv(p, K)) != DKV_OK) return st;
  if ((st = check_kv(p, V)) != DKV_OK) return st;
  if (K->format != DKV_KV_DENSE || V->format != DKV_KV_DENSE || K->dtype != V->dtype)
    return DKV_ERR_DTYPE;
  const int d = p->head_dim;
  const int64_t N = p->seq_len;
  // the score pass reads K as one contiguous row per token
  if (K->stride_h != N * d || K->stride_b != static_cast<int64_t>(p->num_kv_heads) * N * d)
    return DKV_ERR_UNSUPPORTED;
  if (p->seq_lens != nullptr) return DKV_ERR_UNSUPPORTED;
  if (out_dtype != DKV_FP32 && out_dtype != DKV_BF16 && out_dtype != DKV_FP16)
    return DKV_ERR_DTYPE;
  if (selected != nullptr && (reinterpret_cast<uintptr_t>(selected) & 3u)) return DKV_ERR_ALIGN;
  size_t o_scores, o_sel, o_bits;
  const size_t need = token_layout(p, top_k, &o_scores, &o_sel, &o_bits);
  if (workspace == nullptr) return DKV_ERR_WORKSPACE;
  if (!aligned16(workspace)) return DKV_ERR_ALIGN;
  if (workspace_bytes < need) return DKV_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool f16 = K->dtype == DKV_FP16;
  const int G = p->num_q_heads / p->num_kv_heads;
  const int rows = p->batch * p->num_q_heads;
  const int kk = static_cast<int>(top_k < N ? top_k : N);
  float* scores = reinterpret_cast<float*>(ws + o_scores);
  int32_t* sel = selected != nullptr ? selected : reinterpret_cast<int32_t*>(ws + o_sel);

  // exact scores: the bound score over single-token pages (m = M = k)
  dkv::ScoreArgs sa{};
  sa.q = q;
  sa.q_sb = p->q_stride_b;
  sa.q_sh = p->q_stride_h;
  sa.meta_min = K->data;
  sa.meta_max = K->data;
  sa.B = p->batch;
  sa.Hq = p->num_q_heads;
  sa.Hkv = p->num_kv_heads;
  sa.G = G;
  sa.P = static_cast<int>(N);
  sa.scores = scores;
  sa.exact = 1;
  if ((st = cuda_status(dkv::launch_score(d, f16, sa, s))) != DKV_OK) return st;
  // the top-K tokens, ties to the lower index, ascending
  dkv::TopkArgs ta{};
  ta.scores = scores;
  ta.rows = rows;
  ta.P = static_cast<int>(N);
  ta.kk = kk;
  ta.Hq = p->num_q_heads;
  ta.group = 1;
  ta.N = static_cast<int>(N);
  ta.S = 1;
  ta.selected = sel;
  ta.bitmaps = reinterpret_cast<uint32_t*>(ws + o_bits);
  ta.W32 = static_cast<int>(ceil_div(N, 32));
  if ((st = cuda_status(dkv::launch_topk(ta, s))) != DKV_OK) return st;
  dkv::TokenAttnArgs aa{};
  aa.scores = scores;
  aa.selected = sel;
  aa.kk = kk;
  aa.N = static_cast<int>(N);
  aa.Hq = p->num_q_heads;
  aa.G = G;
  aa.v = V->data;
  aa.v_sb = V->stride_b;
  aa.v_sh = V->stride_h;
  aa.v_st = d;
  aa.scale_log2 = p->scale * 1.4426950408889634f;
  aa.out = out;
  aa.out_dtype = out_code(out_dtype);
  aa.o_sb = p->o_stride_b;
  aa.o_sh = p->o_stride_h;
  return cuda_status(dkv::launch_token_attn(d, f16, aa, rows, s));
}

dkv_status dkv_read_device_status(void* workspace, void* stream) {
  if (workspace == nullptr) return DKV_ERR_NULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DKV_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof v, s) != cudaSuccess) return DKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DKV_ERR_CUDA;
  return static_cast<dkv_status>(v);
}

dkv_status dkv_attn_ctas_per_sm(int32_t head_dim, int32_t dtype, int32_t format, int32_t sparse,
                                int32_t* ctas_per_sm) {
  if (ctas_per_sm == nullptr) return DKV_ERR_NULL;
  if (head_dim != 64 && head_dim != 128) return DKV_ERR_UNSUPPORTED;
  if (format == DKV_KV_DENSE ? (dtype != DKV_BF16 && dtype != DKV_FP16)
                             : (format != DKV_KV_Q4G64 || dtype != DKV_FP16))
    return DKV_ERR_UNSUPPORTED;
  int n = 0;
  const cudaError_t e = dkv::attn_ctas_per_sm(head_dim, dtype == DKV_FP16, sparse != 0,
                                              format == DKV_KV_Q4G64, &n);
  if (e != cudaSuccess) return DKV_ERR_CUDA;
  *ctas_per_sm = n;
  return DKV_OK;
}

const char* dkv_status_string(int32_t status) {
  switch (status) {
    case DKV_OK: return "ok";
    case DKV_ERR_NULL: return "a required pointer is NULL";
    case DKV_ERR_SHAPE: return "a size or stride is out of range";
    case DKV_ERR_ALIGN: return "a pointer or stride is not 16-byte aligned";
    case DKV_ERR_DTYPE: return "unsupported dtype or format combination";
    case DKV_ERR_UNSUPPORTED: return "head_dim, page_size or query group outside the kernels";
    case DKV_ERR_WORKSPACE: return "workspace missing or too small";
    case DKV_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case DKV_ERR_DEVICE_TIMEOUT: return "device: a bounded wait expired";
    case DKV_ERR_DEVICE_CHECK: return "device: an in-kernel check failed";
    default: return "unknown status";
  }
}

}  // extern "C"

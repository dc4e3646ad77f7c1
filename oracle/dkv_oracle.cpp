// dkv_oracle.cpp -- the slow, plain CPU oracle for single-token decode attention
// over a paged KV cache.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
// this file: only the test suite, the smoke check and the benchmark's CPU
// baseline leg use it.  It shares no source, header, table or helper with the
// CUDA library; it is written from the pages' definitions alone:
//
//   [TS]  "TinyServe: Query-Aware Cache Selection for Efficient LLM Serving"
//         - 结构化内存布局 (pages of S tokens, P = ceil(t/S))
//         - 相关性函数实例化 (page metadata phi = (m_j, M_j), bound score r)
//         - 问题公式化定义 (S_t = TopK_j r, |S_t| = K; SparseAttn over S_t)
//         - 标准Transformer解码层的注意力计算 (Attn(q_t, K, V))
//         - Algorithm 1 "Fused Query-Aware Sparse Attention Kernel", steps 1-4
//   [HI]  "论文阅读：HeadInfer" - 核心 idea (A^(h) = Softmax(Q K^T / sqrt(d_k)) V,
//         heads independent, head-by-head evaluation identical to all heads)
//   [FG]  "FlexGen: High-Throughput Generative Inference of Large Language
//         Models with a Single GPU" (解读) - 4-bit 近似方法 (groups of 64,
//         per-group min/max, 4-bit integers, dequantised to FP16; KV grouped
//         along the hidden dimension)
//
// Arithmetic: every accumulation is in double.  The 4-bit format is a storage
// format, not an accumulation, so it is defined by the exact IEEE fp32/fp16
// operations listed at oracle_quant4 / oracle_dequant4; this file must be
// compiled with -ffp-contract=off so that no multiply-add is fused behind our
// back.  Readings of points the pages leave open are stated where they apply.
//
// Layouts (row-major, innermost last):
//   q      [B, Hq, d]            16-bit float bits (bf16 or fp16)
//   K, V   [B, Hkv, N, d]        16-bit float bits
//   meta   [B, Hkv, P, d]        16-bit float bits, P = ceil(N / S)
//   meta8  codes [B, Hkv, P, d] u8 (min and max); lo, step [B, Hkv, P] fp32
//   codes  [rows, d/2]           u8, channel 2i in the low nibble of byte i
//   gmin, gmax [rows, d/64]      fp16 bits
//   scores [B, Hq, P]            double
//   sel    [B, Hq, kk]           int32, kk = min(K, P), ascending page indices
//   out    [B, Hq, d]            double

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <numeric>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// 16-bit float formats, decoded from their IEEE / bfloat16 definitions.
// ---------------------------------------------------------------------------

// bfloat16: the upper 16 bits of an IEEE binary32.
double bf16_value(uint16_t h) {
  uint32_t w = static_cast<uint32_t>(h) << 16;
  float f;
  std::memcpy(&f, &w, sizeof f);
  return static_cast<double>(f);
}

// IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
double fp16_value(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1f;
  const int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(f), -24);  // zero or subnormal
  } else if (e == 31) {
    v = f ? std::nan("") : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(1024 + f), e - 25);
  }
  return sign ? -v : v;
}

double value16(uint16_t h, int is_fp16) { return is_fp16 ? fp16_value(h) : bf16_value(h); }

// Round a double to the nearest IEEE binary16, ties to even, overflow to inf.
// The input is taken as an exact real number: this is the single rounding the
// 4-bit format's dequantisation performs.
uint16_t fp16_round(double x) {
  if (std::isnan(x)) return 0x7e00;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  if (a == 0.0) return sign;
  // Quantum of the binade containing a (subnormals share the 2^-24 quantum).
  int e2;
  std::frexp(a, &e2);           // a = m * 2^e2, m in [0.5, 1)
  int exp_unbiased = e2 - 1;    // a in [2^exp, 2^(exp+1))
  if (exp_unbiased < -14) exp_unbiased = -14;
  const double quantum = std::ldexp(1.0, exp_unbiased - 10);
  const double n = std::nearbyint(a / quantum);  // FE_TONEAREST: ties to even
  const double r = n * quantum;                  // exact
  if (r >= 65536.0) return sign | 0x7c00;        // rounds past the largest finite
  // Encode the exactly representable r.
  if (r < std::ldexp(1.0, -14)) {
    return sign | static_cast<uint16_t>(r / std::ldexp(1.0, -24));
  }
  int e3;
  std::frexp(r, &e3);
  const int ex = e3 - 1;  // r in [2^ex, 2^(ex+1))
  const uint16_t frac = static_cast<uint16_t>(r / std::ldexp(1.0, ex - 10) - 1024.0);
  return sign | static_cast<uint16_t>((ex + 15) << 10) | frac;
}

// Total order on 16-bit float bit patterns: numeric order, with -0 below +0.
// Min/max of stored values then always returns one of the stored bit patterns.
// (NaN inputs are outside the supported domain.)
bool less16(uint16_t a, uint16_t b, int is_fp16) {
  const double va = value16(a, is_fp16), vb = value16(b, is_fp16);
  if (va != vb) return va < vb;
  return (a & 0x8000) && !(b & 0x8000);
}

// Run f(unit) for unit in [0, n) on `threads` std::threads (0 = all cores).
int g_threads = 0;
void parallel_for(int64_t n, const std::function<void(int64_t)>& f) {
  int t = g_threads > 0 ? g_threads : static_cast<int>(std::thread::hardware_concurrency());
  if (t < 1) t = 1;
  if (n < t) t = static_cast<int>(std::max<int64_t>(n, 1));
  if (t == 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> pool;
  for (int i = 0; i < t; ++i) {
    pool.emplace_back([&] {
      for (int64_t u = next.fetch_add(1); u < n; u = next.fetch_add(1)) f(u);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Threads used by every oracle routine (0 = std::thread::hardware_concurrency).
void oracle_set_threads(int n) { g_threads = n; }
int oracle_get_threads(void) {
  return g_threads > 0 ? g_threads : static_cast<int>(std::thread::hardware_concurrency());
}

// Format helpers, exposed so the tests can pin them against independent
// library conversions.
double oracle_value16(uint16_t h, int is_fp16) { return value16(h, is_fp16); }
uint16_t oracle_fp16_round(double x) { return fp16_round(x); }

// ---------------------------------------------------------------------------
// Page metadata  [TS 结构化内存布局, 相关性函数实例化]
// The keys of one (batch, kv-head) are split into P = ceil(N/S) pages of S
// consecutive tokens (the last page may be ragged).  phi(K_j) = (m_j, M_j):
// the channel-wise minimum and maximum over the page's tokens.
// ---------------------------------------------------------------------------
void oracle_meta(int B, int Hkv, int N, int d, int S, int is_fp16, const uint16_t* K,
                 uint16_t* meta_min, uint16_t* meta_max) {
  const int P = (N + S - 1) / S;
  parallel_for(static_cast<int64_t>(B) * Hkv, [&](int64_t bh) {
    const uint16_t* Kbh = K + bh * static_cast<int64_t>(N) * d;
    uint16_t* mn = meta_min + bh * static_cast<int64_t>(P) * d;
    uint16_t* mx = meta_max + bh * static_cast<int64_t>(P) * d;
    for (int j = 0; j < P; ++j) {
      const int t0 = j * S, t1 = std::min(N, (j + 1) * S);
      for (int i = 0; i < d; ++i) {
        uint16_t lo = Kbh[static_cast<int64_t>(t0) * d + i], hi = lo;
        for (int t = t0 + 1; t < t1; ++t) {
          const uint16_t k = Kbh[static_cast<int64_t>(t) * d + i];
          if (less16(k, lo, is_fp16)) lo = k;
          if (less16(hi, k, is_fp16)) hi = k;
        }
        mn[static_cast<int64_t>(j) * d + i] = lo;
        mx[static_cast<int64_t>(j) * d + i] = hi;
      }
    }
  });
}

// ---------------------------------------------------------------------------
// Bound score  [TS 相关性函数实例化; Algorithm 1 step 1]
//   r(q, phi_j) = sum_i ( q_i >= 0 ? q_i * M_{j,i} : q_i * m_{j,i} )
// for every (batch, q-head, page); q-head h reads kv-head h / (Hq/Hkv).
// ---------------------------------------------------------------------------
void oracle_scores(int B, int Hq, int Hkv, int P, int d, int is_fp16, const uint16_t* q,
                   const uint16_t* meta_min, const uint16_t* meta_max, double* scores) {
  const int G = Hq / Hkv;
  parallel_for(static_cast<int64_t>(B) * Hq, [&](int64_t bh) {
    const int64_t b = bh / Hq, h = bh % Hq, kvh = h / G;
    const uint16_t* qv = q + bh * d;
    const uint16_t* mn = meta_min + (b * Hkv + kvh) * static_cast<int64_t>(P) * d;
    const uint16_t* mx = meta_max + (b * Hkv + kvh) * static_cast<int64_t>(P) * d;
    for (int j = 0; j < P; ++j) {
      double s = 0.0;
      for (int i = 0; i < d; ++i) {
        const double qi = value16(qv[i], is_fp16);
        if (qi >= 0.0) {
          s += qi * value16(mx[static_cast<int64_t>(j) * d + i], is_fp16);
        } else {
          s += qi * value16(mn[static_cast<int64_t>(j) * d + i], is_fp16);
        }
      }
      scores[bh * P + j] = s;
    }
  });
}

// ---------------------------------------------------------------------------
// 8-bit page metadata: a smaller phi that keeps r an upper bound
// [TS 相关性函数实例化; the metadata scan is the "lightweight" per-step term of
// the page's cost model].  The pages keep (m_j, M_j) at the keys' precision and
// print no compressed form; this one is the plainest that keeps the bound.  Per
// page j (one batch entry and kv head):
//   lo = min_i m_{j,i},  hi = max_i M_{j,i}        (a zero is stored as +0)
//   dec(c) = fma(c, step, lo)                      one fp32 rounding
//   step   = fp32(fp32(hi - lo) / 255), raised one ulp at a time until
//            dec(255) >= hi                        (0 when hi == lo)
//   cm_i   = the largest c in [0, 255] with dec(c) <= m_{j,i}
//   cM_i   = the smallest c in [0, 255] with dec(c) >= M_{j,i}
// dec is non-decreasing in c and dec(0) = lo, so both codes exist, and
// dec(cm_i) <= m_{j,i} <= k_i <= M_{j,i} <= dec(cM_i) for every key of the page:
// the score with dec(cm), dec(cM) in place of m, M bounds max_k q.k again.
// Metadata is finite (hi - lo finite).
// ---------------------------------------------------------------------------
float dec8(int c, float step, float lo) { return std::fmaf(static_cast<float>(c), step, lo); }

void oracle_meta8(int64_t pages, int d, int is_fp16, const uint16_t* meta_min,
                  const uint16_t* meta_max, uint8_t* code_min, uint8_t* code_max, float* lo_out,
                  float* step_out) {
  parallel_for(pages, [&](int64_t pg) {
    const uint16_t* mn = meta_min + pg * d;
    const uint16_t* mx = meta_max + pg * d;
    float lo = static_cast<float>(value16(mn[0], is_fp16));
    float hi = static_cast<float>(value16(mx[0], is_fp16));
    for (int i = 1; i < d; ++i) {
      lo = std::min(lo, static_cast<float>(value16(mn[i], is_fp16)));
      hi = std::max(hi, static_cast<float>(value16(mx[i], is_fp16)));
    }
    if (lo == 0.0f) lo = 0.0f;  // +0
    if (hi == 0.0f) hi = 0.0f;
    float step = 0.0f;
    if (hi > lo) {
      const float range = hi - lo;  // one fp32 rounding
      step = range / 255.0f;        // one fp32 rounding
      while (dec8(255, step, lo) < hi) step = std::nextafterf(step, INFINITY);
    }
    lo_out[pg] = lo;
    step_out[pg] = step;
    for (int i = 0; i < d; ++i) {
      const float m = static_cast<float>(value16(mn[i], is_fp16));
      const float M = static_cast<float>(value16(mx[i], is_fp16));
      int cm = 0, cM = 0;
      if (step > 0.0f) {
        // a first guess from the division, then the definitions decide
        const float em = (m - lo) / step, eM = (M - lo) / step;
        cm = em >= 255.0f ? 255 : (em >= 0.0f ? static_cast<int>(em) : 0);
        cM = eM >= 255.0f ? 255 : (eM >= 0.0f ? static_cast<int>(std::ceil(eM)) : 0);
        while (cm < 255 && dec8(cm + 1, step, lo) <= m) ++cm;
        while (cm > 0 && dec8(cm, step, lo) > m) --cm;
        while (cM > 0 && dec8(cM - 1, step, lo) >= M) --cM;
        while (cM < 255 && dec8(cM, step, lo) < M) ++cM;
      }
      code_min[pg * d + i] = static_cast<uint8_t>(cm);
      code_max[pg * d + i] = static_cast<uint8_t>(cM);
    }
  });
}

// The bound score over 8-bit metadata, in float64 over the decoded values:
//   r8(q, j) = sum_i ( q_i >= 0 ? q_i * dec(cM_{j,i}) : q_i * dec(cm_{j,i}) )
void oracle_scores8(int B, int Hq, int Hkv, int P, int d, int is_fp16, const uint16_t* q,
                    const uint8_t* code_min, const uint8_t* code_max, const float* lo,
                    const float* step, double* scores) {
  const int G = Hq / Hkv;
  parallel_for(static_cast<int64_t>(B) * Hq, [&](int64_t bh) {
    const int64_t b = bh / Hq, h = bh % Hq, kvh = h / G;
    const uint16_t* qv = q + bh * d;
    for (int j = 0; j < P; ++j) {
      const int64_t pg = (b * Hkv + kvh) * P + j;
      double s = 0.0;
      for (int i = 0; i < d; ++i) {
        const double qi = value16(qv[i], is_fp16);
        const uint8_t c = qi >= 0.0 ? code_max[pg * d + i] : code_min[pg * d + i];
        s += qi * static_cast<double>(dec8(c, step[pg], lo[pg]));
      }
      scores[bh * P + j] = s;
    }
  });
}

// ---------------------------------------------------------------------------
// Top-K page selection  [TS 问题公式化定义; Algorithm 1 step 2]
// S_t = the K pages with the largest score (K clamped to P).  Ties, which the
// pages leave open, go to the lower page index.  The result is returned in
// ascending page order.
// ---------------------------------------------------------------------------
void oracle_topk(int BH, int P, int K, const double* scores, int32_t* sel) {
  const int kk = std::min(K, P);
  parallel_for(BH, [&](int64_t bh) {
    const double* r = scores + bh * P;
    std::vector<int32_t> idx(P);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) {
      if (r[a] != r[b]) return r[a] > r[b];
      return a < b;
    });
    idx.resize(kk);
    std::sort(idx.begin(), idx.end());
    std::copy(idx.begin(), idx.end(), sel + bh * kk);
  });
}

// ---------------------------------------------------------------------------
// Decode attention  [HI 核心 idea; TS 标准Transformer解码层的注意力计算,
//                    问题公式化定义 (SparseAttn), Algorithm 1 steps 3-4]
// For q-head h of batch b (kv-head h / G):
//   tokens T = all N context tokens (sel == NULL), or the tokens of the pages
//              in sel[b, h, :] taken in the order given (ascending pages);
//   s_t = scale * q . k_t;  w_t = exp(s_t - max_t s_t);
//   out = sum_t w_t v_t / sum_t w_t.
// The softmax normalises over T only.  The cache holds every context token
// (the current token's K/V already appended), and all of them are attended.
// ---------------------------------------------------------------------------
void oracle_attention(int B, int Hq, int Hkv, int N, int d, int S, int is_fp16,
                      const uint16_t* q, const uint16_t* K, const uint16_t* V, double scale,
                      const int32_t* sel, int nsel, double* out) {
  const int G = Hq / Hkv;
  parallel_for(static_cast<int64_t>(B) * Hq, [&](int64_t bh) {
    const int64_t b = bh / Hq, h = bh % Hq, kvh = h / G;
    const uint16_t* qv = q + bh * d;
    const uint16_t* Kbh = K + (b * Hkv + kvh) * static_cast<int64_t>(N) * d;
    const uint16_t* Vbh = V + (b * Hkv + kvh) * static_cast<int64_t>(N) * d;
    std::vector<int32_t> tokens;
    if (sel == nullptr) {
      tokens.resize(N);
      std::iota(tokens.begin(), tokens.end(), 0);
    } else {
      for (int u = 0; u < nsel; ++u) {
        const int j = sel[bh * nsel + u];
        for (int t = j * S; t < std::min(N, (j + 1) * S); ++t) tokens.push_back(t);
      }
    }
    std::vector<double> qd(d), s(tokens.size());
    for (int i = 0; i < d; ++i) qd[i] = value16(qv[i], is_fp16);
    double smax = -INFINITY;
    for (size_t u = 0; u < tokens.size(); ++u) {
      const uint16_t* k = Kbh + static_cast<int64_t>(tokens[u]) * d;
      double dot = 0.0;
      for (int i = 0; i < d; ++i) dot += qd[i] * value16(k[i], is_fp16);
      s[u] = scale * dot;
      smax = std::max(smax, s[u]);
    }
    std::vector<double> acc(d, 0.0);
    double denom = 0.0;
    for (size_t u = 0; u < tokens.size(); ++u) {
      const double w = std::exp(s[u] - smax);
      denom += w;
      const uint16_t* v = Vbh + static_cast<int64_t>(tokens[u]) * d;
      for (int i = 0; i < d; ++i) acc[i] += w * value16(v[i], is_fp16);
    }
    for (int i = 0; i < d; ++i) out[bh * d + i] = acc[i] / denom;
  });
}

// ---------------------------------------------------------------------------
// 4-bit KV format  [FG 4-bit 近似方法]
// The page fixes: groups of 64 elements along the hidden dimension of each
// (token, head) row, per-group min and max, 4-bit integer codes, values
// dequantised back to FP16 before use.  It leaves the step and the rounding
// open.  The reading adopted here, and shared by the GPU kernels through the
// format, puts 16 levels at mn + c * s, c = 0 .. 15, with the step s rounded
// DOWN from (mx - mn) / 15, so no level passes the group max:
//   mn, mx  = min / max of the group's fp16 values (total order, -0 < +0)
//   range   = fp32_down(mx - mn)
//   normal groups (range >= 451 * 2^-24):
//     s = fp16_down( fp32_down( range / 15 ) )
//   tiny groups (range < 451 * 2^-24, where an fp16 step is too coarse):
//     e = floor(log2(max(|mn|, |mx|))), g = 2^(e - 22),
//     s = floor(range / (15 g)) * g                (0 when range == 0)
//   code_i = 0 if s == 0, else the c in [0, 15] nearest to (x_i - mn) / s in
//            exact arithmetic (ties to the even c; above 15 -> 15)
//   x^_i   = fp16_rn( mn + code_i * s )  -- the exact value, rounded once
// fp32_down / fp16_down: the largest binary32 / binary16 value <= the exact
// result.  Why this bounds the error by (mx - mn)/30 + half an fp16 ulp of x^
// for every finite group: s <= (mx - mn)/15, so every x in [mn, mn + 15 s] is
// within s/2 of a level; and s >= (29/30)(mx - mn)/15 (normal groups: two
// downward roundings of 2^-23 or less each and one fp16 rounding of 2^-10
// relative, or of less than 2^-24 absolute with range >= 451 * 2^-24; tiny
// groups: g <= (mx - mn)/450), so x in (mn + 15 s, mx] is within
// mx - mn - 15 s <= (mx - mn)/30 of the top level.  The level mn + c s is
// exact in double here, so x^ is one rounding of it.  Codes are packed two per
// byte, channel 2i in the low nibble.
// ---------------------------------------------------------------------------
namespace {
// The largest binary32 value <= v (v an exactly known real held in a double).
float f32_down(double v) {
  float f = static_cast<float>(v);  // round to nearest
  if (static_cast<double>(f) > v) f = std::nextafterf(f, -INFINITY);
  return f;
}

// The largest binary16 value <= v, for 0 <= v < 65520, as a double.
double f16_down(double v) {
  if (v <= 0.0) return 0.0;
  int e2;
  std::frexp(v, &e2);
  int ex = e2 - 1;  // v in [2^ex, 2^(ex+1))
  if (ex < -14) ex = -14;
  const double quantum = std::ldexp(1.0, ex - 10);
  return std::floor(v / quantum) * quantum;  // v / quantum is exact (power of two)
}

// fp32_down(r / 15) for a binary32 r >= 0: the largest binary32 q with
// 15 q <= r (15 q and r are exact in double).
float div15_down(float r) {
  float q = static_cast<float>(static_cast<double>(r) / 15.0);
  while (15.0 * static_cast<double>(q) > static_cast<double>(r)) q = std::nextafterf(q, 0.0f);
  while (15.0 * static_cast<double>(std::nextafterf(q, INFINITY)) <= static_cast<double>(r))
    q = std::nextafterf(q, INFINITY);
  return q;
}

// The group's step s (exact, as a double) from its stored min / max.
double group_step(uint16_t mn, uint16_t mx, int* tiny) {
  const double fmn = fp16_value(mn), fmx = fp16_value(mx);
  const float range = f32_down(fmx - fmn);  // fmx - fmn is exact in double
  if (static_cast<double>(range) >= 451.0 * std::ldexp(1.0, -24)) {
    if (tiny) *tiny = 0;
    return f16_down(static_cast<double>(div15_down(range)));
  }
  if (tiny) *tiny = 1;
  const double a = std::max(std::fabs(fmn), std::fabs(fmx));
  if (range == 0.0f || a == 0.0) return 0.0;
  int e2;
  std::frexp(a, &e2);  // a = m 2^e2, m in [0.5, 1): floor(log2 a) = e2 - 1
  const double g = std::ldexp(1.0, e2 - 1 - 22);
  const double r = static_cast<double>(range) / g;  // an integer below 2^24: exact
  return std::floor(r / 15.0) * g;
}

// The code of x: the nearest level index, ties to even, clamped to [0, 15].
int nearest_code(double x, double mn, double s) {
  if (s == 0.0) return 0;
  const double diff = x - mn;  // exact: both fp16
  int c = static_cast<int>(std::floor(diff / s));
  while ((c + 1) * s <= diff) ++c;  // c s is exact: c < 2^5, s has < 25 bits
  while (c > 0 && c * s > diff) --c;
  const double r = 2.0 * diff - (2.0 * c + 1.0) * s;  // exact
  if (r > 0.0 || (r == 0.0 && (c & 1))) ++c;
  return std::min(c, 15);
}
}  // namespace

// The step and regime of the group (mn, mx), exposed so the tests can pin the
// step's bracket (29/30)(mx - mn)/15 <= s <= (mx - mn)/15 directly.
double oracle_q4_step(uint16_t mn, uint16_t mx, int* tiny) { return group_step(mn, mx, tiny); }

void oracle_quant4(int64_t rows, int d, const uint16_t* x, uint8_t* codes, uint16_t* gmin,
                   uint16_t* gmax) {
  const int ng = d / 64;
  parallel_for(rows, [&](int64_t r) {
    const uint16_t* xr = x + r * d;
    uint8_t* cr = codes + r * (d / 2);
    for (int g = 0; g < ng; ++g) {
      uint16_t lo = xr[g * 64], hi = lo;
      for (int i = 1; i < 64; ++i) {
        const uint16_t v = xr[g * 64 + i];
        if (less16(v, lo, 1)) lo = v;
        if (less16(hi, v, 1)) hi = v;
      }
      gmin[r * ng + g] = lo;
      gmax[r * ng + g] = hi;
      const double step = group_step(lo, hi, nullptr);
      const double fmn = fp16_value(lo);
      for (int i = 0; i < 64; i += 2) {
        const int c0 = nearest_code(fp16_value(xr[g * 64 + i]), fmn, step);
        const int c1 = nearest_code(fp16_value(xr[g * 64 + i + 1]), fmn, step);
        cr[(g * 64 + i) / 2] = static_cast<uint8_t>(c0 | (c1 << 4));
      }
    }
  });
}

void oracle_dequant4(int64_t rows, int d, const uint8_t* codes, const uint16_t* gmin,
                     const uint16_t* gmax, uint16_t* x) {
  const int ng = d / 64;
  parallel_for(rows, [&](int64_t r) {
    for (int g = 0; g < ng; ++g) {
      const uint16_t lo = gmin[r * ng + g], hi = gmax[r * ng + g];
      const double step = group_step(lo, hi, nullptr);
      const double mn = fp16_value(lo);
      for (int i = 0; i < 64; ++i) {
        const int ch = g * 64 + i;
        const uint8_t byte = codes[r * (d / 2) + ch / 2];
        const int c = (ch & 1) ? (byte >> 4) : (byte & 0xf);
        // mn + c * step is exact in double (fewer than 43 significant bits); round once.
        x[r * d + ch] = fp16_round(mn + static_cast<double>(c) * step);
      }
    }
  });
}

}  // extern "C"

/* Exhaustive check of the 4-bit format's round-trip bound on small groups.
 *
 * For every pair of finite fp16 values mn < mx with mx - mn <= KMAX * 2^-24,
 * and every fp16 value x in [mn, mx], a 64-element group holding mn, mx and x
 * is quantised and dequantised by the oracle library (loaded with dlopen; the
 * path is argv[1]), and
 *     |x^ - x| <= (mx - mn) / 30 + half an fp16 ulp of x^
 * is checked in exact arithmetic (30 |x^ - x| <= (mx - mn) + 30 half_ulp, all
 * terms dyadic and exact in double).  The bound is the one the 4-bit format of
 * "FlexGen: High-Throughput Generative Inference of Large Language Models with
 * a Single GPU" (4-bit 近似方法: groups of 64, per-group min / max) must keep:
 * half of one of its 15 steps, plus the fp16 rounding of the result.  Groups
 * this narrow are where an fp16 step runs out of precision.
 *
 * Prints "checked N violations V" and exits 1 on any violation.
 */
#include <dlfcn.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

typedef void (*quant_fn)(int64_t, int, const uint16_t*, uint8_t*, uint16_t*, uint16_t*);
typedef void (*dequant_fn)(int64_t, int, const uint8_t*, const uint16_t*, const uint16_t*,
                           uint16_t*);

static double half_value(uint16_t h) {
  const int e = (h >> 10) & 31, f = h & 1023;
  const double v = e ? ldexp(1024.0 + f, e - 25) : ldexp((double)f, -24);
  return (h & 0x8000) ? -v : v;
}

static double half_ulp(double v) { /* half the fp16 spacing at |v| */
  const double a = fabs(v);
  if (a < ldexp(1.0, -14)) return ldexp(1.0, -25);
  int e2;
  frexp(a, &e2);
  return ldexp(1.0, e2 - 1 - 11);
}

#define BATCH 65536

static uint16_t xs[BATCH * 64], xh[BATCH * 64], gmin[BATCH], gmax[BATCH];
static uint8_t codes[BATCH * 32];
static signed char used[BATCH][64]; /* element holds a value under test */
static uint16_t sorted_bits[65536];
static double sorted_val[65536];
static quant_fn quant;
static dequant_fn dequant;
static long long checked, viol;

static int cmp(const void* a, const void* b) {
  const double x = half_value(*(const uint16_t*)a), y = half_value(*(const uint16_t*)b);
  return (x > y) - (x < y);
}

/* Quantise, dequantise and check the ng groups held in the buffers. */
static void flush(int ng) {
  quant(ng, 64, xs, codes, gmin, gmax);
  dequant(ng, 64, codes, gmin, gmax, xh);
  for (int q = 0; q < ng; ++q) {
    const double mn = half_value(gmin[q]), mx = half_value(gmax[q]);
    for (int e = 0; e < 64; ++e) {
      if (!used[q][e]) continue;
      const double x = half_value(xs[(size_t)q * 64 + e]);
      const double y = half_value(xh[(size_t)q * 64 + e]);
      ++checked;
      if (30.0 * fabs(y - x) > (mx - mn) + 30.0 * half_ulp(y)) {
        if (viol < 10) printf("violation: mn=%a mx=%a x=%a x^=%a\n", mn, mx, x, y);
        ++viol;
      }
    }
  }
}

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  const int kmax = argc > 2 ? atoi(argv[2]) : 600;
  void* lib = dlopen(argv[1], RTLD_NOW);
  if (!lib) {
    fprintf(stderr, "%s\n", dlerror());
    return 2;
  }
  quant = (quant_fn)dlsym(lib, "oracle_quant4");
  dequant = (dequant_fn)dlsym(lib, "oracle_dequant4");
  if (!quant || !dequant) return 2;
  int n = 0;
  for (int h = 0; h < 65536; ++h) {
    if (((h >> 10) & 31) == 31 || h == 0x8000) continue; /* finite, one zero */
    sorted_bits[n++] = (uint16_t)h;
  }
  qsort(sorted_bits, n, sizeof(uint16_t), cmp);
  for (int i = 0; i < n; ++i) sorted_val[i] = half_value(sorted_bits[i]);
  const double unit = ldexp(1.0, -24);
  int ng = 0;
  for (int i = 0; i < n; ++i) {
    for (int j = i + 1; j < n && sorted_val[j] - sorted_val[i] <= kmax * unit; ++j) {
      /* the pair (i, j) and every value between, 62 interior values a group */
      for (int l0 = i; l0 <= j; l0 += 62) {
        uint16_t* g = xs + (size_t)ng * 64;
        g[0] = sorted_bits[i];
        g[1] = sorted_bits[j];
        used[ng][0] = used[ng][1] = 1;
        for (int e = 2; e < 64; ++e) {
          const int l = l0 + e - 2;
          g[e] = l <= j ? sorted_bits[l] : sorted_bits[i];
          used[ng][e] = l <= j;
        }
        if (++ng == BATCH) {
          flush(ng);
          ng = 0;
        }
      }
    }
  }
  if (ng > 0) flush(ng);
  printf("checked %lld violations %lld\n", checked, viol);
  return viol ? 1 : 0;
}

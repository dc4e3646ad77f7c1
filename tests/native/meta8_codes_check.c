/* Check of the branch-free 8-bit code rule against its definition.
 *
 * Grid of a page: dec(c) = fma(c, step, lo), c = 0..255, with lo the page's
 * smallest m, step = fl(fl(hi - lo) / 255) raised one ulp at a time until
 * dec(255) >= hi.  The codes are defined as
 *   code_min(m) = the largest c with dec(c) <= m,
 *   code_max(M) = the smallest c with dec(c) >= M,
 * found here by trying all 256 codes.  The rule checked against them:
 *   inv = fl(1 / step),  em = fl(fl(m - lo) * inv),  eM = fl(fl(M - lo) * inv),
 *   fm = floor(em),      gM = ceil(eM)   (as x + 3 2^22 - 1 rounded down / up),
 *   code_min = fm - 1 + [dec(fm) <= m] + [dec(fm + 1) <= m],
 *   code_max = gM - 1 + [dec(gM) < M] + [dec(gM - 1) < M],
 * each comparison taken, as the kernel takes it, from the sign bit of a
 * difference (rounded down for the <= comparisons).
 * It holds when the defining code is within one of the guess; that follows
 * from |em - t| <= 256 * 3 * 2^-24 (t the exact (m - lo) / step) and from a
 * 16-bit page's step being at least 16 fp32 ulps of any value in the page
 * (the smallest range of two distinct fp16 values is one fp16 ulp, 2^13 fp32
 * ulps, over 255).  The rule is used for steps in [2^-100, inf) (1 / step
 * finite and normal); pages with a smaller step (bf16 values below about
 * 2^-92 throughout) or an infinite one (a bf16 range above the largest
 * float) take a search and are counted, not checked, here.  Checked without
 * that argument:
 *   mode "tight": every pair lo < hi of finite 16-bit values at most W
 *     values apart (sorted order) and every 16-bit value v in [lo, hi] taken
 *     as m and as M -- the pages where the step is smallest against the ulp;
 *   mode "pages": random pairs up to maxw values apart, every value between
 *     taken as m and as M;
 *   mode "exact": random pairs up to maxw values apart, every grid point
 *     dec(c) that is exactly c step + lo and a 16-bit value taken as m and
 *     as M (where the rounded guesses land one past the code most often);
 *   mode "random": random pairs over all finite values, with m and M drawn
 *     at and beside the 16-bit values nearest to grid points dec(c).
 * Arguments: fmt (0 bf16, 1 fp16), mode (tight | random), then for tight:
 * W, first and one-past-last lo index; for pages and exact: count, seed,
 * maxw; for random: count, seed.
 * Exit status 0 and "ok <checked> <pages outside the rule>" when every code
 * agrees; the first mismatch otherwise. */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static float from16(uint16_t h, int fp16) {
  if (!fp16) {
    const uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
  }
  const int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  const double v = e == 0 ? ldexp((double)m, -24) : ldexp((double)(1024 + m), e - 25);
  return (float)(s ? -v : v);
}

static int finite16(uint16_t h, int fp16) {
  return fp16 ? ((h >> 10) & 31) != 31 : ((h >> 7) & 255) != 255;
}

static int cmpf(const void* a, const void* b) {
  const float x = *(const float*)a, y = *(const float*)b;
  return x < y ? -1 : (x > y ? 1 : 0);
}

static float dec8(int c, float step, float lo) { return fmaf((float)c, step, lo); }

static float add_dir(float a, float b, int up) {
  const float s = a + b;
  const double exact = (double)a + (double)b; /* exact: |a| < 2^9, b < 2^24 */
  if (!up && (double)s > exact) return nextafterf(s, -INFINITY);
  if (up && (double)s < exact) return nextafterf(s, INFINITY);
  return s;
}

static float page_step(float lo, float hi) {
  if (!(hi > lo)) return 0.0f;
  float step = (hi - lo) / 255.0f;
  while (dec8(255, step, lo) < hi) step = nextafterf(step, INFINITY);
  return step;
}

static int def_min(float m, float step, float lo) {
  int c = -1;
  for (int k = 0; k < 256; ++k)
    if (dec8(k, step, lo) <= m) c = k;
  return c;
}

static int def_max(float M, float step, float lo) {
  for (int k = 0; k < 256; ++k)
    if (dec8(k, step, lo) >= M) return k;
  return -1;
}

/* 3 2^22: x + K - 1 (0 <= x < 2^22) lies where floats are spaced by one, so
 * its rounding down / up is K - 1 + floor(x) / ceil(x), and the float bits of
 * K + j are those of K plus j */
static const float kMagic = 12582912.0f;

/* the sign bit of a difference: fl(x - y) is negative exactly when x < y (+0
 * when equal); rounded down, an exact zero is -0, so the sign bit of
 * fl_down(x - y) is set exactly when x <= y */
static uint32_t sign_of(float d) { return bits_of(d) >> 31; }
static float sub_down(float a, float b) {
  fesetround(FE_DOWNWARD);
  volatile float r = a - b;
  fesetround(FE_TONEAREST);
  return r;
}

static int rule_min(float m, float step, float lo, float inv) {
  const float em = (m - lo) * inv;
  const float tm = add_dir(em, kMagic - 1.0f, 0); /* K - 1 + floor(em) */
  const int64_t c = (int64_t)bits_of(tm) + sign_of(sub_down(fmaf(tm - (kMagic - 1.0f), step, lo), m)) +
                    sign_of(sub_down(fmaf(tm - (kMagic - 2.0f), step, lo), m));
  return (int)(c - (int64_t)bits_of(kMagic));
}

static int rule_max(float M, float step, float lo, float inv) {
  const float eM = (M - lo) * inv;
  const float tM = add_dir(eM, kMagic - 1.0f, 1); /* K - 1 + ceil(eM) */
  const int64_t c = (int64_t)bits_of(tM) + sign_of(fmaf(tM - (kMagic - 1.0f), step, lo) - M) +
                    sign_of(fmaf(tM - kMagic, step, lo) - M);
  return (int)(c - (int64_t)bits_of(kMagic));
}

static unsigned long long n_checked = 0, n_other = 0;

static int check(float lo, float hi, float v, int fp16) {
  if (lo == 0.0f) lo = 0.0f;
  if (hi == 0.0f) hi = 0.0f;
  const float step = page_step(lo, hi);
  if (!(step >= 0x1p-100f && step < INFINITY)) { ++n_other; return 0; }
  const float inv = 1.0f / step;
  if (v >= lo) {
    const int want = def_min(v, step, lo), got = rule_min(v, step, lo, inv);
    if (want != got) {
      printf("code_min mismatch fmt=%d lo=%a hi=%a m=%a step=%a: got %d want %d\n", fp16, lo,
             hi, v, step, got, want);
      return 1;
    }
    ++n_checked;
  }
  if (v <= hi) {
    const int want = def_max(v, step, lo), got = rule_max(v, step, lo, inv);
    if (want != got) {
      printf("code_max mismatch fmt=%d lo=%a hi=%a M=%a step=%a: got %d want %d\n", fp16, lo,
             hi, v, step, got, want);
      return 1;
    }
    ++n_checked;
  }
  return 0;
}

static uint64_t rng_state;
static uint64_t next_u64(void) { /* splitmix64 */
  uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* index of the largest value <= x in the sorted table */
static int64_t floor_index(const float* vals, int64_t n, float x) {
  int64_t a = 0, b = n - 1;
  if (x < vals[0]) return 0;
  while (a < b) {
    const int64_t mid = (a + b + 1) / 2;
    if (vals[mid] <= x) a = mid; else b = mid - 1;
  }
  return a;
}

int main(int argc, char** argv) {
  if (argc < 4) return 2;
  const int fp16 = atoi(argv[1]);
  float* vals = malloc(sizeof(float) * 65536);
  int64_t n = 0;
  for (uint32_t h = 0; h < 65536; ++h)
    if (finite16((uint16_t)h, fp16) && h != 0x8000u) vals[n++] = from16((uint16_t)h, fp16);
  qsort(vals, (size_t)n, sizeof(float), cmpf);
  if (strcmp(argv[2], "tight") == 0) {
    const int W = atoi(argv[3]);
    const int64_t a0 = argc > 4 ? atoll(argv[4]) : 0, a1 = argc > 5 ? atoll(argv[5]) : n;
    for (int64_t a = a0; a < a1 && a < n; ++a)
      for (int64_t b = a + 1; b <= a + W && b < n; ++b)
        for (int64_t k = a; k <= b; ++k)
          if (check(vals[a], vals[b], vals[k], fp16)) return 1;
  } else if (strcmp(argv[2], "pages") == 0) {
    const long long count = atoll(argv[3]);
    rng_state = argc > 4 ? strtoull(argv[4], 0, 0) : 1;
    const int64_t maxw = argc > 5 ? atoll(argv[5]) : 4096;
    for (long long i = 0; i < count; ++i) {
      const int64_t a = (int64_t)(next_u64() % (uint64_t)n);
      const int64_t b = a + 1 + (int64_t)(next_u64() % (uint64_t)maxw);
      for (int64_t k = a; k <= b && b < n; ++k)
        if (check(vals[a], vals[b], vals[k], fp16)) return 1;
    }
  } else if (strcmp(argv[2], "exact") == 0) {
    const long long count = atoll(argv[3]);
    rng_state = argc > 4 ? strtoull(argv[4], 0, 0) : 1;
    const int64_t maxw = argc > 5 ? atoll(argv[5]) : 4096;
    for (long long i = 0; i < count; ++i) {
      const int64_t a = (int64_t)(next_u64() % (uint64_t)n);
      const int64_t b = a + 1 + (int64_t)(next_u64() % (uint64_t)maxw);
      if (b >= n) continue;
      const float lo = vals[a] == 0.0f ? 0.0f : vals[a], hi = vals[b] == 0.0f ? 0.0f : vals[b];
      const float step = page_step(lo, hi);
      for (int c = 1; c < 255; ++c) {
        const float x = dec8(c, step, lo);
        if ((double)x != (double)c * (double)step + (double)lo) continue; /* not exact */
        const int64_t k = floor_index(vals, n, x);
        if (vals[k] == x && check(lo, hi, x, fp16)) return 1;
      }
    }
  } else {
    const long long count = atoll(argv[3]);
    rng_state = argc > 4 ? strtoull(argv[4], 0, 0) : 1;
    for (long long i = 0; i < count; ++i) {
      int64_t a = (int64_t)(next_u64() % (uint64_t)n), b = (int64_t)(next_u64() % (uint64_t)n);
      if (a == b) continue;
      if (a > b) { const int64_t t = a; a = b; b = t; }
      const float lo = vals[a], hi = vals[b];
      const float step = page_step(lo == 0.0f ? 0.0f : lo, hi == 0.0f ? 0.0f : hi);
      const int c = (int)(next_u64() % 256);
      const int64_t k0 = floor_index(vals, n, dec8(c, step, lo == 0.0f ? 0.0f : lo));
      for (int64_t k = k0 - 2; k <= k0 + 2; ++k)
        if (k >= a && k <= b && check(lo, hi, vals[k], fp16)) return 1;
      const int64_t r = a + (int64_t)(next_u64() % (uint64_t)(b - a + 1));
      if (check(lo, hi, vals[r], fp16)) return 1;
    }
  }
  printf("ok %llu %llu\n", n_checked, n_other);
  free(vals);
  return 0;
}

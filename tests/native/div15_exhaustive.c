/* Exhaustive check of division by 15 with a fused multiply-add correction
 * (Markstein's method for division by a constant; Brisebarre and Muller,
 * "Correctly rounded multiplication by arbitrary precision constants"):
 *   c = RN(1/15); q = RN(x * c); r = RN(fma(-q, 15, x)); q' = RN(fma(r, c, q))
 * against the IEEE quotient RN(x / 15), for every binary32 x in [0, 2^18)
 * (the range of fl(max - min) for two finite fp16 values is [0, 131008]);
 * and the quotient rounded down from it, q' or the binary32 just below q' as
 * the exact remainder fma(-q', 15, x) is >= 0 or < 0, against the largest
 * binary32 q with 15 q <= x (15 q is exact in double).
 * Optional arguments: the first and one-past-last bit patterns to check (so
 * the range can be split over processes).  Exit status 0 when every x agrees;
 * prints the first mismatch otherwise. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

int main(int argc, char** argv) {
  const float c = 1.0f / 15.0f;
  const uint32_t begin = argc > 2 ? (uint32_t)strtoul(argv[1], 0, 0) : 0u;
  const uint32_t end = argc > 2 ? (uint32_t)strtoul(argv[2], 0, 0) : 0x48800000u; /* 2^18 */
  unsigned long long n = 0;
  for (uint32_t u = begin; u < end; ++u) {
    const float x = from_bits(u);
    const float q = x * c;
    const float r = fmaf(-q, 15.0f, x);
    const float q2 = fmaf(r, c, q);
    const float want = x / 15.0f;
    if (memcmp(&q2, &want, 4) != 0) {
      printf("mismatch at x=%a: got %a want %a\n", x, q2, want);
      return 1;
    }
    const float r2 = fmaf(-q2, 15.0f, x);
    const float down = r2 < 0.0f ? nextafterf(q2, 0.0f) : q2;
    if (15.0 * (double)down > (double)x ||
        15.0 * (double)nextafterf(down, INFINITY) <= (double)x) {
      printf("rounded-down mismatch at x=%a: got %a\n", x, down);
      return 1;
    }
    ++n;
  }
  printf("ok %llu values\n", n);
  return 0;
}

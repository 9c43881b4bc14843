/* Exhaustive check of the device codec's quotient method (plain C, fp32).
 *
 * The device forms v / d from an approximate reciprocal r and one fused
 * multiply-add refinement (Markstein's method): q0 = v r, q1 = q0 -
 * (q0 d - v) r, the residual formed so that v = -0 gives -0. This program
 * checks, for every nonzero e4m3 scale d and every bf16 v with |v| <= 9 d in
 * both signs (+-0 included), and for every r within three ulps of the
 * correctly rounded 1 / d, that q1 converts to the same e2m1 code as the
 * correctly rounded quotient v / d; and, for d = 6 (the block scale amax / 6)
 * and every finite bf16 amax, the same e4m3 code. The conversions here are written from the value sets (nearest, ties
 * to the even code, saturating), independently of the oracle and the device.
 * Exit status 0 and the counts on stdout when every case agrees. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float from_bits(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t to_bits(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

/* value of an e4m3 (E4M3FN) code 0x00..0x7E */
static float e4m3_value(int c) {
  const int e = (c >> 3) & 15, m = c & 7;
  return e == 0 ? ldexpf((float)m, -9) : ldexpf(1.0f + m / 8.0f, e - 7);
}

/* e2m1 code, nearest with ties to the even code, saturating at 6 */
static int e2m1_code(float x) {
  static const float mid[7] = {0.25f, 0.75f, 1.25f, 1.75f, 2.5f, 3.5f, 5.0f};
  const float a = fabsf(x);
  int c = 0;
  for (int i = 0; i < 7; ++i) {
    if (a > mid[i]) c = i + 1;
    else { if (a == mid[i]) c = (i % 2 == 0) ? i : i + 1; break; }
  }
  return c | (signbit(x) ? 8 : 0);
}

/* e4m3 code of x >= 0: the nearest of the 127 values, ties to the even code,
 * saturating at 448 */
static int e4m3_code(float x) {
  if (!(x > 0.0f)) return 0;
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    const double dist = fabs((double)e4m3_value(c) - (double)x);
    if (dist < bd || (dist == bd && (c & 1) == 0)) { bd = dist; best = c; }
  }
  return best;
}

static float refined(float v, float d, float r) {
  const float q0 = v * r;
#ifdef WITHOUT_REFINEMENT /* the check must reject the plain product v r */
  return q0;
#else
  return fmaf(-fmaf(q0, d, -v), r, q0);
#endif
}

int main(void) {
  long pairs = 0, code_bad = 0, scale_bad = 0, scales = 0;
  for (int c = 1; c <= 0x7E; ++c) {
    const float d = e4m3_value(c), r0 = 1.0f / d;
    for (int k = -3; k <= 3; ++k) {
      const float r = from_bits(to_bits(r0) + (uint32_t)k);
      for (uint32_t h = 0; h < 0x7F80u; ++h) {
        const float v = from_bits(h << 16);
        if (v > 9.0f * d) break;
        for (int s = 0; s < 2; ++s) {
          const float x = s ? -v : v;
          ++pairs;
          if (e2m1_code(x / d) != e2m1_code(refined(x, d, r))) {
            if (code_bad++ < 5) printf("e2m1 mismatch: scale 0x%02x, r %+d ulp, v %a\n", c, k, x);
          }
        }
      }
    }
  }
  for (int k = -3; k <= 3; ++k) {
    const float r = from_bits(to_bits(1.0f / 6.0f) + (uint32_t)k);
    for (uint32_t h = 0; h < 0x7F80u; ++h) {
      const float a = from_bits(h << 16);
      ++scales;
      if (e4m3_code(a / 6.0f) != e4m3_code(refined(a, 6.0f, r))) {
        if (scale_bad++ < 5) printf("e4m3 mismatch: r %+d ulp, amax %a\n", k, a);
      }
    }
  }
  printf("e2m1 pairs %ld mismatches %ld; e4m3 scales %ld mismatches %ld\n", pairs, code_bad, scales, scale_bad);
  return (code_bad || scale_bad) ? 1 : 0;
}

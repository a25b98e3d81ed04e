/* Host check used by test_fma_division.py (test infrastructure).
 *
 * The CUDA block quantizer divides each scaled element a = RN(x * gs) by the
 * block's E4M3 scale s. Instead of one correctly rounded division per element
 * it forms rcp = RN(1/s) once per block and then, per element,
 *     q0 = RN(a * rcp);  r = fma(-q0, s, a);  q = copysign(fma(r, rcp, q0), a)
 * This program checks q == RN(a / s) bit for bit for every non-zero E4M3 scale
 * s (codes 0x01-0x7E) and every f32 a in [1, 2) (rounding repeats in every
 * other binade as long as nothing is subnormal), both signs of zero, and a
 * spread of other exponents. Exit status 0 iff no mismatch. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static double e4m3_value(int c) {
  const int e = (c >> 3) & 15, m = c & 7;
  return e == 0 ? m * ldexp(1.0, -9) : (1.0 + m / 8.0) * ldexp(1.0, e - 7);
}

static float quotient(float a, float s, float rcp) {
  const float q0 = a * rcp;
  const float r = fmaf(-q0, s, a);
  return copysignf(fmaf(r, rcp, q0), a);
}

int main(void) {
  long n = 0, bad = 0;
  for (int c = 1; c <= 0x7E; ++c) {
    const float s = (float)e4m3_value(c);
    const float rcp = 1.0f / s;
    const float zeros[2] = {0.0f, -0.0f};
    for (int z = 0; z < 2; ++z) {
      ++n;
      if (u_of(quotient(zeros[z], s, rcp)) != u_of(zeros[z] / s)) ++bad;
    }
    for (uint32_t m = 0; m < (1u << 23); ++m) {
      const float a = f_of(0x3F800000u | m);                 /* [1, 2) */
      ++n;
      if (u_of(quotient(a, s, rcp)) != u_of(a / s)) ++bad;
      if ((m & 4095u) == 0) {                                 /* other binades and signs */
        for (int e = -20; e <= 20; e += 5) {
          const float b = -ldexpf(a, e);
          ++n;
          if (u_of(quotient(b, s, rcp)) != u_of(b / s)) ++bad;
        }
      }
    }
  }
  printf("checked %ld quotients, %ld mismatches\n", n, bad);
  return bad != 0;
}

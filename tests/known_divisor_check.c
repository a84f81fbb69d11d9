/*
 * Exhaustive check of division by a divisor known in advance, as the quantising append does
 * it for bf16 inputs: r = RN(1/s) once per divisor, then for each x
 *     q0 = RN(x * r),   q = RN(q0 - r * RN(q0 * s - x))     (the last two as fused multiply-adds)
 * must equal the IEEE quotient RN(x / s). Every bf16 value is a significand of at most 8 bits
 * times a power of two, and the steps above commute with powers of two while no intermediate
 * is subnormal or overflows, so it suffices to run x over the 128 significands in [1, 2) and s
 * over all 2^23 fp32 values in [1, 2). Prints the number of cases, the cases where the
 * corrected quotient differs, and (as a control showing the check can fail) the cases where
 * the uncorrected q0 differs; then the signs of the quotients of +0 and -0 (0 if both are
 * right).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint32_t u_of(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

int main(void) {
  long n = 0, wrong = 0, wrong_uncorrected = 0;
#pragma omp parallel for reduction(+ : n, wrong, wrong_uncorrected) schedule(dynamic, 4096)
  for (long sb = 0x3f800000L; sb < 0x40000000L; ++sb) {
    volatile float sv = f_of((uint32_t)sb);
    const float s = sv;
    const float r = 1.0f / s;
    for (int m = 128; m < 256; ++m) {
      const float x = (float)m / 128.0f;
      const float ref = x / s;
      const float q0 = x * r;
      const float q = fmaf(-fmaf(q0, s, -x), r, q0);
      wrong += u_of(q) != u_of(ref);
      wrong_uncorrected += u_of(q0) != u_of(ref);
      ++n;
    }
  }
  int zero_signs = 0;
  for (int neg = 0; neg < 2; ++neg) {
    volatile float sv = 0.37f, xv = neg ? -0.0f : 0.0f;
    const float s = sv, r = 1.0f / s, x = xv;
    const float q0 = x * r;
    volatile float rem = fmaf(q0, s, -x);  /* (kept apart: no rewrite of -fma into fnma) */
    const float q = fmaf(-rem, r, q0);
    zero_signs += (signbit(q) != 0) != neg;
  }
  printf("%ld %ld %ld %d\n", n, wrong, wrong_uncorrected, zero_signs);
  return 0;
}

/*
 * Host check of the NVFP4 quantizer's element encode (nvfp4.cu): with
 * y = RN(x * RN(1/D)), the E2M1 code of y is kept when y * (1 - 2^-20) and
 * y * (1 + 2^-20) (rounded) have the same code, else the IEEE quotient
 * RN(x / D) is encoded; the result equals the E2M1 code of RN(x / D), for
 * every finite bf16 x and divisors D = g * s, s every
 * positive E4M3 value and g = m 2^k with small odd m (quotients on and one
 * ulp beside the boundaries) or random.  The control run without the
 * fallback must find mismatches, so the divisors do reach the boundaries.
 * Host binary32 arithmetic is IEEE round-to-nearest-even, as the device's
 * __fmul_rn, __frcp_rn and __fdiv_rn are.  Exit status 0 = pass.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t b_of(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

/* E2M1 values, nearest with ties to the even code, saturating, sign kept. */
static const double kE2m1[8] = {0, .5, 1, 1.5, 2, 3, 4, 6};
static int e2m1(float v) {
  const double a = fabs((double)v);
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double dc = fabs(kE2m1[c] - a), db = fabs(kE2m1[best] - a);
    if (dc < db || (dc == db && (c & 1) == 0)) best = c;
  }
  if (a > 6.0) best = 7;
  return best | (signbit(v) ? 8 : 0);
}
static double e4m3(int c) {
  const int e = c >> 3, m = c & 7;
  return e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m, -9);
}
/* the kernel's test: the codes at the two ends of a bracket of y differ */
static int near_boundary(float y) {
  volatile float lo = y * (1.0f - 0x1p-20f), hi = y * (1.0f + 0x1p-20f);
  return e2m1(lo) != e2m1(hi);
}

int main(void) {
  unsigned long long n = 0, slow = 0, bad = 0, bad_control = 0;
  uint32_t seed = 12345;
  for (int t = 0; t < 8 + 16 * 5; ++t) {
    float g;
    if (t < 8) {
      seed = seed * 1664525u + 1013904223u;
      g = f_of(((uint32_t)(87 + (seed >> 8) % 60) << 23) | ((seed * 2654435761u) >> 9));
    } else {
      const int u = t - 8, m = 2 * (u % 16) + 1, k = u / 16 - 2;
      g = (float)ldexp((double)m, 3 * k - 6);
    }
    for (int sc = 1; sc <= 0x7E; ++sc) {
      volatile float d = g * (float)e4m3(sc);
      if (!(d >= 0x1p-126f)) continue;
      volatile float r = 1.0f / d;
      for (uint32_t xb = 0; xb < 0x10000; ++xb) {
        if ((xb & 0x7F80u) == 0x7F80u) continue; /* inf / nan */
        const float x = f_of(xb << 16);
        volatile float q = x / d;
        volatile float y = x * r;
        const int want = e2m1(q);
        const int got = near_boundary(y) ? (++slow, e2m1(q)) : e2m1(y);
        if (got != want) {
          if (bad < 5) printf("MISMATCH x=%a d=%a y=%a q=%a\n", x, d, y, q);
          ++bad;
        }
        if (e2m1(y) != want) ++bad_control;
        ++n;
      }
    }
  }
  printf("pairs %llu, fallback %llu, mismatches %llu, control mismatches %llu\n", n, slow, bad,
         bad_control);
  return (bad == 0 && bad_control > 0) ? 0 : 1;
}

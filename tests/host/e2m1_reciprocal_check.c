/*
 * Host check of the NVFP4 quantizer's element encode (nvfp4.cu): with
 * y = RN(x * RN(1/D)), the E2M1 code of y is kept when y * (1 - 2^-20) and
 * y * (1 + 2^-20) (rounded) have the same code, else the IEEE quotient
 * RN(x / D) is encoded; the result equals the E2M1 code of RN(x / D), for
 * every finite bf16 x and divisors D = g * s, s every
 * positive E4M3 value and g = m 2^k with small odd m (quotients on and one
 * ulp beside the boundaries) or random.  The kernel's reciprocal is the
 * hardware approximation (at most 1 ulp from 1/D, for 2^-126 <= D <=
 * 2^125), so every fp32 value within 1 ulp of 1/D is tried: RN(1/D) and
 * its two neighbours.  The control run without the fallback must find
 * mismatches, so the divisors do reach the boundaries.
 *
 * The block scale takes the same route: E4M3(RN(amax * RN(1/d6))) when
 * the E4M3 codes of that product times 1 -+ 2^-20 agree, else
 * E4M3(RN(amax / d6)); checked against E4M3(RN(amax / d6)) for every
 * finite non-negative bf16 amax and d6 = RN(6 g) over the same g.
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
/* E4M3 code of v >= 0: nearest, ties to the even code, saturating at 448
 * (the device's cvt.rn.satfinite.e4m3x2.f32 on non-negative input). */
static int e4m3_code_of(float v) {
  if (v >= 448.0f) return 0x7E;
  int lo = 0, hi = 0x7E; /* largest code with value <= v */
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (e4m3(mid) <= (double)v) lo = mid; else hi = mid - 1;
  }
  if (lo == 0x7E) return lo;
  const double dl = (double)v - e4m3(lo), dh = e4m3(lo + 1) - (double)v;
  if (dl < dh) return lo;
  if (dh < dl) return lo + 1;
  return (lo & 1) ? lo + 1 : lo;
}

/* the kernel's test: the codes at the two ends of a bracket of y differ */
static int near_boundary(float y) {
  volatile float lo = y * (1.0f - 0x1p-20f), hi = y * (1.0f + 0x1p-20f);
  return e2m1(lo) != e2m1(hi);
}

int main(void) {
  unsigned long long n = 0, slow = 0, bad = 0, bad_control = 0;
  unsigned long long sn = 0, sslow = 0, sbad = 0, sbad_control = 0;
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
      if (!(d >= 0x1p-126f) || d > 0x1p125f) continue; /* the kernel divides there */
      const float rn = 1.0f / d;
      const float rs[3] = {nextafterf(rn, 0.0f), rn, nextafterf(rn, INFINITY)};
      for (int ri = 0; ri < 3; ++ri) {
        volatile float r = rs[ri];
        for (uint32_t xb = 0; xb < 0x10000; ++xb) {
          if ((xb & 0x7F80u) == 0x7F80u) continue; /* inf / nan */
          const float x = f_of(xb << 16);
          volatile float q = x / d;
          volatile float y = x * r;
          const int want = e2m1(q);
          const int got = near_boundary(y) ? (++slow, e2m1(q)) : e2m1(y);
          if (got != want) {
            if (bad < 5) printf("MISMATCH x=%a d=%a r=%a y=%a q=%a\n", x, d, r, y, q);
            ++bad;
          }
          if (e2m1(y) != want) ++bad_control;
          ++n;
        }
      }
    }
    /* block scale: d6 = RN(6 g), r6 = RN(1 / d6), every non-negative bf16 amax */
    volatile float d6 = 6.0f * g;
    if (d6 >= 0x1p-125f && d6 <= 0x1p125f) {
      volatile float r6 = 1.0f / d6;
      for (uint32_t ab = 0; ab < 0x7F80u; ++ab) {
        const float amax = f_of(ab << 16);
        volatile float te = amax / d6;
        volatile float t = amax * r6;
        volatile float tl = t * (1.0f - 0x1p-20f), th = t * (1.0f + 0x1p-20f);
        const int want = e4m3_code_of(te);
        const int cl = e4m3_code_of(tl), ch = e4m3_code_of(th);
        const int got = cl == ch ? cl : (++sslow, want);
        if (got != want) {
          if (sbad < 5) printf("SCALE MISMATCH amax=%a d6=%a t=%a te=%a\n", amax, d6, t, te);
          ++sbad;
        }
        if (e4m3_code_of(t) != want) ++sbad_control;
        ++sn;
      }
    }
  }
  printf("pairs %llu, fallback %llu, mismatches %llu, control mismatches %llu\n", n, slow, bad,
         bad_control);
  printf("scales %llu, fallback %llu, mismatches %llu, control mismatches %llu\n", sn, sslow,
         sbad, sbad_control);
  return (bad == 0 && bad_control > 0 && sbad == 0 && sbad_control > 0) ? 0 : 1;
}

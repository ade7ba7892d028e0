// Device helpers of the quantizers, shared by the quantizer kernels and the
// GEMM that quantizes its activations itself: 16-byte streaming loads and
// stores, the exact amax of bf16 groups, the group scale (fp32 or UE8M0),
// the E4M3 encode with the division-free exact quotient (see quant.cu for
// the method and its check) and the E2M1 pair conversion of the FP4
// quantizers.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "fgq_device.cuh"

namespace fgq {
namespace {

constexpr int kScaleFp32 = 0;
constexpr int kScaleUe8m0 = 1;

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream_8(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_stream_16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Max of |x| over 8 bf16 held in a uint4, as a pair of 16-bit magnitudes.
__device__ __forceinline__ uint32_t absmax_pairs(uint4 v) {
  const uint32_t m = 0x7FFF7FFFu;
  uint32_t a = __vmaxu2(v.x & m, v.y & m);
  uint32_t b = __vmaxu2(v.z & m, v.w & m);
  return __vmaxu2(a, b);
}

// Eight fp32 -> eight E2M1 codes in 32 bits: byte j = element 2j (low
// nibble) and element 2j+1 (high nibble).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&y)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
  return r;
}

__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Packed fp32 pair arithmetic (one instruction for two lanes of data).
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 A, B, D;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\t"
      "mul.rn.f32x2 D, A, B;\n\tmov.b64 {%0, %1}, D;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{.reg .b64 A, B, C, D;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\tmov.b64 C, {%6, %7};\n\t"
      "fma.rn.f32x2 D, A, B, C;\n\tmov.b64 {%0, %1}, D;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// Per-group constants of the encode step.
struct GroupScale {
  float s;       // dequantisation multiplier written to the scale tensor
  float2 r2;     // {RN(1/s), RN(1/s)} (fp32 mode) or {2^-e, 2^-e} (UE8M0)
  float2 ns2;    // {-s, -s}
  bool exact;    // fp32 mode with s < 2^-100: use IEEE division
};

template <int MODE>
__device__ __forceinline__ GroupScale group_scale(uint32_t mag_bits) {
  GroupScale g;
  const float amax = __uint_as_float(mag_bits << 16);
  float s;
  if (amax == 0.0f) {
    s = 1.0f;
  } else {
    const float t = __fdiv_rn(amax, 448.0f);
    if (MODE == kScaleFp32) {
      s = t;
    } else {
      // smallest power of two >= t, exponent clamped at -127 (t < 2^120)
      const uint32_t b = __float_as_uint(t);
      const uint32_t e = b >> 23, man = b & 0x7FFFFFu;
      if (e == 0)
        s = __uint_as_float(b <= 0x00400000u ? 0x00400000u : 0x00800000u);
      else
        s = __uint_as_float((man != 0 ? e + 1 : e) << 23);
    }
  }
  const float r = __frcp_rn(s);  // exact for powers of two
  g.s = s;
  g.r2 = make_float2(r, r);
  g.ns2 = make_float2(-s, -s);
  g.exact = (MODE == kScaleFp32) && !(s >= 0x1p-100f);
  return g;
}

// Codes of the 8 bf16 of v, little-endian in 8 bytes: E4M3(fl32(x / s)).
template <int MODE>
__device__ __forceinline__ uint2 encode8(uint4 v, const GroupScale& g) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
  if (MODE == kScaleUe8m0) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 q = mul2(bf16x2_to_f32x2(w[p]), g.r2);
      c[p] = cvt_e4m3x2(q.x, q.y);
    }
  } else if (!g.exact) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 x = bf16x2_to_f32x2(w[p]);
      const float2 q0 = mul2(x, g.r2);
      const float2 d = fma2(q0, g.ns2, x);  // x - q0 * s, exact
      const float2 q = fma2(d, g.r2, q0);
      c[p] = cvt_e4m3x2(q.x, q.y);
    }
  } else {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 x = bf16x2_to_f32x2(w[p]);
      c[p] = cvt_e4m3x2(__fdiv_rn(x.x, g.s), __fdiv_rn(x.y, g.s));
    }
  }
  // Sign bit of each code from the sign of its bf16 input (bytes 1 and 3 of
  // each input word carry the signs of its two elements).
  const uint32_t s01 = __byte_perm(v.x, v.y, 0x7531) & 0x80808080u;
  const uint32_t s23 = __byte_perm(v.z, v.w, 0x7531) & 0x80808080u;
  uint2 r;
  r.x = __byte_perm(c[0], c[1], 0x5410) | s01;
  r.y = __byte_perm(c[2], c[3], 0x5410) | s23;
  return r;
}

}  // namespace
}  // namespace fgq

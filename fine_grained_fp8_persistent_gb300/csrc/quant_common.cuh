// quant_common.cuh -- the 1x128 / 128x128 E4M3 quantization arithmetic shared by
// the quantize kernels and by the GEMM epilogue that quantizes its own output, so
// that both produce the same bits.
//
// "DeepGEMM dissected", section on fine-grained quantization: a group's scale
// maps its max |x| to the top of the E4M3 range, s = amax / 448; with
// power-of-two (UE8M0) scales the exponent is rounded up so nothing saturates.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fgf8 {
namespace quant {

constexpr float kE4M3Max = 448.0f;

// ceil(log2(amax / 448)) computed exactly from the bits of the FP32 quotient,
// clamped to the UE8M0 range; 0 for amax == 0.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
  if (amax == 0.0f) return 0;
  const float t = __fdiv_rn(amax, kE4M3Max);
  const uint32_t b = __float_as_uint(t);
  const int ex = static_cast<int>((b >> 23) & 0xFFu);
  const uint32_t man = b & 0x7FFFFFu;
  int e;
  if (ex != 0) {
    e = ex - 127 + (man != 0u ? 1 : 0);
  } else {                                   // subnormal quotient: t = man * 2^-149
    const int msb = 31 - __clz(man);
    e = msb - 149 + ((man & (man - 1u)) != 0u ? 1 : 0);
  }
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// x / s rounded to nearest for an FP32 scale s, without the IEEE division
// routine: Markstein's FMA-based division (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev.
// 34(1), 1990).  With y = 1/s correctly rounded and a quotient q within one ulp of
// x / s, the remainder x - q * s is exact in an FMA and q + (x - q * s) * y
// rounded to nearest is the correctly rounded quotient.  q0 = x * y can be 1.5
// ulps off, so a first correction makes it faithful and a second rounds it.  The
// theorem needs every intermediate to stay normal: the remainder is ~2^-23 |x|
// and |x| >= 2^-10 s wherever the E4M3 code is not zero, so scales from 2^-93 up
// are safe; smaller ones (groups with max |x| below ~4.5e-26) take the IEEE
// routine, flagged by y = 0.  The sign is x's, as the quotient's (the correction
// turns -0 into +0).
constexpr float kMinFmaDivScale = 0x1p-93f;

__device__ __forceinline__ float scale_reciprocal(float s) {
  return s >= kMinFmaDivScale ? __frcp_rn(s) : 0.0f;
}

// Two quotients x0 / s, x1 / s on paired FP32 instructions; y from scale_reciprocal.
__device__ __forceinline__ void div_by_scale2(float x0, float x1, float s, float y, float& q0, float& q1) {
  if (y == 0.0f) {
    q0 = __fdiv_rn(x0, s);
    q1 = __fdiv_rn(x1, s);
    return;
  }
  float a, b;
  asm("{\n\t.reg .b64 x, yy, ns, q, e;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 yy, {%4, %4};\n\t"
      "mov.b64 ns, {%5, %5};\n\t"
      "mul.rn.f32x2 q, x, yy;\n\t"
      "fma.rn.f32x2 e, q, ns, x;\n\t"
      "fma.rn.f32x2 q, e, yy, q;\n\t"
      "fma.rn.f32x2 e, q, ns, x;\n\t"
      "fma.rn.f32x2 q, e, yy, q;\n\t"
      "mov.b64 {%0, %1}, q;\n\t}"
      : "=f"(a), "=f"(b)
      : "f"(x0), "f"(x1), "f"(y), "f"(-s));
  q0 = copysignf(a, x0);
  q1 = copysignf(b, x1);
}

// 2^-e as an FP32 value, e in [-127, 127].
__device__ __forceinline__ float exp2_neg(int e) {
  const int be = 127 - e;
  return be >= 1 ? __uint_as_float(static_cast<uint32_t>(be) << 23) : __uint_as_float(0x00400000u);
}

// A group's scale from its max |x|.  FP32: s = amax / 448 (1 for an all-zero
// group).  UE8M0: exponent e, the exact multiplier 2^-e, and the stored byte e + 127.
struct GroupScale {
  float s;         // FP32 scale
  float inv;       // UE8M0: 2^-e
  uint32_t byte;   // UE8M0: e + 127
};
template <bool UE8M0>
__device__ __forceinline__ GroupScale group_scale(float amax) {
  GroupScale g{1.0f, 1.0f, 127u};
  if (UE8M0) {
    const int e = ue8m0_exponent(amax);
    g.inv = exp2_neg(e);
    g.byte = static_cast<uint32_t>(e + 127);
  } else if (amax != 0.0f) {
    g.s = __fdiv_rn(amax, kE4M3Max);
  }
  return g;
}

// One value scaled into the E4M3 range: FP32 scales divide (rounded to nearest),
// power-of-two scales multiply by the exact 2^-e.
template <bool UE8M0>
__device__ __forceinline__ float scaled(float x, const GroupScale& g) {
  return UE8M0 ? x * g.inv : __fdiv_rn(x, g.s);
}

// Four values -> four packed E4M3 bytes (RNE, saturating), first value lowest.
template <bool UE8M0>
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, const GroupScale& g) {
  return static_cast<uint32_t>(ptx::cvt_e4m3x2(scaled<UE8M0>(a, g), scaled<UE8M0>(b, g))) |
         (static_cast<uint32_t>(ptx::cvt_e4m3x2(scaled<UE8M0>(c, g), scaled<UE8M0>(d, g))) << 16);
}

}  // namespace quant
}  // namespace fgf8

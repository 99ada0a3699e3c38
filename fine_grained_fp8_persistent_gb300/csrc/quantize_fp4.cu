// quantize_fp4.cu -- BF16 -> 4-bit E2M1 with block scales along K: MXFP4 (an E8M0
// power-of-two scale per 32 elements) and NVFP4 (an E4M3 scale per 16 elements).
//
// "GPU GEMM part 4: tcgen05 & Blackwell", section 6.1: every SV consecutive K
// elements of a row share one scale (both operands, so the same kernel serves
// activations and weights); section 6.3: MXFP4 = E2M1 + E8M0 per 32, NVFP4 =
// E2M1 + E4M3 per 16; section 7.1: two 4-bit elements per byte along K.
//   MXFP4 scale 2^e, e = ceil(log2(amax / 6)) (FP32 quotient), codes E2M1(x 2^-e);
//   NVFP4 scale s = E4M3(amax / 6) (FP32 quotient, nearest even, saturating),
//         codes E2M1(x / s) of the FP32 quotient (0 when s is 0; computed by
//         nv_quotient without a full division);
//   an all-zero group has scale 1; E2M1 rounds to nearest even, saturating at 6.
//
// An HBM stream: 2 bytes read and half a byte written per element, plus one
// scale byte per 32 or 16 elements.  One warp per (row, 512-element chunk): lane
// l holds 16 consecutive elements (two 16-byte loads), i.e. one NVFP4 group or
// half an MXFP4 group, and writes its 8 code bytes, so a warp reads 1 KB and
// writes 256 contiguous bytes.  Scale bytes are gathered by shuffles into the
// little-endian words of the M-major table int32 [ceil(K / SV / 4)][align4(R)].
#include <cuda_bf16.h>

#include <cstdint>

#include "fgf8_internal.h"
#include "ptx.cuh"

namespace fgf8 {
namespace {

// ceil(log2(amax / 6)) from the bits of the FP32 quotient, clamped to [-127, 127].
__device__ __forceinline__ int mx_exponent(float amax) {
  if (amax == 0.0f) return 0;
  const float t = __fdiv_rn(amax, 6.0f);
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

// E2M1(x / s) for NVFP4 without a full IEEE division, giving the code the
// correctly rounded FP32 quotient gives.  x is a bf16 value (at most 8
// significant bits) and s an E4M3 scale (at most 4), so x / s is either exactly
// one of the E2M1 rounding midpoints m (0.25, 0.75, ..., 5: at most 3 significant
// bits, and m * s is exact in FP32) or at least 2^-8 (relative) away from every
// one of them: x - m * s is a nonzero multiple of the coarser of the two values'
// last-bit weights.  q0 = x * (1 / s) is within 2^-23 of x / s, so it lies on the
// same side of every midpoint except in the exact case; one correction step with
// the exact remainder (the FMA remainder step of Markstein's division), q1 = q0 +
// (x - q0 * s) * (1 / s), lands exactly on m then (its error is ~2^-46 relative).  cvt then rounds q1 to nearest even as it
// would the correctly rounded quotient.  s comes from the group's own max |x|, so
// |x / s| stays below ~12 and nothing overflows.  The correction turns x = -0
// into +0, so the sign is taken from x (as the quotient's is).  Two values per
// call, on paired FP32 instructions; r = 1 / s, ns = -s.
__device__ __forceinline__ void nv_quotient2(float x0, float x1, float r, float ns, float& y0, float& y1) {
  float q0, q1;
  asm("{\n\t.reg .b64 x, rr, nn, q, e;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 rr, {%4, %4};\n\t"
      "mov.b64 nn, {%5, %5};\n\t"
      "mul.rn.f32x2 q, x, rr;\n\t"
      "fma.rn.f32x2 e, q, nn, x;\n\t"
      "fma.rn.f32x2 q, e, rr, q;\n\t"
      "mov.b64 {%0, %1}, q;\n\t}"
      : "=f"(q0), "=f"(q1)
      : "f"(x0), "f"(x1), "f"(r), "f"(ns));
  y0 = copysignf(q0, x0);
  y1 = copysignf(q1, x1);
}

// 2^-e as an FP32 value, e in [-127, 127].
__device__ __forceinline__ float pow2_neg(int e) {
  const int be = 127 - e;
  return be >= 1 ? __uint_as_float(static_cast<uint32_t>(be) << 23) : __uint_as_float(0x00400000u);
}

template <bool NV>
__global__ void __launch_bounds__(256) quantize_fp4_kernel(const __nv_bfloat16* __restrict__ X,
                                                           uint8_t* __restrict__ Xq,
                                                           uint32_t* __restrict__ SF, int R, int K) {
  ptx::griddep_wait();                          // X may come from the previous kernel
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int nchunk = (K + 511) / 512;
  const int ld = (R + 3) / 4 * 4;
  const int nw = (K / (NV ? 16 : 32) + 3) / 4;  // scale words per row
  const long long item = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  if (item >= static_cast<long long>(ld) * nchunk) return;      // warp-uniform
  const int r = static_cast<int>(item / nchunk);
  const int c = static_cast<int>(item - static_cast<long long>(r) * nchunk);
  const int col0 = c * 512 + 16 * lane;
  const bool active = r < R && col0 < K;
  float f[16];
  float amax = 0.0f;
  if (active) {
    const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<size_t>(r) * K + col0);
    const uint4 w0 = __ldg(src), w1 = __ldg(src + 1);
    const uint32_t u[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[2 * i] = __uint_as_float(u[i] << 16);
      f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
  if (!NV) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));   // 32-element group: two lanes
  uint32_t byte;
  float mul = 1.0f, s = 1.0f, rs = 1.0f;
  if (NV) {
    byte = amax == 0.0f ? 0x38u : static_cast<uint32_t>(ptx::cvt_e4m3x2(__fdiv_rn(amax, 6.0f), 0.0f) & 0xFFu);
    s = ptx::e4m3_value(byte);
    rs = s == 0.0f ? 0.0f : __frcp_rn(s);
  } else {
    const int e = mx_exponent(amax);
    byte = static_cast<uint32_t>(e + 127);
    mul = pow2_neg(e);
  }
  if (active) {
    float q0[8], q1[8];
    if (NV) {
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        nv_quotient2(f[i], f[i + 1], rs, -s, q0[i], q0[i + 1]);
        nv_quotient2(f[8 + i], f[9 + i], rs, -s, q1[i], q1[i + 1]);
      }
      if (s == 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q0[i] = q1[i] = 0.0f;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        q0[i] = f[i] * mul;
        q1[i] = f[8 + i] * mul;
      }
    }
    *reinterpret_cast<uint2*>(Xq + static_cast<size_t>(r) * (K / 2) + col0 / 2) =
        make_uint2(ptx::cvt_e2m1x8(q0), ptx::cvt_e2m1x8(q1));
  }
  // scale bytes -> words: NVFP4 group = lane, word = 4 lanes; MXFP4 group = lane
  // pair, word = 8 lanes.  Inactive lanes (padding rows, past K) contribute 0.
  uint32_t v;
  int w;
  bool writer;
  if (NV) {
    v = active ? byte << (8 * (lane & 3)) : 0u;
    v |= __shfl_xor_sync(0xffffffffu, v, 1);
    v |= __shfl_xor_sync(0xffffffffu, v, 2);
    w = c * 8 + lane / 4;
    writer = (lane & 3) == 0;
  } else {
    v = (active && (lane & 1) == 0) ? byte << (8 * ((lane >> 1) & 3)) : 0u;
    v |= __shfl_xor_sync(0xffffffffu, v, 1);
    v |= __shfl_xor_sync(0xffffffffu, v, 2);
    v |= __shfl_xor_sync(0xffffffffu, v, 4);
    w = c * 4 + lane / 8;
    writer = (lane & 7) == 0;
  }
  if (writer && w < nw) SF[static_cast<size_t>(w) * ld + r] = v;
}

template <bool NV>
int launch_fp4(const void* X, void* Xq, void* SF, int R, int K, cudaStream_t stream) {
  const long long items = static_cast<long long>((R + 3) / 4 * 4) * ((K + 511) / 512);
  const long long blocks = (items + 7) / 8;
  if (blocks > 0x7FFFFFFFLL) return set_error(2, "quantize_fp4: problem too large");
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_fp4_kernel<NV>, static_cast<const __nv_bfloat16*>(X),
                                           static_cast<uint8_t*>(Xq), static_cast<uint32_t*>(SF), R, K);
  if (e != cudaSuccess) return set_error(4, "quantize_fp4 launch: %s", cudaGetErrorString(e));
  return 0;
}

}  // namespace

int launch_quantize_fp4(const void* X, void* Xq, void* SF, int R, int K, int fmt, cudaStream_t stream) {
  return fmt ? launch_fp4<true>(X, Xq, SF, R, K, stream) : launch_fp4<false>(X, Xq, SF, R, K, stream);
}

}  // namespace fgf8

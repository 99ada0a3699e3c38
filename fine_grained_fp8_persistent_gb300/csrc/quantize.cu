// quantize.cu -- BF16 -> E4M3 quantization with fine-grained scales.
//
// "DeepGEMM dissected", section on fine-grained quantization: activations are
// grouped 1 x 128 (one token, 128 channels), weights 128 x 128; each group's
// scale comes online from its max |x| and maps it to the top of the E4M3 range
// (448), s = amax / 448 (the page's worked example s = 40/448).  With
// power-of-two (UE8M0) scales, the exponent is rounded up so nothing saturates.
//
// Both kernels are HBM-bound streams: 2 bytes read and 1 byte written per
// element plus the small scale tables.  Loads are 16-byte vectors, each warp
// covers a contiguous 1 KB (1x128) or 256 B row segments (128x128), and the
// packed UE8M0 words are assembled on chip so each scale word is written once.
#include <cuda_bf16.h>

#include <cstdint>

#include "fgf8_internal.h"
#include "ptx.cuh"

namespace fgf8 {
namespace {

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

// 2^-e as an FP32 value, e in [-127, 127].
__device__ __forceinline__ float exp2_neg(int e) {
  const int be = 127 - e;
  return be >= 1 ? __uint_as_float(static_cast<uint32_t>(be) << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// Quantize 8 values with the group's scale; returns 8 packed E4M3 bytes.
__device__ __forceinline__ uint2 quant8(const float (&f)[8], bool f32_scale, float s,
                                        float inv_pow2) {
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = f32_scale ? __fdiv_rn(f[i], s) : f[i] * inv_pow2;
  uint2 r;
  r.x = static_cast<uint32_t>(ptx::cvt_e4m3x2(q[0], q[1])) |
        (static_cast<uint32_t>(ptx::cvt_e4m3x2(q[2], q[3])) << 16);
  r.y = static_cast<uint32_t>(ptx::cvt_e4m3x2(q[4], q[5])) |
        (static_cast<uint32_t>(ptx::cvt_e4m3x2(q[6], q[7])) << 16);
  return r;
}

// One warp per (row m, group of four 128-wide K blocks); each warp handles two
// such items per iteration with all four 16-byte loads in flight before any
// arithmetic.  Lane l covers elements [16 l, 16 l + 16) of a 512-element chunk,
// so lanes 8j..8j+7 own K block j of the group.
constexpr int kItemsPerIter = 2;

__device__ __forceinline__ void quant_item_1x128(const float (&f0)[8], const float (&f1)[8],
                                                 bool active, int lane, int ue8m0, int m, int M,
                                                 int qw, int kb, int nkb, int K, int ld,
                                                 uint8_t* __restrict__ Xq, void* __restrict__ SF) {
  float amax = 0.0f;
  if (active) {
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(f0[i]), fabsf(f1[i])));
  }
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  float s = 1.0f, inv = 1.0f;
  int e = 0;
  if (ue8m0) {
    e = ue8m0_exponent(amax);
    inv = exp2_neg(e);
  } else if (amax != 0.0f) {
    s = __fdiv_rn(amax, kE4M3Max);
  }
  if (active) {
    const uint2 lo = quant8(f0, !ue8m0, s, inv), hi = quant8(f1, !ue8m0, s, inv);
    *reinterpret_cast<uint4*>(Xq + static_cast<size_t>(m) * K + static_cast<size_t>(qw) * 512 +
                              16 * lane) = make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  if (ue8m0) {
    // gather the four exponent bytes of the group into one little-endian word
    const uint32_t byte = active ? static_cast<uint32_t>(e + 127) : 0u;
    const uint32_t b1 = __shfl_sync(0xffffffffu, byte, 8);
    const uint32_t b2 = __shfl_sync(0xffffffffu, byte, 16);
    const uint32_t b3 = __shfl_sync(0xffffffffu, byte, 24);
    if (lane == 0)
      reinterpret_cast<uint32_t*>(SF)[static_cast<size_t>(qw) * ld + m] =
          byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
  } else if ((lane & 7) == 0 && kb < nkb) {
    reinterpret_cast<float*>(SF)[static_cast<size_t>(kb) * ld + m] = (m < M) ? s : 0.0f;
  }
}

__global__ void __launch_bounds__(256) quantize_1x128_kernel(const __nv_bfloat16* __restrict__ X,
                                                             uint8_t* __restrict__ Xq,
                                                             void* __restrict__ SF, int M, int K,
                                                             int ue8m0) {
  const int lane = threadIdx.x & 31;
  const int nkb = K / 128;
  const int kq = (nkb + 3) / 4;
  const int ld = (M + 3) / 4 * 4;
  const long long items = static_cast<long long>(ld) * kq;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const int j = lane >> 3;                     // K block within the group
  for (long long base = (static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32) *
                        kItemsPerIter;
       base < items; base += warps * kItemsPerIter) {
    int m[kItemsPerIter], qw[kItemsPerIter], kb[kItemsPerIter];
    bool active[kItemsPerIter];
    uint4 w[kItemsPerIter][2];
#pragma unroll
    for (int u = 0; u < kItemsPerIter; ++u) {
      const long long it = base + u;
      m[u] = static_cast<int>(it / kq);
      qw[u] = static_cast<int>(it - static_cast<long long>(m[u]) * kq);
      kb[u] = 4 * qw[u] + j;
      active[u] = it < items && m[u] < M && kb[u] < nkb;
      if (active[u]) {
        const uint4* src = reinterpret_cast<const uint4*>(
            X + static_cast<size_t>(m[u]) * K + static_cast<size_t>(qw[u]) * 512 + 16 * lane);
        w[u][0] = __ldg(src);
        w[u][1] = __ldg(src + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < kItemsPerIter; ++u) {
      if (base + u >= items) break;             // warp-uniform
      float f0[8], f1[8];
      if (active[u]) {
        unpack8(w[u][0], f0);
        unpack8(w[u][1], f1);
      }
      quant_item_1x128(f0, f1, active[u], lane, ue8m0, m[u], M, qw[u], kb[u], nkb, K, ld, Xq, SF);
    }
  }
}

// One CTA per (expert g, 128-row block nb, group of four 128-wide K blocks), in
// two passes over the 128 x 512 region so that every warp reads whole 1 KB row
// segments: pass 1 finds each K block's max |w| (warp w takes rows w, w+8, ...,
// lane l the 16 columns at 16 l, so lanes 8j..8j+7 cover K block j), pass 2
// re-reads the region (an L2 hit: at most four such CTAs per SM keep the
// working set well inside L2) and quantizes it with the block scales.
__global__ void __launch_bounds__(256, 4) quantize_128x128_kernel(const __nv_bfloat16* __restrict__ W,
                                                                  uint8_t* __restrict__ Wq,
                                                                  void* __restrict__ SF, int N, int K,
                                                                  int ue8m0) {
  __shared__ float warp_max[8][4];
  const int nkb = K / 128;
  const int kq = (nkb + 3) / 4;
  const int nnb = (N + 127) / 128;
  const int ldn = (N + 3) / 4 * 4;
  const int qw = blockIdx.x % kq;
  const int nb = (blockIdx.x / kq) % nnb;
  const int g = blockIdx.x / (kq * nnb);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane >> 3;
  const int kb = 4 * qw + j;
  const bool col_ok = kb < nkb;
  const size_t col = static_cast<size_t>(qw) * 512 + 16 * lane;
  const __nv_bfloat16* Wg = W + static_cast<size_t>(g) * N * K;
  uint8_t* Wqg = Wq + static_cast<size_t>(g) * N * K;
  const int row0 = nb * 128 + warp;

  // pass 1: block maxima
  float amax = 0.0f;
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int n = row0 + 8 * i;
    if (col_ok && n < N) {
      const uint4* src = reinterpret_cast<const uint4*>(Wg + static_cast<size_t>(n) * K + col);
      float f0[8], f1[8];
      unpack8(__ldg(src), f0);
      unpack8(__ldg(src + 1), f1);
#pragma unroll
      for (int x = 0; x < 8; ++x) amax = fmaxf(amax, fmaxf(fabsf(f0[x]), fabsf(f1[x])));
    }
  }
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((lane & 7) == 0) warp_max[warp][j] = amax;
  __syncthreads();
  amax = warp_max[0][j];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, warp_max[w][j]);

  float s = 1.0f, inv = 1.0f;
  int e = 0;
  if (ue8m0) {
    e = ue8m0_exponent(amax);
    inv = exp2_neg(e);
  } else if (amax != 0.0f) {
    s = __fdiv_rn(amax, kE4M3Max);
  }

  // pass 2: quantize
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int n = row0 + 8 * i;
    if (col_ok && n < N) {
      const uint4* src = reinterpret_cast<const uint4*>(Wg + static_cast<size_t>(n) * K + col);
      float f0[8], f1[8];
      unpack8(__ldg(src), f0);
      unpack8(__ldg(src + 1), f1);
      const uint2 lo = quant8(f0, !ue8m0, s, inv), hi = quant8(f1, !ue8m0, s, inv);
      *reinterpret_cast<uint4*>(Wqg + static_cast<size_t>(n) * K + col) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
  }

  // scale table
  if (!ue8m0) {
    if (warp == 0 && (lane & 7) == 0 && col_ok)
      reinterpret_cast<float*>(SF)[(static_cast<size_t>(g) * nnb + nb) * nkb + kb] = s;
  } else {
    const uint32_t byte = col_ok ? static_cast<uint32_t>(e + 127) : 0u;
    const uint32_t b0 = __shfl_sync(0xffffffffu, byte, 0);
    const uint32_t b1 = __shfl_sync(0xffffffffu, byte, 8);
    const uint32_t b2 = __shfl_sync(0xffffffffu, byte, 16);
    const uint32_t b3 = __shfl_sync(0xffffffffu, byte, 24);
    const uint32_t word = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    if (threadIdx.x < 128) {
      const int n = nb * 128 + threadIdx.x;
      if (n < ldn)
        reinterpret_cast<uint32_t*>(SF)[(static_cast<size_t>(g) * kq + qw) * ldn + n] =
            (n < N) ? word : 0u;
    }
  }
}

}  // namespace

int launch_quantize_1x128(const void* X, void* Xq, void* SF, int M, int K, int fmt,
                          cudaStream_t stream) {
  const int kq = (K / 128 + 3) / 4;
  const long long items = static_cast<long long>((M + 3) / 4 * 4) * kq;
  const long long blocks_needed = (items + 8 * kItemsPerIter - 1) / (8 * kItemsPerIter);
  const long long cap = static_cast<long long>(device_sm_count()) * 16;
  const int grid = static_cast<int>(blocks_needed < cap ? blocks_needed : cap);
  quantize_1x128_kernel<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(X),
                                                  static_cast<uint8_t*>(Xq), SF, M, K, fmt);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return set_error(4, "quantize_1x128 launch: %s", cudaGetErrorString(err));
  return 0;
}

int launch_quantize_128x128(const void* W, void* Wq, void* SF, int G, int N, int K, int fmt,
                            cudaStream_t stream) {
  const int kq = (K / 128 + 3) / 4;
  const long long grid = static_cast<long long>(G) * ((N + 127) / 128) * kq;
  if (grid > 0x7FFFFFFFLL) return set_error(2, "quantize_128x128: problem too large");
  quantize_128x128_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(W), static_cast<uint8_t*>(Wq), SF, N, K, fmt);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess)
    return set_error(4, "quantize_128x128 launch: %s", cudaGetErrorString(err));
  return 0;
}

}  // namespace fgf8

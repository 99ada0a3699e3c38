// quantize.cu -- BF16 -> E4M3 quantization with fine-grained scales.
//
// "DeepGEMM dissected", section on fine-grained quantization: activations are
// grouped 1 x 128 (one token, 128 channels), weights 128 x 128; each group's
// scale comes online from its max |x| and maps it to the top of the E4M3 range
// (448), s = amax / 448 (the page's worked example s = 40/448).  With
// power-of-two (UE8M0) scales, the exponent is rounded up so nothing saturates.
//
// Both kernels are HBM-bound streams: 2 bytes read and 1 byte written per
// element plus the small scale tables, each input byte read once.  Loads are
// 16-byte vectors; a warp covers a contiguous 1 KB (1x128) or two 256-byte row
// segments (128x128).
#include <cuda_bf16.h>

#include <cstdint>
#include <cstring>

#include "fgf8_internal.h"
#include "ptx.cuh"
#include "quant_common.cuh"

namespace fgf8 {
namespace {

using quant::exp2_neg;
using quant::kE4M3Max;
using quant::ue8m0_exponent;

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// Quantize 8 values with the group's scale; returns 8 packed E4M3 bytes.  FP32
// scales divide (x / s, rounded to nearest, by quant::div_by_scale2 with inv the
// scale's reciprocal from quant::scale_reciprocal); power-of-two scales multiply
// by the exact 2^-e (inv).  The format is a template parameter so each kernel
// carries only its own arithmetic.
template <bool UE8M0>
__device__ __forceinline__ uint2 quant8(const float (&f)[8], float s, float inv) {
  float q[8];
  if (UE8M0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = f[i] * inv;
  } else {
#pragma unroll
    for (int i = 0; i < 8; i += 2) quant::div_by_scale2(f[i], f[i + 1], s, inv, q[i], q[i + 1]);
  }
  uint2 r;
  r.x = static_cast<uint32_t>(ptx::cvt_e4m3x2(q[0], q[1])) |
        (static_cast<uint32_t>(ptx::cvt_e4m3x2(q[2], q[3])) << 16);
  r.y = static_cast<uint32_t>(ptx::cvt_e4m3x2(q[4], q[5])) |
        (static_cast<uint32_t>(ptx::cvt_e4m3x2(q[6], q[7])) << 16);
  return r;
}

// One warp per item (row m, group of four 128-wide K blocks).  Lane l covers
// elements [16 l, 16 l + 16) of the item's 512-element chunk, so lanes 8j..8j+7
// own K block j.  The grid holds as many warps as are resident at once; each warp
// walks a contiguous range of items two at a time and issues the loads of the
// next pair before it quantizes the current one (four 16-byte loads in flight per
// lane), so the stream never waits on a cold load between items.
struct Item1x128 {
  int m, qw, kb;
  bool valid, active;
};

__device__ __forceinline__ Item1x128 item_1x128(int it, int end, int kq, int M, int nkb, int j) {
  Item1x128 r;
  r.valid = it < end;
  r.m = it / kq;
  r.qw = it - r.m * kq;
  r.kb = 4 * r.qw + j;
  r.active = r.valid && r.m < M && r.kb < nkb;
  return r;
}

__device__ __forceinline__ void load_1x128(const __nv_bfloat16* __restrict__ X, const Item1x128& t,
                                           int K, int lane, uint4 (&w)[2]) {
  if (t.active) {
    const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<size_t>(t.m) * K +
                                                      static_cast<size_t>(t.qw) * 512 + 16 * lane);
    w[0] = __ldg(src);
    w[1] = __ldg(src + 1);
  }
}

template <bool UE8M0>
__device__ __forceinline__ void quant_item_1x128(const uint4 (&w)[2], const Item1x128& t, int lane,
                                                 int M, int nkb, int K, int ld,
                                                 uint8_t* __restrict__ Xq, void* __restrict__ SF) {
  float f0[8], f1[8];
  float amax = 0.0f;
  if (t.active) {
    unpack8(w[0], f0);
    unpack8(w[1], f1);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(f0[i]), fabsf(f1[i])));
  }
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  float s = 1.0f, inv = 1.0f;
  int e = 0;
  if (UE8M0) {
    e = ue8m0_exponent(amax);
    inv = exp2_neg(e);
  } else {
    if (amax != 0.0f) s = __fdiv_rn(amax, kE4M3Max);
    inv = quant::scale_reciprocal(s);
  }
  if (t.active) {
    const uint2 lo = quant8<UE8M0>(f0, s, inv), hi = quant8<UE8M0>(f1, s, inv);
    *reinterpret_cast<uint4*>(Xq + static_cast<size_t>(t.m) * K + static_cast<size_t>(t.qw) * 512 +
                              16 * lane) = make_uint4(lo.x, lo.y, hi.x, hi.y);
  }
  if (UE8M0) {
    // gather the four exponent bytes of the group into one little-endian word
    const uint32_t byte = t.active ? static_cast<uint32_t>(e + 127) : 0u;
    const uint32_t b1 = __shfl_sync(0xffffffffu, byte, 8);
    const uint32_t b2 = __shfl_sync(0xffffffffu, byte, 16);
    const uint32_t b3 = __shfl_sync(0xffffffffu, byte, 24);
    if (lane == 0)
      reinterpret_cast<uint32_t*>(SF)[static_cast<size_t>(t.qw) * ld + t.m] =
          byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
  } else if ((lane & 7) == 0 && t.kb < nkb) {
    reinterpret_cast<float*>(SF)[static_cast<size_t>(t.kb) * ld + t.m] = (t.m < M) ? s : 0.0f;
  }
}

template <bool UE8M0>
__global__ void __launch_bounds__(256, 3) quantize_1x128_kernel(const __nv_bfloat16* __restrict__ X,
                                                             uint8_t* __restrict__ Xq,
                                                             void* __restrict__ SF, int M, int K,
                                                             int per_warp) {
  ptx::griddep_wait();                          // X may come from the previous kernel
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int nkb = K / 128;
  const int kq = (nkb + 3) / 4;
  const int ld = (M + 3) / 4 * 4;
  const int items = ld * kq;
  const int j = lane >> 3;                     // K block within the group
  const int gw = static_cast<int>(blockIdx.x) * (blockDim.x / 32) + static_cast<int>(threadIdx.x / 32);
  const long long first = static_cast<long long>(gw) * per_warp;
  if (first >= items) return;                  // warp-uniform
  int it = static_cast<int>(first);
  const int end = min(it + per_warp, items);
  uint4 cur[2][2], nxt[2][2];
  Item1x128 tc[2], tn[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    tc[u] = item_1x128(it + u, end, kq, M, nkb, j);
    load_1x128(X, tc[u], K, lane, cur[u]);
  }
  for (; it < end; it += 2) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      tn[u] = item_1x128(it + 2 + u, end, kq, M, nkb, j);
      load_1x128(X, tn[u], K, lane, nxt[u]);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (tc[u].valid) quant_item_1x128<UE8M0>(cur[u], tc[u], lane, M, nkb, K, ld, Xq, SF);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      tc[u] = tn[u];
      cur[u][0] = nxt[u][0];
      cur[u][1] = nxt[u][1];
    }
  }
}

// One CTA (256 threads) per (expert g, 128-row block nb, 128-wide K block kb), in
// a single pass: the 32 KB block is loaded into registers (thread t holds the 8
// columns at 8 (t % 16) of rows 16 i + t / 16, i = 0..7, so a half-warp reads one
// 256-byte row segment), reduced to its max |w|, quantized from the registers and
// written.  Weights are read from HBM exactly once.  UE8M0 exponents are written
// as single bytes straight into their packed words (byte kb % 4 of the word of
// each row), so the four CTAs sharing a word never read-modify-write it.
template <bool UE8M0>
__global__ void __launch_bounds__(256, 3) quantize_128x128_kernel(const __nv_bfloat16* __restrict__ W,
                                                                  uint8_t* __restrict__ Wq,
                                                                  void* __restrict__ SF, int N, int K) {
  __shared__ float warp_max[8];
  ptx::griddep_wait();                          // W may come from the previous kernel
  ptx::griddep_launch_dependents();
  const int nkb = K / 128;
  const int nnb = (N + 127) / 128;
  const int kb = static_cast<int>(blockIdx.x % nkb);
  const int nb = static_cast<int>((blockIdx.x / nkb) % nnb);
  const int g = static_cast<int>(blockIdx.x / (static_cast<unsigned>(nkb) * nnb));
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int rsub = t >> 4;
  const size_t col = static_cast<size_t>(kb) * 128 + 8 * (t & 15);
  const __nv_bfloat16* Wg = W + static_cast<size_t>(g) * N * K + col;
  uint8_t* Wqg = Wq + static_cast<size_t>(g) * N * K + col;

  uint4 w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int n = nb * 128 + 16 * i + rsub;
    w[i] = n < N ? __ldg(reinterpret_cast<const uint4*>(Wg + static_cast<size_t>(n) * K))
                 : make_uint4(0u, 0u, 0u, 0u);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float f[8];
    unpack8(w[i], f);
#pragma unroll
    for (int x = 0; x < 8; ++x) amax = fmaxf(amax, fabsf(f[x]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_max[i]);

  float s = 1.0f, inv = 1.0f;
  int e = 0;
  if (UE8M0) {
    e = ue8m0_exponent(amax);
    inv = exp2_neg(e);
  } else {
    if (amax != 0.0f) s = __fdiv_rn(amax, kE4M3Max);
    inv = quant::scale_reciprocal(s);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int n = nb * 128 + 16 * i + rsub;
    if (n < N) {
      float f[8];
      unpack8(w[i], f);
      *reinterpret_cast<uint2*>(Wqg + static_cast<size_t>(n) * K) = quant8<UE8M0>(f, s, inv);
    }
  }

  // scale table
  if (!UE8M0) {
    if (t == 0) reinterpret_cast<float*>(SF)[(static_cast<size_t>(g) * nnb + nb) * nkb + kb] = s;
  } else if (t < 128) {
    const int kq = (nkb + 3) / 4;
    const int ldn = (N + 3) / 4 * 4;
    const int n = nb * 128 + t;
    if (n < ldn) {
      uint8_t* word = reinterpret_cast<uint8_t*>(SF) +
                      ((static_cast<size_t>(g) * kq + kb / 4) * ldn + n) * 4;
      word[kb & 3] = n < N ? static_cast<uint8_t>(e + 127) : static_cast<uint8_t>(0);
      // the last K block also clears the bytes of the K blocks past the end
      if (kb == nkb - 1)
        for (int b = (kb & 3) + 1; b < 4; ++b) word[b] = 0;
    }
  }
}

}  // namespace

namespace {

// 256-thread launch, with programmatic stream serialization when enabled.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <bool UE8M0>
int launch_1x128(const void* X, void* Xq, void* SF, int M, int K, cudaStream_t stream) {
  const int kq = (K / 128 + 3) / 4;
  const long long items = static_cast<long long>((M + 3) / 4 * 4) * kq;
  if (items > 0x7F000000LL) return set_error(2, "quantize_1x128: problem too large");
  static int blocks_per_sm = 0;
  if (blocks_per_sm == 0) {
    int b = 0;
    const cudaError_t e =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, quantize_1x128_kernel<UE8M0>, 256, 0);
    if (e != cudaSuccess || b <= 0) return set_error(4, "quantize_1x128 occupancy: %s", cudaGetErrorString(e));
    blocks_per_sm = b;
  }
  // one resident wave of warps, each with a contiguous range of items
  const long long warps_cap = static_cast<long long>(device_sm_count()) * blocks_per_sm * 8;
  const long long warps = items < warps_cap ? items : warps_cap;
  const long long per_warp = (items + warps - 1) / warps;
  const long long grid = (warps + 7) / 8;
  const cudaError_t err =
      launch_pdl(quantize_1x128_kernel<UE8M0>, static_cast<unsigned>(grid), stream,
                 static_cast<const __nv_bfloat16*>(X), static_cast<uint8_t*>(Xq), SF, M, K, static_cast<int>(per_warp));
  if (err != cudaSuccess) return set_error(4, "quantize_1x128 launch: %s", cudaGetErrorString(err));
  return 0;
}

template <bool UE8M0>
int launch_128x128(const void* W, void* Wq, void* SF, int G, int N, int K, cudaStream_t stream) {
  const long long grid = static_cast<long long>(G) * ((N + 127) / 128) * (K / 128);
  if (grid > 0x7FFFFFFFLL) return set_error(2, "quantize_128x128: problem too large");
  const cudaError_t err = launch_pdl(quantize_128x128_kernel<UE8M0>, static_cast<unsigned>(grid), stream,
                                     static_cast<const __nv_bfloat16*>(W), static_cast<uint8_t*>(Wq), SF, N, K);
  if (err != cudaSuccess)
    return set_error(4, "quantize_128x128 launch: %s", cudaGetErrorString(err));
  return 0;
}

}  // namespace

int launch_quantize_1x128(const void* X, void* Xq, void* SF, int M, int K, int fmt,
                          cudaStream_t stream) {
  return fmt ? launch_1x128<true>(X, Xq, SF, M, K, stream) : launch_1x128<false>(X, Xq, SF, M, K, stream);
}

int launch_quantize_128x128(const void* W, void* Wq, void* SF, int G, int N, int K, int fmt,
                            cudaStream_t stream) {
  return fmt ? launch_128x128<true>(W, Wq, SF, G, N, K, stream)
             : launch_128x128<false>(W, Wq, SF, G, N, K, stream);
}

}  // namespace fgf8

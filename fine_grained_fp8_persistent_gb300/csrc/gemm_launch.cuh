// gemm_launch.cuh -- host-side launch of one GEMM kernel instantiation, tensor-map
// set-up and the tile-shape heuristic shared by the launcher translation units.
#pragma once
#include <cstring>

#include "gemm_kernel.cuh"

namespace fgf8 {

// Persistent grid: one CTA per SM (the SMEM footprint keeps it at one), never
// more CTAs than tiles.
inline int persistent_grid(long long tiles) {
  const long long sms = device_sm_count();
  if (tiles <= 0) return 1;
  return static_cast<int>(tiles < sms ? tiles : sms);
}

template <Kind KIND, Sched SCHED, int BN, int STAGES>
int launch_instance(const GemmArgs& a, const TensorMaps& tm, int grid, cudaStream_t stream) {
  using C = GemmCfg<KIND, SCHED, BN, STAGES>;
  auto* fn = &gemm_kernel<KIND, SCHED, BN, STAGES>;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (C::SMEM_BYTES > device_max_smem_optin())
    return set_error(2, "tile %dx%d needs %d bytes of shared memory", C::BM, BN, C::SMEM_BYTES);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return set_error(4, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured[dev] = true;
  }
  fn<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tm.a, tm.b, tm.sfa, tm.sfb, a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(4, "gemm launch: %s", cudaGetErrorString(e));
  return 0;
}

// Tiles of the problem for a given BN (masked: the upper bound with every expert full).
inline long long tile_count(const GemmArgs& a, Sched s, int bn) {
  const long long mt = (a.M + 127) / 128;
  const long long nt = (a.N + bn - 1) / bn;
  return (s == Sched::Masked ? a.G : 1) * mt * nt;
}

// Pick the widest tile that does not cost extra waves: estimated time is
// waves * (BN + 32), where 32 stands for the per-tile cost that does not scale
// with BN (the A tile, the epilogue drain).  Wide tiles make the MMA and the
// B traffic per output cheaper; narrow tiles spread a skinny problem over more
// SMs (the DeepGEMM page's unaligned-BLOCK_N argument: 112 vs 128 blocks on 132
// SMs).
inline int pick_bn(const GemmArgs& a, Sched s, const int* cands, int n) {
  const long long sms = device_sm_count();
  int best = cands[0];
  long long best_cost = -1;
  for (int i = 0; i < n; ++i) {
    const long long tiles = tile_count(a, s, cands[i]);
    const long long waves = (tiles + sms - 1) / sms;
    const long long cost = waves * (cands[i] + 32);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = cands[i];
    }
  }
  return best;
}

// A and B operand maps: K-major rows of 128 bytes per stage, 128-byte swizzle.
inline int make_operand_maps(TensorMaps& tm, CUtensorMapDataType dt, int elem_bytes, const void* A,
                             long long a_rows, const void* B, long long b_rows, int K, int bn) {
  std::memset(&tm, 0, sizeof(tm));
  const uint32_t bk = 128 / elem_bytes;
  if (!encode_tmap_2d(&tm.a, dt, A, K, a_rows, static_cast<uint64_t>(K) * elem_bytes, bk, 128, true))
    return 4;
  if (!encode_tmap_2d(&tm.b, dt, B, K, b_rows, static_cast<uint64_t>(K) * elem_bytes, bk, bn, true))
    return 4;
  return 0;
}

}  // namespace fgf8

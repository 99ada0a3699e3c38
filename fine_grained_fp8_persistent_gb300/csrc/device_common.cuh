// device_common.cuh -- descriptors, bounded waits and the tile schedulers shared by
// the GEMM kernels.
#pragma once
#include <cstdint>

#include "fgf8_internal.h"
#include "ptx.cuh"

namespace fgf8 {

// ---------------------------------------------------------------------------
// Instruction descriptors ("GPU GEMM part 4: tcgen05 & Blackwell", section 3.3
// bit table; the block-scaled variant puts b_sf_id at bits 4-5, the scale format
// at bit 23 and a_sf_id at bits 29-30).  M = 128 (one CTA), K-major A and B.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr uint32_t idesc_dense(uint32_t a_fmt, uint32_t b_fmt, uint32_t n,
                                                   uint32_t m) {
  return (1u << 4)            // c_format: F32 accumulator
         | (a_fmt << 7)       // a_format
         | (b_fmt << 10)      // b_format
         | ((n >> 3) << 17)   // n_dim = N/8
         | ((m >> 4) << 24);  // m_dim = M/16
}
// kind::f16 formats: 0 = F16, 1 = BF16.  kind::f8f6f4 / mxf8f6f4: 0 = E4M3.
__host__ __device__ constexpr uint32_t idesc_mxf8(uint32_t n, uint32_t m, uint32_t a_sf_id,
                                                  uint32_t b_sf_id) {
  return (b_sf_id << 4)       // b_sf_id
         | (0u << 7)          // a_format E4M3
         | (0u << 10)         // b_format E4M3
         | ((n >> 3) << 17)   // n_dim
         | (1u << 23)         // scale_format: E8M0
         | ((m >> 4) << 24)   // m_dim
         | (a_sf_id << 29);   // a_sf_id
}

// 4-bit block-scaled (kind::mxf4nvf4): E2M1 A and B (format code 1), scale
// format bit 23 (1 = E8M0 for MXFP4, 0 = E4M3 for NVFP4); the sf ids are ORed in
// per instruction (b_sf_id bits 4-5, a_sf_id bits 29-30).
__host__ __device__ constexpr uint32_t idesc_fp4(uint32_t n, uint32_t m, bool e8m0_scales) {
  return (1u << 7)                        // a_format E2M1
         | (1u << 10)                     // b_format E2M1
         | ((n >> 3) << 17)               // n_dim
         | ((e8m0_scales ? 1u : 0u) << 23)  // scale_format
         | ((m >> 4) << 24);              // m_dim
}

// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor (same page, section 3.4): start address,
// leading and stride byte offsets in 16-byte units, version 1 at bits 46-47,
// layout type at bits 61-63 (2 = 128-byte swizzle, 0 = none).
// K-major operand tiles written by TMA with 128-byte swizzle: rows of 128 bytes,
// 8-row groups 1024 bytes apart (SBO = 1024); LBO unused inside one swizzle atom.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;             // LBO (ignored for this layout)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;     // SBO
  d |= static_cast<uint64_t>(1u) << 46;             // version
  d |= static_cast<uint64_t>(2u) << 61;             // SWIZZLE_128B
  return d;
}
// ---------------------------------------------------------------------------
// Persistent tile schedulers.  A CTA walks tiles blockIdx.x, blockIdx.x+grid, ...
// (the static round-robin of the DeepGEMM page's scheduler section); every role
// of the CTA walks the same sequence, so they agree without communicating.
// ---------------------------------------------------------------------------
struct Tile {
  int m_blk;      // M block (within the expert for masked)
  int n_blk;      // N block
  int group;      // expert (0 for dense)
  int a_row0;     // first row of the A tile in the 2-D view of A
  int b_row0;     // first row of the B tile in the 2-D view of B
  int row_limit;  // rows >= row_limit (within the tile's M range) are not stored
};

// Dense: raster of the m x n tile grid in bands of `band_n` N-blocks; inside a
// band the N index runs fastest, then the next M block (so tiles running at the
// same time share A rows and a narrow band of B rows in L2).
__device__ __forceinline__ void dense_tile(int t, int num_m, int num_n, int band_n, int& m,
                                           int& n) {
  const int per_band = band_n * num_m;
  const int band = t / per_band;
  const int in_band = t - band * per_band;
  const int width = min(band_n, num_n - band * band_n);
  m = in_band / width;
  n = band * band_n + in_band % width;
}

}  // namespace fgf8

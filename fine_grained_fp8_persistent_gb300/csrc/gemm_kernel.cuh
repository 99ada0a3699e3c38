// gemm_kernel.cuh -- the persistent, warp-specialised NT GEMM for sm_103a.
//
//   D[M,N] = A[M,K] * B[N,K]^T, FP32 accumulation, 16-bit output.
//
// One CTA per SM walks output tiles (BM = 128 rows x BN columns).  Roles:
//   warp 0      TMA producer: fills a STAGES-deep ring of 128-byte-swizzled A/B
//               tiles (and, for MXFP8, the packed UE8M0 scale words) guarded by
//               full/empty mbarriers.
//   warp 1      MMA issuer: one thread issues tcgen05.mma into TMEM and signals
//               completion with tcgen05.commit; the warp also owns TMEM.
//   warps 2..   epilogue (F16, MXF8: 4 warps read the finished accumulator with
//               tcgen05.ld, cast and store) or promotion (F8F32: 8 warps read a
//               per-128-K partial from TMEM and accumulate scale_a*scale_b*partial
//               in FP32 registers on the CUDA cores).
//
// The structure follows the warp-specialised persistent pipeline of
// "TIRx and high-performance GEMM (part 2)" (Step 7: tma2mma / mma2tma /
// mma2ld / ld2mma barriers) and "GPU GEMM part 4: tcgen05 & Blackwell" (section 7:
// producer, single MMA thread, epilogue warps, double-buffered accumulator).
// The FP32-scale promotion follows the main loop of "DeepGEMM dissected"
// (final += scale_a * scale_b * partial once per 128-wide K block), with the
// partial living in TMEM instead of registers.  The UE8M0 path uses the
// block-scaled MMA of "GPU GEMM part 4" section 6.2, with the scale words staged
// SMEM -> tcgen05.cp -> TMEM ("Blackwell Tensor Core: tcgen05.mma", Block-Scaled MMA).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"

namespace fgf8 {

template <Kind KIND, Sched SCHED, int BN_, int STAGES_>
struct GemmCfg {
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  static constexpr int STAGES = STAGES_;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN must be a multiple of 32 in [32,256]");
  static_assert(STAGES >= 2 && STAGES <= 16, "stage count");
  static constexpr bool kMX = KIND == Kind::MXF8;
  static constexpr bool kF32S = KIND == Kind::F8F32;
  // One stage covers one 128-byte swizzle row of K: 64 16-bit or 128 8-bit elements.
  static constexpr int BK = (KIND == Kind::F16) ? 64 : 128;
  static constexpr int MMA_K_BYTES = 32;                 // K=16 (16-bit) or K=32 (8-bit)
  static constexpr int MMAS_PER_STAGE = 128 / MMA_K_BYTES;
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int SFB_ROWS = (BN + 127) / 128 * 128;
  static constexpr int SFA_BYTES = kMX ? BM * 4 : 0;
  static constexpr int SFB_BYTES = kMX ? SFB_ROWS * 4 : 0;
  static constexpr int NUM_EPI_WARPS = kF32S ? 8 : 4;
  static constexpr int THREADS = 64 + 32 * NUM_EPI_WARPS;
  static constexpr int MAX_GROUPS = 1024;

  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
  static constexpr int OFF_BAR = (OFF_SFB + STAGES * SFB_BYTES + 7) / 8 * 8;
  // barrier indices
  static constexpr int BAR_FULL = 0;
  static constexpr int BAR_EMPTY = STAGES;
  static constexpr int BAR_ACC_FULL = 2 * STAGES;       // 2 (accumulators or partials)
  static constexpr int BAR_ACC_EMPTY = 2 * STAGES + 2;  // 2
  static constexpr int BAR_SF_FREE = 2 * STAGES + 4;    // 2
  static constexpr int BAR_DRAIN = 2 * STAGES + 6;      // 1
  static constexpr int NUM_BARS = 2 * STAGES + 7;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // tmem base, abort flag
  static constexpr int OFF_PREFIX = (OFF_MISC + 16 + 15) / 16 * 16;
  static constexpr int PREFIX_BYTES = (SCHED == Sched::Masked) ? (MAX_GROUPS + 1) * 4 : 0;
  static constexpr int SMEM_BYTES = OFF_PREFIX + PREFIX_BYTES + 1024;  // + alignment slack

  // TMEM columns: two accumulator (or partial) buffers, then two scale slots.
  static constexpr int ACC_COLS = 2 * BN;
  static constexpr int SF_SLOT_COLS = 4 + SFB_ROWS / 32;
  static constexpr int SF_COL0 = ACC_COLS;
  static constexpr int TMEM_USED = ACC_COLS + (kMX ? 2 * SF_SLOT_COLS : 0);
  static constexpr int TMEM_ALLOC = TMEM_USED <= 32    ? 32
                                    : TMEM_USED <= 64  ? 64
                                    : TMEM_USED <= 128 ? 128
                                    : TMEM_USED <= 256 ? 256
                                                       : 512;
  static_assert(TMEM_USED <= 512, "TMEM budget");
};

// Transpose 128 scale words in place so that word (32*j + lane) moves to
// (4*lane + j): the 32 x 128-bit layout tcgen05.cp copies, where TMEM lane l,
// column j holds the scale of row 32*j + l.
__device__ __forceinline__ void sf_transpose128(uint32_t* p, uint32_t lane) {
  uint32_t v0 = p[lane], v1 = p[32 + lane], v2 = p[64 + lane], v3 = p[96 + lane];
  __syncwarp();
  *reinterpret_cast<uint4*>(p + 4 * lane) = make_uint4(v0, v1, v2, v3);
  __syncwarp();
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Store 32 consecutive FP32 values of one output row as 16-bit values
// (columns col0 .. col0+31, clipped at N; N is a multiple of 8).
__device__ __forceinline__ void store_chunk32(void* D, size_t row_off, int col0, int N,
                                              const float* v, bool bf16) {
  uint16_t* out = reinterpret_cast<uint16_t*>(D) + row_off;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int col = col0 + 8 * j;
    if (col < N) {
      uint4 w;
      w.x = pack2(v[8 * j + 0], v[8 * j + 1], bf16);
      w.y = pack2(v[8 * j + 2], v[8 * j + 3], bf16);
      w.z = pack2(v[8 * j + 4], v[8 * j + 5], bf16);
      w.w = pack2(v[8 * j + 6], v[8 * j + 7], bf16);
      *reinterpret_cast<uint4*>(out + col) = w;
    }
  }
}

template <Kind KIND, Sched SCHED, int BN, int STAGES>
__global__ void __launch_bounds__(GemmCfg<KIND, SCHED, BN, STAGES>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_sfa,
                const __grid_constant__ CUtensorMap tm_sfb, const GemmArgs args) {
  using C = GemmCfg<KIND, SCHED, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;

  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);
  int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);

  const int M = args.M, N = args.N, K = args.K, G = args.G;
  const int nkb = (K + C::BK - 1) / C::BK;          // stages per tile
  const int num_n = (N + BN - 1) / BN;
  const int num_m = (M + C::BM - 1) / C::BM;        // per expert for masked
  const int kq = (K / 128 + 3) / 4;                 // packed UE8M0 words per row

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(C::BAR_FULL + s), 1);
      ptx::mbar_init(bar(C::BAR_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(bar(C::BAR_ACC_FULL + b), 1);
      ptx::mbar_init(bar(C::BAR_ACC_EMPTY + b), C::NUM_EPI_WARPS);
      ptx::mbar_init(bar(C::BAR_SF_FREE + b), 1);
    }
    ptx::mbar_init(bar(C::BAR_DRAIN), 1);
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if constexpr (SCHED == Sched::Masked) {
    // Tiles per expert: ceil(masked_m[g] / BM) * num_n; an exclusive prefix over
    // experts lets every role map a linear tile index to (expert, m, n) and skip
    // empty experts (the DeepGEMM page's masked-layout scheduler).
    if (warp == 2) {
      int run = 0;
      for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + static_cast<int>(lane);
        int mm = (g < G) ? args.masked_m[g] : 0;
        if (mm < 0 || mm > M) {
          atomicOr(args.status, FGF8_DEVERR_INPUT);
          mm = mm < 0 ? 0 : M;
        }
        int v = (mm + C::BM - 1) / C::BM * num_n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xffffffffu, v, off);
          if (static_cast<int>(lane) >= off) v += o;
        }
        if (g < G) prefix[g + 1] = run + v;
        run += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) prefix[0] = 0;
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TMEM_ALLOC);
    ptx::tmem_relinquish();
    ptx::tc_fence_before();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int num_tiles;
  if constexpr (SCHED == Sched::Masked) num_tiles = prefix[G];
  else num_tiles = num_m * num_n;

  // Tile t -> coordinates.  Returns false for tiles with nothing to compute.
  auto get_tile = [&](int t, Tile& tl) -> bool {
    if constexpr (SCHED == Sched::Dense) {
      int m, n;
      dense_tile(t, num_m, num_n, 16, m, n);
      tl.m_blk = m; tl.n_blk = n; tl.group = 0;
      tl.a_row0 = m * C::BM; tl.b_row0 = n * BN;
      tl.row_limit = M - m * C::BM;
      return true;
    } else if constexpr (SCHED == Sched::Contiguous) {
      int m, n;
      dense_tile(t, num_m, num_n, 16, m, n);
      const int g = __ldg(args.m_indices + m * C::BM);
      if (g < 0 || g >= G) return false;
      tl.m_blk = m; tl.n_blk = n; tl.group = g;
      tl.a_row0 = m * C::BM; tl.b_row0 = g * N + n * BN;
      tl.row_limit = M - m * C::BM;
      return true;
    } else {
      int lo = 0, hi = G - 1;                      // expert g with prefix[g] <= t < prefix[g+1]
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
      }
      const int g = lo;
      int mm = __ldg(args.masked_m + g);
      mm = mm < 0 ? 0 : (mm > M ? M : mm);
      const int mt = (mm + C::BM - 1) / C::BM;
      const int local = t - prefix[g];
      tl.n_blk = local / mt;                        // M blocks of one B tile adjacent
      tl.m_blk = local - tl.n_blk * mt;
      tl.group = g;
      tl.a_row0 = g * M + tl.m_blk * C::BM;
      tl.b_row0 = g * N + tl.n_blk * BN;
      tl.row_limit = mm - tl.m_blk * C::BM;
      return true;
    }
  };

  WaitCtl ctl{abort_flag, args.status, args.timeout_ns, 0};

  if (warp == 0) {
    // ============================================================ TMA producer
    // The whole warp walks the pipeline (so it stays converged); lane 0 issues.
    ctl.role_bit = FGF8_DEVERR_ROLE_PRODUCER;
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_a);
      ptx::prefetch_tmap(&tm_b);
      if constexpr (C::kMX) {
        ptx::prefetch_tmap(&tm_sfa);
        ptx::prefetch_tmap(&tm_sfb);
      }
    }
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      Tile tl;
      if (!get_tile(t, tl)) continue;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!wait_bar_warp(bar(C::BAR_EMPTY + stage), phase ^ 1u, ctl)) { ok = false; break; }
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        if (lane == 0) {
          const bool sf = C::kMX && (kb % 4 == 0);
          const uint32_t bytes = C::A_BYTES + C::B_BYTES + (sf ? (C::BM * 4 + BN * 4) : 0);
          const uint32_t full = bar(C::BAR_FULL + stage);
          ptx::mbar_arrive_expect_tx(full, bytes);
          ptx::tma_load_2d(sbase + C::OFF_A + stage * C::A_BYTES, &tm_a, full, kb * C::BK,
                           tl.a_row0);
          ptx::tma_load_2d(sbase + C::OFF_B + stage * C::B_BYTES, &tm_b, full, kb * C::BK,
                           tl.b_row0);
          if (sf) {
            const int sfa_row = (SCHED == Sched::Masked ? tl.group * kq : 0) + kb / 4;
            ptx::tma_load_2d(sbase + C::OFF_SFA + stage * C::SFA_BYTES, &tm_sfa, full,
                             tl.m_blk * C::BM, sfa_row);
            ptx::tma_load_2d(sbase + C::OFF_SFB + stage * C::SFB_BYTES, &tm_sfb, full,
                             tl.n_blk * BN, tl.group * kq + kb / 4);
          }
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    // Every load issued must have landed before the CTA may exit.
    WaitCtl drain = ctl;
    uint32_t zero = 0;
    drain.abort_flag = &zero;
    for (int s = 0; s < STAGES; ++s)
      if (armed & (1u << s)) wait_bar_warp(bar(C::BAR_FULL + s), (armed_parity >> s) & 1u, drain);
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    ctl.role_bit = FGF8_DEVERR_ROLE_MMA;
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t sf_uses0 = 0u, sf_uses1 = 0u;   // completed uses of each scale slot
    uint32_t gctr = 0;
    bool ok = true;
    // kind::f16 operand format: 0 = F16, 1 = BF16; kind::f8f6f4: 0 = E4M3.
    const uint32_t in_fmt = (KIND == Kind::F16 && args.in_bf16) ? 1u : 0u;
    const uint32_t idesc_plain = idesc_dense(in_fmt, in_fmt, BN, C::BM);
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      Tile tl;
      if (!get_tile(t, tl)) continue;
      if constexpr (!C::kF32S) {
        if (!wait_bar_warp(bar(C::BAR_ACC_EMPTY + acc), acc_phase ^ 1u, ctl)) { ok = false; break; }
        ptx::tc_fence_after();
      }
      uint32_t slot = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!wait_bar_warp(bar(C::BAR_FULL + stage), phase, ctl)) { ok = false; break; }
        if constexpr (C::kF32S) {
          if (!wait_bar_warp(bar(C::BAR_ACC_EMPTY + acc), acc_phase ^ 1u, ctl)) { ok = false; break; }
        }
        ptx::tc_fence_after();
        if constexpr (C::kMX) {
          if (kb % 4 == 0) {
            slot = gctr & 1u;
            const uint32_t uses = slot ? sf_uses1 : sf_uses0;
            if (uses > 0 && !wait_bar_warp(bar(C::BAR_SF_FREE + slot), (uses - 1u) & 1u, ctl)) {
              ok = false;
              break;
            }
            uint32_t* sfa = reinterpret_cast<uint32_t*>(smem + C::OFF_SFA + stage * C::SFA_BYTES);
            uint32_t* sfb = reinterpret_cast<uint32_t*>(smem + C::OFF_SFB + stage * C::SFB_BYTES);
            sf_transpose128(sfa, lane);
#pragma unroll
            for (int c = 0; c < C::SFB_ROWS / 128; ++c) sf_transpose128(sfb + 128 * c, lane);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              ptx::tc_fence_after();
              const uint32_t col = tmem_base + C::SF_COL0 + slot * C::SF_SLOT_COLS;
              ptx::tmem_cp_32x128b_warpx4(col, smem_desc_plain_rows16(ptx::smem_u32(sfa)));
#pragma unroll
              for (int c = 0; c < C::SFB_ROWS / 128; ++c)
                ptx::tmem_cp_32x128b_warpx4(col + 4 + 4 * c,
                                            smem_desc_plain_rows16(ptx::smem_u32(sfb + 128 * c)));
            }
          }
        }
        if (lane == 0) {
          // accumulator buffer of this tile, or (FP32-scale path) partial buffer of this K block
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
          const uint32_t a0 = sbase + C::OFF_A + stage * C::A_BYTES;
          const uint32_t b0 = sbase + C::OFF_B + stage * C::B_BYTES;
#pragma unroll
          for (int k = 0; k < C::MMAS_PER_STAGE; ++k) {
            const uint64_t ad = smem_desc_sw128(a0 + k * C::MMA_K_BYTES);
            const uint64_t bd = smem_desc_sw128(b0 + k * C::MMA_K_BYTES);
            if constexpr (C::kMX) {
              const uint32_t id = idesc_mxf8(BN, C::BM, kb % 4, kb % 4);
              const uint32_t col = tmem_base + C::SF_COL0 + slot * C::SF_SLOT_COLS;
              ptx::mma_mxf8(d_tmem, ad, bd, id, col, col + 4, (kb > 0 || k > 0) ? 1u : 0u);
            } else if constexpr (C::kF32S) {
              ptx::mma_f8(d_tmem, ad, bd, idesc_plain, k > 0 ? 1u : 0u);
            } else {
              ptx::mma_f16(d_tmem, ad, bd, idesc_plain, (kb > 0 || k > 0) ? 1u : 0u);
            }
          }
          ptx::mma_commit(bar(C::BAR_EMPTY + stage));
          if constexpr (C::kMX) {
            if (kb % 4 == 3 || kb == nkb - 1) ptx::mma_commit(bar(C::BAR_SF_FREE + slot));
          }
          if constexpr (C::kF32S) ptx::mma_commit(bar(C::BAR_ACC_FULL + acc));
        }
        __syncwarp();
        if constexpr (C::kMX) {
          if (kb % 4 == 3 || kb == nkb - 1) {
            if (slot) ++sf_uses1; else ++sf_uses0;
            ++gctr;
          }
        }
        if constexpr (C::kF32S) {
          // the partial buffer alternates every K block
          if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if constexpr (!C::kF32S) {
        if (lane == 0) ptx::mma_commit(bar(C::BAR_ACC_FULL + acc));
        __syncwarp();
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
    }
    // Drain: every tcgen05 op this thread issued completes before TMEM is freed.
    if (lane == 0) ptx::mma_commit(bar(C::BAR_DRAIN));
    __syncwarp();
    WaitCtl drain = ctl;
    uint32_t zero = 0;
    drain.abort_flag = &zero;
    wait_bar_warp(bar(C::BAR_DRAIN), 0u, drain);
  } else if constexpr (!C::kF32S) {
    // ============================================================ epilogue
    ctl.role_bit = FGF8_DEVERR_ROLE_EPILOGUE;
    const uint32_t q = warp & 3u;                   // TMEM lane quarter of this warp
    const bool bf16 = args.out_bf16 != 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      Tile tl;
      if (!get_tile(t, tl)) continue;
      if (!wait_bar_warp(bar(C::BAR_ACC_FULL + acc), acc_phase, ctl)) break;
      ptx::tc_fence_after();
      const int r = static_cast<int>(q * 32 + lane);
      bool row_ok = r < tl.row_limit;
      if constexpr (SCHED == Sched::Contiguous) {
        if (row_ok) {
          const int g = __ldg(args.m_indices + tl.a_row0 + r);
          if (g != tl.group) {
            if (g >= 0) atomicOr(args.status, FGF8_DEVERR_INPUT);
            row_ok = false;
          }
        }
      }
      const size_t row_off = static_cast<size_t>(tl.a_row0 + r) * static_cast<size_t>(N);
      const uint32_t taddr = tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + 32u * c, v);
        ptx::tmem_wait_ld();
        if (c == BN / 32 - 1) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(bar(C::BAR_ACC_EMPTY + acc));
        }
        if (row_ok)
          store_chunk32(args.D, row_off, tl.n_blk * BN + 32 * c, N,
                        reinterpret_cast<const float*>(v), bf16);
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  } else {
    // ============================================================ promotion
    ctl.role_bit = FGF8_DEVERR_ROLE_EPILOGUE;
    constexpr int HALF = BN / 2;
    const uint32_t q = warp & 3u;
    const int h = static_cast<int>(warp - 2) >> 2;  // which half of the tile's columns
    const bool bf16 = args.out_bf16 != 0;
    const int nkb128 = K / 128;
    const int nnb = (N + 127) / 128;
    const int ld_a = (M + 3) / 4 * 4;
    int pbuf = 0;
    uint32_t pphase = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      Tile tl;
      if (!get_tile(t, tl)) continue;
      const int r = static_cast<int>(q * 32 + lane);
      bool row_ok = r < tl.row_limit;
      if constexpr (SCHED == Sched::Contiguous) {
        if (row_ok) {
          const int g = __ldg(args.m_indices + tl.a_row0 + r);
          if (g != tl.group) {
            if (g >= 0) atomicOr(args.status, FGF8_DEVERR_INPUT);
            row_ok = false;
          }
        }
      }
      const int col0 = tl.n_blk * BN + h * HALF;
      const bool col_ok = col0 < N;
      // scale tables: activation rows of this tile's expert, weight block of these columns
      const int m_local = tl.m_blk * C::BM + r;
      const float* sfa = args.sfa_f32 +
                         (SCHED == Sched::Masked ? static_cast<size_t>(tl.group) * nkb128 * ld_a : 0) +
                         m_local;
      const float* sfb = args.sfb_f32 +
                         (static_cast<size_t>(tl.group) * nnb + (col_ok ? col0 / 128 : 0)) * nkb128;
      float accv[HALF];
#pragma unroll
      for (int i = 0; i < HALF; ++i) accv[i] = 0.0f;
      float sa = row_ok ? __ldg(sfa) : 0.0f;
      float sb = col_ok ? __ldg(sfb) : 0.0f;
      for (int kb = 0; kb < nkb; ++kb) {
        const float s = sa * sb;
        if (kb + 1 < nkb) {
          sa = row_ok ? __ldg(sfa + static_cast<size_t>(kb + 1) * ld_a) : 0.0f;
          sb = col_ok ? __ldg(sfb + kb + 1) : 0.0f;
        }
        if (!wait_bar_warp(bar(C::BAR_ACC_FULL + pbuf), pphase, ctl)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t taddr = tmem_base + ((q * 32u) << 16) +
                               static_cast<uint32_t>(pbuf * BN + h * HALF);
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(taddr + 32u * c, v);
          ptx::tmem_wait_ld();
          if (c == HALF / 32 - 1) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(C::BAR_ACC_EMPTY + pbuf));
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) accv[32 * c + j] = fmaf(s, __uint_as_float(v[j]), accv[32 * c + j]);
        }
        if (++pbuf == 2) { pbuf = 0; pphase ^= 1u; }
      }
      if (!ok) break;
      if (row_ok) {
        const size_t row_off = static_cast<size_t>(tl.a_row0 + r) * static_cast<size_t>(N);
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c)
          store_chunk32(args.D, row_off, col0 + 32 * c, N, accv + 32 * c, bf16);
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::TMEM_ALLOC);
  }
}

}  // namespace fgf8

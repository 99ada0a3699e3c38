// gemm_persistent.cuh -- persistent, warp-specialised NT GEMM for sm_103a, on one
// CTA or on a CTA pair (cta_group::2).
//
//   D[M,N] = A[M,K] * B[N,K]^T, FP32 accumulation, 16-bit output.
//
// A tile is (128 * NCTA) rows x BN columns.  With NCTA = 2 the two CTAs of a
// cluster form a pair: each holds its own 128 rows of A and half of the BN rows
// of B; one thread of the even CTA issues tcgen05.mma.cta_group::2 with M = 256,
// and each CTA's TMEM receives its own 128 accumulator rows ("GPU GEMM part 4:
// tcgen05 & Blackwell", section 5.2: A and D split along M, B along N; "Blackwell
// Tensor Core: tcgen05.mma", cta_group::2 M = 256 layout).  Halving each CTA's B
// tile cuts both its SMEM footprint and its L2->SMEM traffic per FLOP by a third,
// which leaves room for a deeper pipeline.
//
// Pipeline unit.  The producer fills, and the MMA warp consumes, KPU K blocks
// per full/empty handshake: two (one hand-off covers 8 MMAs); for FP32 scales two
// where four partial buffers fit, else one; four on the decode tiles.
//
// Decode tiles (AROWS = 64, dense GEMMs with at most 64 rows) stage 64-row A
// boxes, so more stages of B fit, and read each weight row in 512-byte runs.
// QOUT kernels quantize their output 1x128 in the epilogue (E4M3 codes and
// scales in the quantize_1x128 layout) instead of storing it.
//
// Roles (per CTA):
//   warp 0   TMA producer: A/B tiles into a STAGES-deep ring of 128-byte-swizzled
//            stages.  In a pair both CTAs' loads complete on the even CTA's `full`
//            barrier (cp.async.bulk.tensor .cta_group::2).
//   warp 1   MMA issuer (even CTA; one thread) and TMEM owner (both CTAs).  It
//            never polls an mbarrier: it meets the relay warp at a named barrier
//            and then issues the unit's MMAs and commits back to back.  An
//            mbarrier try_wait (or any shared-memory access) by the thread that
//            issues tcgen05.mma queues behind its pending MMAs, ~170 cycles even on
//            a completed barrier, which starved the tensor pipe between units.
//   warps 2-5 (UE8M0 kernels) scale-factor writers, one per TMEM lane quarter:
//            one lane TMA-loads the packed scale words of each group of four K
//            blocks into a small SMEM ring, three groups ahead; each writer reads
//            them from there and writes them into a TMEM scale slot with
//            tcgen05.st (each quarter gets the same copy), then signals
//            `sf_ready` (counted over the pair).  The block-scaled MMA reads A's
//            scale of row 32 j + l and B's scale of row 32 j + l from lane l,
//            column j of its slot ("Blackwell Tensor Core: tcgen05.mma",
//            Block-Scaled MMA: SFA/SFB live in TMEM).  Writing them from the
//            warps keeps the copy out of the tensor pipe: a tcgen05.cp issued
//            between MMAs stalls the MMA stream for several hundred cycles.
//   next     epilogue: 4 warps (tcgen05.ld -> cast -> store) with two accumulator
//            buffers; 8 warps with a single 256-column buffer (each drains 128
//            columns into registers, releases the buffer, then stores).  For FP32
//            scales, promotion: 8 warps, per-128-K partial from TMEM,
//            acc += sA*sB*partial on the CUDA cores (the DeepGEMM page's
//            promotion loop), one full/empty handshake per unit's slot of partial
//            buffers, the scales loaded one unit ahead into registers.
//   last     relay warp (even CTA): waits, for the MMA warp, on the unit's `full`
//            barrier, the accumulator's `empty` barrier and the scale slot's
//            `sf_ready`, then meets the MMA warp at the named barrier.
// Pipeline handshakes follow the tma2mma / mma2tma / mma2ld / ld2mma barriers of
// "TIRx and high-performance GEMM (part 2)" (Steps 7-8); every mbarrier wait is
// bounded.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <type_traits>

#include "device_common.cuh"
#include "quant_common.cuh"

namespace fgf8 {

// ----------------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared-memory address of the same object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Arrive on a barrier of any CTA of the cluster.  The default (release, CTA
// scope) form is enough: what the waiting side reads next is either TMEM written
// by tcgen05 ops this thread has already waited on (tcgen05.wait + fence pair) or
// shared memory filled by TMA (counted in the barrier's transaction bytes).  A
// cluster-scope release here costs on the order of a thousand cycles.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

template <int NCTA>
__device__ __forceinline__ void tma_load_ab(uint32_t dst, const CUtensorMap* m, uint32_t bar_cluster,
                                            int32_t x, int32_t y) {
  if constexpr (NCTA == 2) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y)
        : "memory");
  } else {
    ptx::tma_load_2d(dst, m, bar_cluster, x, y);
  }
}

// tcgen05 ops with the kernel-wide cta_group.
template <int NCTA>
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  if constexpr (NCTA == 2)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
  else
    ptx::mma_commit(bar);
}
// Arrive on `bar` in every CTA of `mask` once the tracked ops complete.
template <int NCTA>
__device__ __forceinline__ void tc_commit_mc(uint32_t bar, uint16_t mask) {
  if constexpr (NCTA == 2)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
  else
    ptx::mma_commit(bar);
}
template <int NCTA>
__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (NCTA == 2) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    ptx::tmem_alloc(dst_smem, ncols);
    ptx::tmem_relinquish();
  }
}
template <int NCTA>
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (NCTA == 2)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  else
    ptx::tmem_dealloc(taddr, ncols);
}
template <int NCTA, Kind KIND>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc,
                                       uint32_t sfa, uint32_t sfb, uint32_t acc) {
  if constexpr (KIND == Kind::MXF4 || KIND == Kind::NVF4) {
    // E2M1 operands packed two per byte along K, 64 elements (32 bytes) per
    // instruction; two E8M0 (MXFP4) or four E4M3 (NVFP4) scale bytes per row and
    // instruction, read from TMEM starting at the byte the idesc ids select
    // ("GPU GEMM part 4: tcgen05 & Blackwell", sections 3.5 and 6.2-6.3)
    if constexpr (NCTA == 2) {
      if constexpr (KIND == Kind::MXF4)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X"
            " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
            "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
            : "memory");
      else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
            " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
            "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
            : "memory");
    } else {
      if constexpr (KIND == Kind::MXF4)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X"
            " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
            "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
            : "memory");
      else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
            " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
            "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
            : "memory");
    }
  } else if constexpr (NCTA == 2) {
    if constexpr (KIND == Kind::MXF8)
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
          " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
          "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
          : "memory");
    else if constexpr (KIND == Kind::F8F32)
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
          "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
          : "memory");
    else
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
          "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
          : "memory");
  } else {
    if constexpr (KIND == Kind::MXF8) ptx::mma_mxf8(d, ad, bd, idesc, sfa, sfb, acc);
    else if constexpr (KIND == Kind::F8F32) ptx::mma_f8(d, ad, bd, idesc, acc);
    else ptx::mma_f16(d, ad, bd, idesc, acc);
  }
}

// 32 lanes x 4 columns of 32 bits from registers into TMEM (thread l -> lane base + l).
__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
               "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Test a phase of a barrier in this CTA (default acquire, CTA scope; see
// mbar_arrive_cluster for why no cluster-scope ordering is needed).
__device__ __forceinline__ bool try_wait_cluster(uint32_t bar, uint32_t parity) {
  return ptx::mbar_try_wait(bar, parity);
}

// Test a phase of a barrier in this CTA with cluster-scope acquire (the barrier's
// data was stored from another CTA of the cluster).
__device__ __forceinline__ bool try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

struct PairWaitCtl {
  volatile uint32_t* abort_flag;   // this CTA's flag (shared memory)
  uint32_t peer_abort;             // the peer's flag (cluster address), 0 if none
  uint32_t* status;
  uint64_t timeout_ns;
  uint32_t role_bit;
};

template <bool ACQ_CLUSTER = false>
__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, const PairWaitCtl& c) {
  auto test = [&]() { return ACQ_CLUSTER ? try_wait_acq_cluster(bar, parity) : try_wait_cluster(bar, parity); };
  bool ok = test();
  if (!ok) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t i = 1;; ++i) {
      if (test()) { ok = true; break; }
      if ((i & 63u) == 0) {
        if (*c.abort_flag) break;
        if (ptx::globaltimer() - t0 > c.timeout_ns) {
          *c.abort_flag = 1u;
          if (c.peer_abort) st_cluster_u32(c.peer_abort, 1u);
          atomicOr(c.status, FGF8_DEVERR_TIMEOUT | c.role_bit);
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok) != 0;
}

// Weight-stationary E4M3 MMA (kind::f8f6f4, cta_group::1, M = 128): mode 1 reads B
// from shared memory and keeps it in collector buffer 0, mode 2 reads B from that
// buffer and frees it, mode 0 uses no collector ("GPU GEMM part 4: tcgen05 &
// Blackwell", section 3.7).
__device__ __forceinline__ void tc_mma_ws_f8(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc,
                                             int mode) {
  if (mode == 1)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.ws.cta_group::1.kind::f8f6f4.collector::b0::fill [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
  else if (mode == 2)
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.ws.cta_group::1.kind::f8f6f4.collector::b0::lastuse [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.ws.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}

template <Kind KIND, Sched SCHED, int NCTA_, int BN_, int STAGES_, int NACC_ = 2, int AROWS_ = 128,
          bool QOUT_ = false>
struct PCfg {
  static constexpr int NCTA = NCTA_;
  static constexpr int CLUSTER = NCTA;               // a cluster is one CTA or one CTA pair
  static constexpr int BM = 128;                    // rows per CTA (per MMA, per TMEM lane)
  // Weight-stationary tile (FP32 scales; "GPU GEMM part 4: tcgen05 & Blackwell",
  // section 3.7): AROWS = 256 rows of A per CTA, computed as two M = 128 sub-tiles
  // by tcgen05.mma.ws that share each B operand through the MMA unit's collector
  // buffer (the first fills it, the second uses it last), so one weight tile in
  // shared memory feeds 256 rows.
  static constexpr bool kWS = AROWS_ == 2 * BM;
  static constexpr int MSUB = kWS ? 2 : 1;
  static constexpr int TILE_M = BM * NCTA * MSUB;
  static constexpr int BN = BN_;
  static constexpr int PBN = BN * MSUB;             // TMEM columns of one accumulator / K block partial
  static constexpr int BN_LOCAL = BN / NCTA;        // B rows held by each CTA
  static constexpr int STAGES = STAGES_;
  static_assert(NCTA == 1 || NCTA == 2, "one CTA or a pair");
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "BN");
  static_assert(KIND != Kind::F8F32 || BN % 64 == 0, "promotion halves of whole 32-column chunks");
  static_assert(BN_LOCAL % 16 == 0, "B rows per CTA");
  static constexpr bool kMX = KIND == Kind::MXF8;
  // 4-bit E2M1 operands with MXFP4 or NVFP4 block scales
  static constexpr bool kFP4 = KIND == Kind::MXF4 || KIND == Kind::NVF4;
  // block-scaled MMA: scale factors staged into TMEM by the writer warps
  static constexpr bool kBS = kMX || kFP4;
  static constexpr bool kF32S = KIND == Kind::F8F32;
  // TMA x step per K block, in elements of the operand tensor map (bytes for the
  // 8-bit and packed 4-bit operands): every K block is 128 bytes of each row
  static constexpr int BK = (KIND == Kind::F16) ? 64 : 128;
  // K elements per K block: 64 (16-bit), 128 (8-bit), 256 (4-bit, two per byte)
  static constexpr int KB_ELEMS = (KIND == Kind::F16) ? 64 : kFP4 ? 256 : 128;
  static constexpr int MMA_K_BYTES = 32;
  static constexpr int MMAS_PER_STAGE = 128 / MMA_K_BYTES;
  // Rows of A per K block.  A thin tile (AROWS = 64, for a dense GEMM with at most
  // 64 rows) stages 64 A rows, loaded by a box of M rounded up to 8 rows
  // (args.a_box_rows; the stage rows past it are never stored).  With FP32 scales it
  // issues M = 64 MMAs ("Blackwell Tensor Core: tcgen05.mma": the cta_group::1
  // M = 64 accumulator, Layout F, puts row m in TMEM lane 32 (m / 16) + m % 16, so
  // each lane quarter holds 16 rows in its first 16 lanes), which leaves room for
  // more stages.  The block-scaled MMA of one CTA has M = 128 only: there each
  // stage holds its 64 A rows, then its own B rows, padded to 16 KB, so the MMA's
  // upper 64 rows read this stage's landed B and padding (never a stage that TMA
  // is filling) and only feed accumulator rows that are never stored.
  static constexpr bool kThin = AROWS_ < BM;
  static constexpr bool kThinM64 = kThin && !(KIND == Kind::MXF8 || KIND == Kind::MXF4 || KIND == Kind::NVF4);
  static constexpr bool kInterleave = kThin && !kThinM64;
  static constexpr int A_LOAD_ROWS = AROWS_;                           // rows of one A box
  static constexpr int A_ROWS = AROWS_;                                // rows of one A stage
  static constexpr int MMA_M = kThinM64 ? 64 : (kWS ? BM : BM * NCTA);   // rows per MMA instruction
  static constexpr int QROWS = kThinM64 ? 16 : 32;                       // accumulator rows per lane quarter
  static_assert(!kThin || (NCTA == 1 && SCHED == Sched::Dense), "thin A tiles: single CTA, dense layout");
  static_assert(A_ROWS == BM || (A_ROWS == 64 && NCTA == 1 && SCHED == Sched::Dense) ||
                    (kWS && KIND == Kind::F8F32 && NCTA == 1 && BN == 128 && SCHED != Sched::Contiguous && !QOUT_),
                "thin A tiles: single CTA, dense layout; weight-stationary tiles: FP32 scales, one CTA, "
                "128 columns, dense or masked layout");
  static constexpr int A_BYTES = A_ROWS * 128;
  static constexpr int B_BYTES = BN_LOCAL * 128;
  static constexpr int SFB_ROWS = (BN + 127) / 128 * 128;
  // K blocks per pipeline unit: one full/empty handshake, one hand-off to the MMA
  // warp and one stage-release commit per unit.  The FP32-scale path gives every
  // K block of a unit its own partial buffer, so it takes two K blocks per unit
  // only where four partial buffers fit (two units in flight).
  // A thin tile takes four K blocks per unit: the producer then reads 512
  // contiguous bytes of each B row per unit (the FP32-scale one needs eight
  // partial buffers for that).
  static constexpr int KPU = AROWS_ < BM ? 4 : kF32S ? (NACC_ >= 4 ? 2 : 1) : 2;
  static_assert(STAGES % KPU == 0, "stages per unit");
  static constexpr int UNITS = STAGES / KPU;
  static constexpr int SF_WARPS = kBS ? 4 : 0;
  // Scale-word groups.  A packed word holds four scale bytes of a row.  UE8M0
  // FP8: one word per four K blocks (byte kb % 4 per K block), so a group is
  // four K blocks.  4-bit: a K block of 256 elements needs 2 (MXFP4, 8 scales of
  // 32) or 4 (NVFP4, 16 scales of 16) words per row, so a group is one pipeline
  // unit.  WG: words per row per group.
  static constexpr int GK = kFP4 ? KPU : 4;
  static constexpr int WPK = KIND == Kind::MXF4 ? 2 : KIND == Kind::NVF4 ? 4 : 0;
  static constexpr int WG = kFP4 ? GK * WPK : 1;
  // FP32 scales: 8 promotion warps.  A single accumulator buffer (NACC = 1,
  // 256-wide block-scaled tiles) is drained by 8 epilogue warps, two per TMEM
  // lane quarter, so that the MMAs of the next tile wait only for the drain.
  static constexpr int EPI_WARPS = (kF32S || NACC_ == 1) ? 8 : 4;
  static constexpr int EPI_WARP0 = 2 + SF_WARPS;
  static constexpr int RELAY_WARP = EPI_WARP0 + EPI_WARPS;
  // tile scheduler of cluster launch control (idle under the static schedule)
  static constexpr int SCHED_WARP = RELAY_WARP + 1;
  static constexpr int THREADS = 32 * (SCHED_WARP + 1);
  static constexpr int HANDOFF_BAR = 1;              // named barrier: relay warp + MMA warp
  static constexpr int MAX_GROUPS = 1024;

  // TMEM accumulator buffers: 2 for a finished tile (epilogue overlap; 1 on the
  // 256-wide block-scaled tile, drained at once), more for the per-K-block
  // partials of the FP32-scale path (promotion latency slack).
  static constexpr int NACC = NACC_;
  // FP32-scale path: the partial buffers of one unit form a slot with a single
  // full/empty handshake between the MMA warp and the promotion warps
  static constexpr int NSLOT = kF32S ? NACC / KPU : NACC;
  // the epilogue can quantize its own output in 1x128 groups: every group inside
  // one epilogue thread (block-scaled tiles 128 or 256 wide; FP32-scale tiles 256
  // wide, whose promotion warps each hold 128 columns of a row)
  // (QOUT: a separate instantiation, so the plain kernels carry none of it)
  static constexpr bool kFuseQuant = QOUT_;
  static_assert(!QOUT_ || (SCHED == Sched::Dense &&
                           ((KIND == Kind::MXF8 && BN % 128 == 0) || (KIND == Kind::F8F32 && BN == 256))),
                "output quantization: whole 1x128 groups per epilogue thread");
  static_assert(!kF32S || (NACC % KPU == 0 && NSLOT >= 2), "two slots of partial buffers");
  static constexpr int SF_RING = 4;                                // scale-word groups in SMEM
  static constexpr int SFA_RING_BYTES = kBS ? WG * BM * 4 : 0;
  static constexpr int SFB_RING_BYTES = kBS ? WG * SFB_ROWS * 4 : 0;
  static constexpr int STAGE_BYTES = 16384;        // interleaved stage: A, then B, then padding
  static_assert(!kInterleave || A_BYTES + B_BYTES <= STAGE_BYTES, "interleaved stage");
  static constexpr int A_STRIDE = kInterleave ? STAGE_BYTES : A_BYTES;
  static constexpr int B_STRIDE = kInterleave ? STAGE_BYTES : B_BYTES;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = kInterleave ? A_BYTES : OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_SFA = kInterleave ? STAGES * STAGE_BYTES : OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + SF_RING * SFA_RING_BYTES;
  static constexpr int OFF_BAR = (OFF_SFB + SF_RING * SFB_RING_BYTES + 7) / 8 * 8;
  static constexpr int BAR_FULL = 0;                              // UNITS
  static constexpr int BAR_EMPTY = UNITS;                         // UNITS
  static constexpr int BAR_ACC_FULL = 2 * UNITS;                  // NACC
  static constexpr int BAR_ACC_EMPTY = BAR_ACC_FULL + NACC;       // NACC
  // TMEM scale slots: three where they fit next to the accumulators, so the
  // scale writers can run two groups of K blocks ahead of the MMA
  static constexpr int NB_COLS = SFB_ROWS / 32;               // TMEM columns of one SFB word
  static constexpr int SF_SLOT_COLS = WG * (4 + NB_COLS);
  static constexpr int SF_SLOTS = (NACC_ * BN + 3 * SF_SLOT_COLS <= 512) ? 3 : 2;
  static constexpr int BAR_SFR = BAR_ACC_EMPTY + NACC;            // SF_SLOTS: slot written (even CTA)
  static constexpr int BAR_SF_FREE = BAR_SFR + SF_SLOTS;          // SF_SLOTS: slot read (each CTA)
  static constexpr int BAR_SFL = BAR_SF_FREE + SF_SLOTS;          // SF_RING: words landed (local)
  static constexpr int BAR_SFC = BAR_SFL + SF_RING;               // SF_RING: words read (local)
  static constexpr int BAR_DRAIN = BAR_SFC + SF_RING;
  // cluster launch control: the scheduler warp's try_cancel response lands in a
  // 16-byte staging slot (BAR_CLC_STAGE, leader); the tiles it accepts are
  // published as tile ids into a ring of CLC_Q slots in every CTA of the cluster.  A
  // ring slot is full once its tile id is published (one arrival) and empty when
  // every epilogue warp of the cluster has finished that tile.  The ring is
  // deeper than any role runs ahead of the epilogue in tiles: the scale-word loader
  // (three groups ahead of the writers, who are up to three ahead of the MMA, which
  // is up to two tiles ahead of the epilogue) and the producer (up to UNITS units
  // ahead of the MMA), with at least one group and one unit per tile.
  static constexpr int CLC_Q = 12;
  static constexpr int BAR_CLC_FULL = BAR_DRAIN + 1;              // CLC_Q (each CTA)
  static constexpr int BAR_CLC_EMPTY = BAR_CLC_FULL + CLC_Q;      // CLC_Q (leader)
  static constexpr int BAR_CLC_STAGE = BAR_CLC_EMPTY + CLC_Q;     // 1 (leader)
  static constexpr int NUM_BARS = BAR_CLC_STAGE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_PREFIX = (OFF_MISC + 16 + 15) / 16 * 16;
  // contiguous layout on CTA pairs: tiles are cut per expert segment (run of
  // 128-row blocks with the same expert), so the scheduler keeps each run's first
  // block, expert and tile prefix; at most MAX_RUNS runs (M <= MAX_RUNS * 128)
  static constexpr bool kRuns = SCHED == Sched::Contiguous && NCTA == 2;
  static constexpr int MAX_RUNS = 512;
  static constexpr int PREFIX_BYTES = (SCHED == Sched::Masked) ? (MAX_GROUPS + 1) * 4
                                      : kRuns                  ? 3 * (MAX_RUNS + 1) * 4
                                                               : 0;
  // staging response (16 bytes), then CLC_Q published tile ids (int32, -1 = end)
  static constexpr int OFF_CLC = (OFF_PREFIX + PREFIX_BYTES + 15) / 16 * 16;
  // The epilogue stages each warp's 32 x 32 chunk of D in shared memory (two
  // buffers per warp) and writes it with a TMA tensor store, one coalesced bulk
  // transfer instead of 32 rows of 16-byte stores per instruction.  In grouped
  // layouts a warp does so only when all its 32 rows are to be written (rows
  // past masked_m and padding rows must stay untouched); otherwise it stores
  // its valid rows one by one.
  static constexpr int EPI_CHUNK_BYTES = 32 * 32 * 2;
  static constexpr int OFF_EPI = (OFF_CLC + 16 + 4 * CLC_Q + 127) / 128 * 128;
  static constexpr bool kTmaStore = !QOUT_ && !kF32S && NACC_ == 2 && !kWS &&
                                    BN % 32 == 0 && QROWS == 32 &&
                                    OFF_EPI + 2 * EPI_WARPS * EPI_CHUNK_BYTES + 1024 <= 232448;
  static constexpr int EPI_BYTES = kTmaStore ? 2 * EPI_WARPS * EPI_CHUNK_BYTES : 0;
  static constexpr int SMEM_BYTES = OFF_EPI + EPI_BYTES + 1024;

  static constexpr int ACC_COLS = NACC * PBN;
  static constexpr int SF_COL0 = ACC_COLS;
  static constexpr int TMEM_USED = ACC_COLS + (kBS ? SF_SLOTS * SF_SLOT_COLS : 0);
  static constexpr int TMEM_ALLOC = TMEM_USED <= 32    ? 32
                                    : TMEM_USED <= 64  ? 64
                                    : TMEM_USED <= 128 ? 128
                                    : TMEM_USED <= 256 ? 256
                                                       : 512;
  static_assert(TMEM_USED <= 512, "TMEM budget");
  static constexpr uint32_t A_TX = NCTA * (A_LOAD_ROWS * 128 + B_BYTES);   // bytes landing on `full`
  static_assert(kF32S ? NACC >= 2 : (NACC == 2 || (NACC == 1 && BN == 256 && kBS)),
                "accumulator buffers");
  static constexpr uint32_t SF_TX = WG * (BM * 4 + BN * 4);         // bytes landing on `sf_loaded`
  static_assert(!kFP4 || (SCHED == Sched::Dense && !QOUT_ && AROWS_ == BM && BN % 32 == 0 && KPU == GK),
                "4-bit: dense tiles, one scale group per pipeline unit");
};

// Cluster launch control ("Dissecting NVIDIA Blackwell" (EEPW), the feature list):
// asks the hardware to cancel one cluster of this grid that has not launched yet
// (a pair is cancelled whole).  The 16-byte response lands at `resp` and completes
// 16 transaction bytes on the barrier `bar`, both in this CTA.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar) {
  asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::
                   "r"(resp),
               "r"(bar)
               : "memory");
}
// Publishes a tile id to a CTA of the cluster: the store, then an arrive with
// cluster-scope release on that CTA's barrier, so that a waiter there that
// acquires at cluster scope reads the id.
__device__ __forceinline__ void clc_publish(uint32_t slot_cluster, uint32_t bar_cluster, int tile) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(slot_cluster), "r"(tile) : "memory");
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}
// The cluster a response names (the x index of its first CTA over the cluster
// size), or -1 when nothing was cancelled: every cluster has launched.
__device__ __forceinline__ int clc_cluster(uint32_t resp, int cluster) {
  uint32_t x, ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b128 cr;\n\t"
      "ld.shared.b128 cr, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, cr;\n\t"
      "selp.u32 %1, 1, 0, p;\n\t"
      "mov.u32 %0, 0;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, cr;\n\t}"
      : "=r"(x), "=r"(ok)
      : "r"(resp)
      : "memory");
  return ok ? static_cast<int>(x) / cluster : -1;
}

// Named-barrier rendezvous of `nthreads` threads (whole warps).  It goes through the
// CTA barrier unit, not shared memory: the MMA warp waits here instead of polling an
// mbarrier, because a shared-memory access by the thread that issues tcgen05.mma
// queues behind its pending MMAs (measured: ~170 cycles for a try_wait on a
// completed barrier, 43 from any other warp).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[16]) {
  ptx::tmem_ld_32x32b_x16(taddr, r);
}
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[32]) {
  ptx::tmem_ld_32x32b_x32(taddr, r);
}

__device__ __forceinline__ uint32_t pack_2x16(float a, float b, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 32 consecutive FP32 values of one output row -> 16-bit, columns col0..col0+31
// clipped at N (N is a multiple of 8).
__device__ __forceinline__ void store_row32(void* D, size_t row_off, int col0, int N,
                                            const float* v, bool bf16) {
  uint16_t* out = reinterpret_cast<uint16_t*>(D) + row_off;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int col = col0 + 8 * j;
    if (col < N) {
      uint4 w;
      w.x = pack_2x16(v[8 * j + 0], v[8 * j + 1], bf16);
      w.y = pack_2x16(v[8 * j + 2], v[8 * j + 3], bf16);
      w.z = pack_2x16(v[8 * j + 4], v[8 * j + 5], bf16);
      w.w = pack_2x16(v[8 * j + 6], v[8 * j + 7], bf16);
      *reinterpret_cast<uint4*>(out + col) = w;
    }
  }
}

// 16 consecutive FP32 values of one output row -> 16-bit, columns col0..col0+15.
__device__ __forceinline__ void store_row16(void* D, size_t row_off, int col0, int N,
                                            const float* v, bool bf16) {
  uint16_t* out = reinterpret_cast<uint16_t*>(D) + row_off;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int col = col0 + 8 * j;
    if (col < N) {
      uint4 w;
      w.x = pack_2x16(v[8 * j + 0], v[8 * j + 1], bf16);
      w.y = pack_2x16(v[8 * j + 2], v[8 * j + 3], bf16);
      w.z = pack_2x16(v[8 * j + 4], v[8 * j + 5], bf16);
      w.w = pack_2x16(v[8 * j + 6], v[8 * j + 7], bf16);
      *reinterpret_cast<uint4*>(out + col) = w;
    }
  }
}


// E4M3 codes of NV values `val(0..NV-1)` (already rounded to bf16) with the
// group's scale, stored as NV contiguous bytes at dst.
template <bool UE8M0, int NV, typename Val>
__device__ __forceinline__ void quantize_codes_out(const Val& val, const quant::GroupScale& gs, uint8_t* dst) {
#pragma unroll
  for (int k = 0; k < NV / 16; ++k) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 16 * k + 4 * i;
      w[i] = quant::e4m3x4<UE8M0>(val(e), val(e + 1), val(e + 2), val(e + 3), gs);
    }
    *reinterpret_cast<uint4*>(dst + 16 * k) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// One 128-column group of one row: its 128 values come from `val(i)`, already
// rounded to bf16 as D would be stored; writes the 128 E4M3 codes and the group's
// scale in the quantize_1x128 layout (scale table [group][ld] of floats, or packed
// UE8M0 words [group / 4][ld] whose byte group % 4 belongs to the group).
template <bool UE8M0, typename Val>
__device__ __forceinline__ void quantize_group_out(const Val& val, float amax, uint8_t* dq_row, void* sfd,
                                                   size_t sf_index) {
  const quant::GroupScale gs = quant::group_scale<UE8M0>(amax);
  quantize_codes_out<UE8M0, 128>(val, gs, dq_row);
  if (UE8M0) reinterpret_cast<uint8_t*>(sfd)[sf_index] = static_cast<uint8_t>(gs.byte);
  else reinterpret_cast<float*>(sfd)[sf_index] = gs.s;
}

// x rounded to bf16 (nearest even), as an FP32 value.
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Value i of 128 bf16 values packed in pairs (low half first).
struct PackedBf16 {
  const uint32_t* h;
  __device__ __forceinline__ float operator()(int i) const {
    const uint32_t w = h[i >> 1];
    return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
};
// Value i of 128 FP32 values, rounded to bf16.
struct RoundedF32 {
  const float* v;
  __device__ __forceinline__ float operator()(int i) const { return bf16_round(v[i]); }
};

// Fused output quantization of group `grp` (128 columns) of output row `grow`:
// the codes and scale of a valid row; a zero scale for a padding row of the
// scale table (rows M .. align4(M) - 1); and, from the row's last group, zeros in
// the unused bytes of its UE8M0 word -- all as quantize_1x128 writes them.
template <typename Val>
__device__ __forceinline__ void fused_group_out(const GemmArgs& args, const Val& val, float amax, int grp,
                                                int grow, bool row_ok) {
  const int M = args.M, N = args.N;
  const int ld = (M + 3) / 4 * 4;
  const int ngroups = N / 128;
  if (grp >= ngroups) return;
  const bool pad_row = !row_ok && grow >= M && grow < ld;
  const bool ue = args.dq_ue8m0 != 0;
  const size_t sf_index = ue ? (static_cast<size_t>(grp / 4) * ld + grow) * 4 + (grp % 4)
                             : static_cast<size_t>(grp) * ld + grow;
  if (row_ok) {
    uint8_t* dq_row = args.dq + static_cast<size_t>(grow) * N + static_cast<size_t>(grp) * 128;
    if (ue) quantize_group_out<true>(val, amax, dq_row, args.sfd, sf_index);
    else quantize_group_out<false>(val, amax, dq_row, args.sfd, sf_index);
  } else if (pad_row) {
    if (ue) reinterpret_cast<uint8_t*>(args.sfd)[sf_index] = 0;
    else reinterpret_cast<float*>(args.sfd)[sf_index] = 0.0f;
  }
  if (ue && grp == ngroups - 1 && (row_ok || pad_row))
    for (int j = grp % 4 + 1; j < 4; ++j) reinterpret_cast<uint8_t*>(args.sfd)[sf_index - grp % 4 + j] = 0;
}

// 32 packed 16-bit values of one output row (16 words) -> D, columns col0..col0+31
// clipped at N (N is a multiple of 8).
__device__ __forceinline__ void store_row32_packed(void* D, size_t row_off, int col0, int N, const uint32_t* h) {
  uint16_t* out = reinterpret_cast<uint16_t*>(D) + row_off;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (col0 + 8 * j < N)
      *reinterpret_cast<uint4*>(out + col0 + 8 * j) = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
}

template <Kind KIND, Sched SCHED, int NCTA, int BN, int STAGES, int NACC, int AROWS, bool QOUT>
__global__ void __launch_bounds__(PCfg<KIND, SCHED, NCTA, BN, STAGES, NACC, AROWS, QOUT>::THREADS, 1)
    gemm_persistent(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_sfa,
                    const __grid_constant__ CUtensorMap tm_sfb,
                    const __grid_constant__ CUtensorMap tm_d, const GemmArgs args) {
  using C = PCfg<KIND, SCHED, NCTA, BN, STAGES, NACC, AROWS, QOUT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const uint32_t warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;
  const uint32_t crank = (C::CLUSTER > 1) ? cluster_rank() : 0u;
  const uint32_t rank = crank;                        // rank within the pair
  const bool leader = rank == 0;
  // commit mask: both CTAs of the pair
  const uint16_t pair_mask = static_cast<uint16_t>((1u << NCTA) - 1u);

  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  // the pair leader's copy of barrier i (cluster address)
  auto lbar = [&](int i) -> uint32_t { return NCTA == 2 ? map_to_rank(bar(i), 0u) : bar(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC + 4);
  int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);

  const int M = args.M, N = args.N, K = args.K, G = args.G;
  const int nkb = (K + C::KB_ELEMS - 1) / C::KB_ELEMS;
  const int num_n = (N + BN - 1) / BN;
  const int num_m = (M + C::TILE_M - 1) / C::TILE_M;   // per expert for masked
  // scale words per row of a scale table
  const int kq = C::kFP4 ? nkb * C::WPK : (K / 128 + 3) / 4;
  const int cluster_id = static_cast<int>(blockIdx.x) / C::CLUSTER;
  const int num_clusters = static_cast<int>(gridDim.x) / C::CLUSTER;

  // ---------------------------------------------------------------- set-up
  // The tensor maps are kernel parameters, not data of the previous kernel: fetch
  // them into the TMA unit's cache now, under the barrier and TMEM set-up (after an
  // L2 flush the first TMA load otherwise waits a DRAM round trip for them).
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_a);
    ptx::prefetch_tmap(&tm_b);
    if constexpr (C::kBS) {
      ptx::prefetch_tmap(&tm_sfa);
      ptx::prefetch_tmap(&tm_sfb);
    }
    if constexpr (C::kTmaStore) ptx::prefetch_tmap(&tm_d);
  }
  if (threadIdx.x == 0) {
    for (int u = 0; u < C::UNITS; ++u) {
      ptx::mbar_init(bar(C::BAR_FULL + u), 1);
      ptx::mbar_init(bar(C::BAR_EMPTY + u), 1);
    }
    for (int b = 0; b < C::NACC; ++b) {
      ptx::mbar_init(bar(C::BAR_ACC_FULL + b), 1);
      ptx::mbar_init(bar(C::BAR_ACC_EMPTY + b), NCTA * C::EPI_WARPS);
    }
    if constexpr (C::kBS) {
      for (int b = 0; b < C::SF_SLOTS; ++b) {
        ptx::mbar_init(bar(C::BAR_SFR + b), NCTA * C::SF_WARPS);
        ptx::mbar_init(bar(C::BAR_SF_FREE + b), 1);
      }
      for (int r = 0; r < C::SF_RING; ++r) {
        ptx::mbar_init(bar(C::BAR_SFL + r), 1);
        ptx::mbar_init(bar(C::BAR_SFC + r), C::SF_WARPS);
      }
    }
    ptx::mbar_init(bar(C::BAR_DRAIN), 1);
    for (int q = 0; q < C::CLC_Q; ++q) {
      ptx::mbar_init(bar(C::BAR_CLC_FULL + q), 1);
      ptx::mbar_init(bar(C::BAR_CLC_EMPTY + q), NCTA * C::EPI_WARPS);
    }
    ptx::mbar_init(bar(C::BAR_CLC_STAGE), 1);
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    tc_alloc<NCTA>(ptx::smem_u32(tmem_slot), C::TMEM_ALLOC);
    ptx::tc_fence_before();
  }
  // Everything above touches only this CTA's shared memory and TMEM, so under a
  // programmatic dependent launch it overlaps the tail of the previous kernel.
  // Every read of global data (operands, scales, m_indices, masked_m) comes after
  // this wait.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  if constexpr (SCHED == Sched::Masked) {
    if (warp == 2) {
      int run = 0;
      for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + static_cast<int>(lane);
        int mm = (g < G) ? args.masked_m[g] : 0;
        if (mm < 0 || mm > M) {
          if (leader) atomicOr(args.status, FGF8_DEVERR_INPUT);
          mm = mm < 0 ? 0 : M;
        }
        int v = (mm + C::TILE_M - 1) / C::TILE_M * num_n;
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
  // contiguous pairs: runs of 128-row blocks whose first row names the same expert
  int* run_start = prefix + (C::MAX_RUNS + 1);          // first block of run r; [R] = nblk
  int* run_expert = prefix + 2 * (C::MAX_RUNS + 1);
  if constexpr (C::kRuns) {
    if (warp == 2) {
      const int nblk = M / C::BM;
      int nrun = 0;
      int prev = 0;
      bool ok = nblk <= C::MAX_RUNS;
      for (int b0 = 0; ok && b0 < nblk; b0 += 32) {
        const int b = b0 + static_cast<int>(lane);
        const int e = b < nblk ? __ldg(args.m_indices + static_cast<size_t>(b) * C::BM) : 0;
        int up = __shfl_up_sync(0xffffffffu, e, 1);
        if (lane == 0) up = prev;
        const bool start = b < nblk && (b == 0 || e != up);
        const uint32_t bal = __ballot_sync(0xffffffffu, start);
        if (start) {
          const int r = nrun + __popc(bal & ((1u << lane) - 1u));
          run_start[r] = b;
          run_expert[r] = e;
        }
        nrun += __popc(bal);
        prev = __shfl_sync(0xffffffffu, e, 31);
      }
      if (!ok) {
        if (lane == 0) atomicOr(args.status, FGF8_DEVERR_INPUT);
        nrun = 0;
      }
      __syncwarp();
      if (lane == 0) run_start[nrun] = nblk;
      __syncwarp();
      // pair tiles of run r: ceil(blocks / 2) x N tiles (runs of padding or of an
      // out-of-range expert contribute none)
      int acc = 0;
      for (int r0 = 0; r0 < nrun; r0 += 32) {
        const int r = r0 + static_cast<int>(lane);
        int v = 0;
        if (r < nrun) {
          const int e = run_expert[r];
          const int len = run_start[r + 1] - run_start[r];
          v = (e >= 0 && e < G) ? (len + 1) / 2 * num_n : 0;
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xffffffffu, v, off);
          if (static_cast<int>(lane) >= off) v += o;
        }
        if (r < nrun) prefix[r + 1] = acc + v;
        acc += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) {
        prefix[0] = 0;
        run_expert[C::MAX_RUNS] = nrun;                 // the run count, for the schedulers
      }
    }
  }
  __syncthreads();
  if constexpr (C::CLUSTER > 1) cluster_sync_all();   // peer barriers initialised before any remote use
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int num_tiles;
  int num_runs = 0;
  if constexpr (SCHED == Sched::Masked) {
    num_tiles = prefix[G];
  } else if constexpr (C::kRuns) {
    num_runs = run_expert[C::MAX_RUNS];
    num_tiles = prefix[num_runs];
  } else {
    num_tiles = num_m * num_n;
  }

  auto get_tile = [&](int t, Tile& tl) -> bool {
    int m, n, g = 0, rows;
    if constexpr (C::kRuns) {
      int lo = 0, hi = num_runs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
      }
      const int len = run_start[lo + 1] - run_start[lo];
      const int pt = (len + 1) / 2;                 // pair tiles of the run along M
      const int local = t - prefix[lo];
      n = local / pt;                               // pairs sharing a B tile are adjacent
      const int j = local - n * pt;
      const int half = 2 * j + static_cast<int>(rank);
      g = run_expert[lo];
      tl.a_row0 = (run_start[lo] + half) * C::BM;
      tl.m_blk = tl.a_row0;                         // activation scales are indexed by global row
      tl.n_blk = n;
      tl.group = g;
      tl.b_row0 = g * N + n * BN + static_cast<int>(rank) * C::BN_LOCAL;
      tl.row_limit = half < len ? C::BM : 0;        // the half past the run's end stores nothing
      return true;
    }
    if constexpr (SCHED == Sched::Masked) {
      int lo = 0, hi = G - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
      }
      g = lo;
      int mm = __ldg(args.masked_m + g);
      rows = mm < 0 ? 0 : (mm > M ? M : mm);
      const int mt = (rows + C::TILE_M - 1) / C::TILE_M;
      const int local = t - prefix[g];
      n = local / mt;                              // M blocks sharing a B tile are adjacent
      m = local - n * mt;
    } else {
      dense_tile(t, num_m, num_n, 16, m, n);
      rows = M;
      if constexpr (SCHED == Sched::Contiguous) {
        g = __ldg(args.m_indices + m * C::TILE_M);
        if (g < 0 || g >= G) return false;
      }
    }
    const int m_in_expert = m * C::TILE_M + static_cast<int>(rank) * C::BM;
    tl.m_blk = m_in_expert;                       // first row of this CTA within the expert
    tl.n_blk = n;
    tl.group = g;
    tl.a_row0 = (SCHED == Sched::Masked ? g * M : 0) + m_in_expert;
    tl.b_row0 = (SCHED == Sched::Dense ? 0 : g * N) + n * BN + static_cast<int>(rank) * C::BN_LOCAL;
    tl.row_limit = rows - m_in_expert;
    return true;
  };

  PairWaitCtl ctl{abort_flag,
                  NCTA == 2 ? map_to_rank(sbase + C::OFF_MISC + 4, crank ^ 1u) : 0u,
                  args.status, args.timeout_ns, 0};
  bool aborted = false;

  // ---------------------------------------------------------------- tile sequence
  // Every role walks the same sequence of tiles.  Static schedule: cluster_id,
  // cluster_id + num_clusters, ...  Cluster launch control (args.clc): the grid has
  // one cluster per tile; sequence index 0 is this cluster's own tile, index i >= 1
  // the tile of the cluster that the i-th request cancelled (slot (i - 1) % CLC_Q
  // of the response ring; requests come from the scheduler warp, and a slot is
  // refilled only after every epilogue warp of the cluster has finished the tile
  // it named: the epilogue is the last role to leave a tile).  Tiles past
  // num_tiles (grouped layouts launch an upper bound) are skipped, not treated as
  // the end.
  constexpr int kSeqEnd = 0x7FFFFFFF;
  struct Seq {
    int t;
    uint32_t i;
  };
  auto seq_begin = [&]() -> Seq {
    Seq sq{cluster_id, 0u};
    if (!args.clc && sq.t >= num_tiles) sq.t = kSeqEnd;
    return sq;
  };
  auto seq_next = [&](Seq& sq) {
    if (!args.clc) {
      sq.t += num_clusters;
      if (sq.t >= num_tiles) sq.t = kSeqEnd;
      return;
    }
    ++sq.i;
    const uint32_t r = sq.i - 1u;
    if (!pwait<true>(bar(C::BAR_CLC_FULL + r % C::CLC_Q), (r / C::CLC_Q) & 1u, ctl)) {
      sq.t = kSeqEnd;
      return;
    }
    const int c = *reinterpret_cast<volatile const int*>(smem + C::OFF_CLC + 16 + 4 * (r % C::CLC_Q));
    sq.t = c < 0 ? kSeqEnd : c;
  };
  // advances to the first tile at or after the cursor that this CTA works on
  auto seq_valid = [&](Seq& sq, Tile& tl) {
    while (sq.t != kSeqEnd && (sq.t >= num_tiles || !get_tile(sq.t, tl))) seq_next(sq);
  };
  // Epilogue warps, after finishing sequence index i >= 1: release its ring slot
  // (every epilogue warp of the cluster, on the leader's barrier).
  auto seq_step_epi = [&](Seq& sq) {
    if (args.clc && sq.i >= 1u) {
      const uint32_t q = (sq.i - 1u) % C::CLC_Q;
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lbar(C::BAR_CLC_EMPTY + q));
      __syncwarp();
    }
    seq_next(sq);
  };

  if (warp == 0) {
    // ============================================================ TMA producer
    ctl.role_bit = FGF8_DEVERR_ROLE_PRODUCER;
    int unit = 0;
    uint32_t phase = 0;
    bool ok = true;
    // bytes landing per K block: a thin tile's A box may be shorter than its stage
    const uint32_t a_tx = (C::kThin && args.a_box_rows > 0)
                              ? static_cast<uint32_t>(NCTA * (args.a_box_rows * 128 + C::B_BYTES))
                              : C::A_TX;
    for (Seq sq = seq_begin(); ok && sq.t != kSeqEnd; seq_next(sq)) {
      Tile tl;
      if (sq.t >= num_tiles || !get_tile(sq.t, tl)) continue;
      for (int kb0 = 0; kb0 < nkb; kb0 += C::KPU) {
        if (!pwait(bar(C::BAR_EMPTY + unit), phase ^ 1u, ctl)) { ok = false; break; }
        if (lane == 0) {
          const int nk = min(C::KPU, nkb - kb0);     // K blocks in this unit (the tail may be short)
          const uint32_t full = lbar(C::BAR_FULL + unit);
          if (leader) ptx::mbar_arrive_expect_tx(bar(C::BAR_FULL + unit), static_cast<uint32_t>(nk) * a_tx);
          for (int j = 0; j < nk; ++j) {
            const int stage = unit * C::KPU + j;
            const int kb = kb0 + j;
            tma_load_ab<NCTA>(sbase + C::OFF_A + stage * C::A_STRIDE, &tm_a, full, kb * C::BK, tl.a_row0);
            tma_load_ab<NCTA>(sbase + C::OFF_B + stage * C::B_STRIDE, &tm_b, full, kb * C::BK, tl.b_row0);
          }
        }
        __syncwarp();
        if (++unit == C::UNITS) { unit = 0; phase ^= 1u; }
      }
    }
    aborted = !ok;
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    // Issues straight from a named-barrier hand-off: the relay warp has already
    // waited for everything the unit needs, so this warp touches no shared memory
    // between MMAs and the tensor pipe never runs dry between units.
    ctl.role_bit = FGF8_DEVERR_ROLE_MMA;
    if (leader) {
      int unit = 0;
      int acc = 0;
      uint32_t gctr = 0u;            // scale-word groups consumed so far (all tiles)
      const uint32_t in_fmt = (KIND == Kind::F16 && args.in_bf16) ? 1u : 0u;
      const uint32_t idesc0 = C::kMX    ? idesc_mxf8(BN, C::MMA_M, 0, 0)
                              : C::kFP4 ? idesc_fp4(BN, C::MMA_M, KIND == Kind::MXF4)
                                        : idesc_dense(in_fmt, in_fmt, BN, C::MMA_M);
      // descriptors are linear in the address (start field = address >> 4)
      const uint64_t adesc0 = smem_desc_sw128(sbase + C::OFF_A);
      const uint64_t bdesc0 = smem_desc_sw128(sbase + C::OFF_B);
      for (Seq sq = seq_begin(); sq.t != kSeqEnd; seq_next(sq)) {
        Tile tl;
        if (sq.t >= num_tiles || !get_tile(sq.t, tl)) continue;
        uint32_t sf_col = 0;
        const bool ws_two = C::kWS && tl.row_limit > C::BM;   // weight-stationary: both sub-tiles hold rows
        (void)ws_two;
        for (int kb0 = 0; kb0 < nkb; kb0 += C::KPU) {
          named_bar_sync(C::HANDOFF_BAR, 64);
          ptx::tc_fence_after();
          const int nk = min(C::KPU, nkb - kb0);
          const int kl = kb0 + nk - 1;                   // last K block of the unit
          const bool group_end = C::kBS && ((kl + 1) % C::GK == 0 || kl == nkb - 1);
          if (lane == 0) {
            if constexpr (C::kBS) {
              if (kb0 % C::GK == 0) sf_col = tmem_base + C::SF_COL0 + (gctr % C::SF_SLOTS) * C::SF_SLOT_COLS;
            }
#pragma unroll
            for (int j = 0; j < C::KPU; ++j) {
              if (j < nk) {
                const int kb = kb0 + j;
                // FP32 scales: K block j of the unit has its own partial buffer
                // in the unit's slot
                const int buf = C::kF32S ? acc * C::KPU + j : acc;
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * C::PBN);
                const uint32_t stage = static_cast<uint32_t>(unit * C::KPU + j);
                const uint64_t ad = adesc0 + stage * (C::A_STRIDE >> 4);
                const uint64_t bd = bdesc0 + stage * (C::B_STRIDE >> 4);
                // UE8M0 FP8: byte kb % 4 of the group's scale word (a_sf_id, b_sf_id)
                const uint32_t sfid = static_cast<uint32_t>(kb & 3);
                const uint32_t id = C::kMX ? (idesc0 | (sfid << 4) | (sfid << 29)) : idesc0;
#pragma unroll
                for (int k = 0; k < C::MMAS_PER_STAGE; ++k) {
                  const uint32_t accum = C::kF32S ? (k > 0 ? 1u : 0u) : ((kb > 0 || k > 0) ? 1u : 0u);
                  uint32_t sfa = sf_col, sfb = sf_col + 4, idk = id;
                  if constexpr (C::kFP4) {
                    // word wi of the group: MXFP4 two instructions per word (bytes
                    // 0-1, then 2-3), NVFP4 one word per instruction (bytes 0-3)
                    const int wi = j * C::WPK + (KIND == Kind::MXF4 ? k / 2 : k);
                    const uint32_t fid = KIND == Kind::MXF4 ? 2u * static_cast<uint32_t>(k & 1) : 0u;
                    sfa = sf_col + 4u * wi;
                    sfb = sf_col + 4u * C::WG + static_cast<uint32_t>(C::NB_COLS * wi);
                    idk = idesc0 | (fid << 4) | (fid << 29);
                  }
                  if constexpr (C::kWS) {
                    // sub-tile 1 (A rows 128-255, 16 KB into the stage) reuses sub-tile
                    // 0's B from the collector; a tile with at most 128 valid rows
                    // skips it
                    const uint64_t ka = ad + (k * C::MMA_K_BYTES >> 4);
                    const uint64_t kbd = bd + (k * C::MMA_K_BYTES >> 4);
                    if (ws_two) {
                      tc_mma_ws_f8(d_tmem, ka, kbd, idk, accum, 1);
                      tc_mma_ws_f8(d_tmem + BN, ka + ((C::BM * 128) >> 4), kbd, idk, accum, 2);
                    } else {
                      tc_mma_ws_f8(d_tmem, ka, kbd, idk, accum, 0);
                    }
                  } else {
                    tc_mma<NCTA, KIND>(d_tmem, ad + (k * C::MMA_K_BYTES >> 4), bd + (k * C::MMA_K_BYTES >> 4), idk,
                                       sfa, sfb, accum);
                  }
                }
              }
            }
            if constexpr (C::kF32S) tc_commit_mc<NCTA>(bar(C::BAR_ACC_FULL + acc), pair_mask);
            tc_commit_mc<NCTA>(bar(C::BAR_EMPTY + unit), pair_mask);
            if (group_end) tc_commit_mc<NCTA>(bar(C::BAR_SF_FREE + gctr % C::SF_SLOTS), pair_mask);
          }
          __syncwarp();
          if (group_end) ++gctr;
          if constexpr (C::kF32S) acc = (acc + 1) % C::NSLOT;
          if (++unit == C::UNITS) unit = 0;
        }
        if constexpr (!C::kF32S) {
          if (lane == 0) tc_commit_mc<NCTA>(bar(C::BAR_ACC_FULL + acc), pair_mask);
          __syncwarp();
          if (++acc == C::NACC) acc = 0;
        }
      }
      // every tcgen05 op issued completes before TMEM is released; this wait
      // ignores an earlier abort and gets at least a second, and if it still
      // runs out the CTA takes the abort path, whose teardown grace period
      // covers MMAs still in flight
      if (lane == 0) tc_commit<NCTA>(bar(C::BAR_DRAIN));
      __syncwarp();
      PairWaitCtl drain = ctl;
      uint32_t zero = 0;
      drain.abort_flag = &zero;
      drain.peer_abort = 0;
      drain.timeout_ns = ctl.timeout_ns > 1000000000ull ? ctl.timeout_ns : 1000000000ull;
      if (!pwait(bar(C::BAR_DRAIN), 0u, drain)) {
        aborted = true;
        if (lane == 0) *abort_flag = 1u;
      }
    }
  } else if (warp < 2 + C::SF_WARPS) {
    // ============================================================ scale-factor writers
    if constexpr (C::kBS) {
    ctl.role_bit = FGF8_DEVERR_ROLE_PRODUCER;
    const uint32_t q = warp & 3u;                      // TMEM lane quarter this warp writes
    const bool loader = warp == 2;                     // lane 0 of this warp issues the loads
    constexpr int NB_COLS = C::NB_COLS;
    constexpr int WG = C::WG;
    struct Pos { Seq sq; int kb; Tile tl; };
    auto advance = [&](Pos& p) {
      p.kb += C::GK;
      if (p.kb >= nkb) {
        p.kb = 0;
        seq_next(p.sq);
        seq_valid(p.sq, p.tl);
      }
    };
    // The loader keeps SF_RING - 1 groups in flight ahead of the writers.  A ring
    // slot is reloaded once all four writers have read its previous group.
    Pos pl;
    pl.kb = 0;
    pl.sq = seq_begin();
    seq_valid(pl.sq, pl.tl);
    uint32_t gl = 0;
    auto issue_load = [&]() -> bool {
      const uint32_t r = gl % C::SF_RING;
      const uint32_t round = gl / C::SF_RING;
      if (round > 0 && !pwait(bar(C::BAR_SFC + r), (round - 1u) & 1u, ctl)) return false;
      if (lane == 0) {
        const uint32_t sfl = bar(C::BAR_SFL + r);
        ptx::mbar_arrive_expect_tx(sfl, C::SF_TX);
        // the group's WG words of every row (box: rows x WG words)
        const int w0 = pl.kb / C::GK * WG;
        const int sfa_row = (SCHED == Sched::Masked ? pl.tl.group * kq : 0) + w0;
        ptx::tma_load_2d(sbase + C::OFF_SFA + r * C::SFA_RING_BYTES, &tm_sfa, sfl, pl.tl.m_blk, sfa_row);
        ptx::tma_load_2d(sbase + C::OFF_SFB + r * C::SFB_RING_BYTES, &tm_sfb, sfl, pl.tl.n_blk * BN,
                         pl.tl.group * kq + w0);
      }
      __syncwarp();
      ++gl;
      advance(pl);
      return true;
    };
    bool ok = true;
    if (loader)
      for (int i = 0; ok && i < C::SF_RING - 1 && pl.sq.t != kSeqEnd; ++i) ok = issue_load();
    Pos pw;
    pw.kb = 0;
    pw.sq = seq_begin();
    seq_valid(pw.sq, pw.tl);
    uint32_t gctr = 0;
    while (ok && pw.sq.t != kSeqEnd) {
      if (loader && pl.sq.t != kSeqEnd && !issue_load()) { ok = false; break; }
      const uint32_t r = gctr % C::SF_RING;
      if (!pwait(bar(C::BAR_SFL + r), (gctr / C::SF_RING) & 1u, ctl)) { ok = false; break; }
      // word w of row 32 j + l -> lane l, column 4 w + j (SFA) or 4 WG + NB_COLS w + j
      // (SFB); the ring slot holds the words as [w][rows] (BM rows of A, BN of B;
      // rows past the tile are never read by the MMA)
      const uint32_t* sfa_s = reinterpret_cast<const uint32_t*>(smem + C::OFF_SFA + r * C::SFA_RING_BYTES);
      const uint32_t* sfb_s = reinterpret_cast<const uint32_t*>(smem + C::OFF_SFB + r * C::SFB_RING_BYTES);
      uint32_t a[WG][4], b[WG][NB_COLS];
#pragma unroll
      for (int w = 0; w < WG; ++w) {
#pragma unroll
        for (int j = 0; j < 4; ++j) a[w][j] = sfa_s[w * C::BM + 32 * j + lane];
#pragma unroll
        for (int j = 0; j < NB_COLS; ++j) b[w][j] = sfb_s[w * BN + 32 * j + lane];
      }
      // The slot is refilled by TMA, an async-proxy write: each lane orders its
      // generic-proxy reads of the slot before that write with a proxy fence
      // (without it the refill of the next round was seen by late readers, so a
      // lane quarter applied the scales of a group four groups ahead).
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(C::BAR_SFC + r));
      const uint32_t slot = gctr % C::SF_SLOTS;
      const uint32_t uses = gctr / C::SF_SLOTS;
      // the TMEM slot was last read by group gctr - SF_SLOTS
      if (uses > 0 && !pwait(bar(C::BAR_SF_FREE + slot), (uses - 1u) & 1u, ctl)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + ((q * 32u) << 16) + C::SF_COL0 + slot * C::SF_SLOT_COLS;
#pragma unroll
      for (int w = 0; w < WG; ++w) {
        tmem_st_x4(taddr + 4 * w, a[w][0], a[w][1], a[w][2], a[w][3]);
#pragma unroll
        for (int j = 0; j < NB_COLS; j += 4)
          tmem_st_x4(taddr + 4 * WG + NB_COLS * w + j, b[w][j], b[w][j + 1], b[w][j + 2], b[w][j + 3]);
      }
      tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lbar(C::BAR_SFR + slot));
      ++gctr;
      advance(pw);
    }
    aborted = !ok;
    }
  } else if (warp == C::SCHED_WARP) {
    // ============================================================ tile scheduler
    // Cluster launch control only, leader CTA: fills the ring with the tiles of
    // sequence indices 1, 2, ...  For each index it waits until every epilogue warp
    // of the cluster has finished the tile the slot held, then cancels clusters one
    // at a time (each request after the previous response has landed, so none is in
    // flight when the CTA exits) until one names a tile this grid works on, and
    // publishes that tile id to both CTAs; a request that finds no cluster left
    // publishes the end.  Clusters past the tiles (grouped layouts launch an upper
    // bound) are cancelled and dropped here, so every published tile is real work.
    if (args.clc && leader) {
      ctl.role_bit = FGF8_DEVERR_ROLE_PRODUCER;
      uint32_t sphase = 0;
      const uint32_t stage = sbase + C::OFF_CLC;
      for (uint32_t idx = 1;; ++idx) {
        const uint32_t q = (idx - 1u) % C::CLC_Q;
        if (idx > static_cast<uint32_t>(C::CLC_Q)) {
          const uint32_t prev = idx - 1u - C::CLC_Q;   // the slot's previous index is prev + 1
          if (!pwait(bar(C::BAR_CLC_EMPTY + q), (prev / C::CLC_Q) & 1u, ctl)) break;
        }
        int tile = -1;
        bool failed = false;
        for (;;) {
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar(C::BAR_CLC_STAGE), 16u);
            clc_try_cancel(stage, bar(C::BAR_CLC_STAGE));
          }
          __syncwarp();
          if (!pwait(bar(C::BAR_CLC_STAGE), sphase, ctl)) { failed = true; break; }
          sphase ^= 1u;
          const int c = clc_cluster(stage, C::CLUSTER);
          if (c < 0) break;
          Tile tl;
          if (c < num_tiles && get_tile(c, tl)) { tile = c; break; }
        }
        if (failed) break;
        if (lane == 0) {
          for (uint32_t rk = 0; rk < static_cast<uint32_t>(NCTA); ++rk) {
            const uint32_t slot = sbase + C::OFF_CLC + 16u + 4u * q;
            clc_publish(NCTA == 2 ? map_to_rank(slot, rk) : slot,
                        NCTA == 2 ? map_to_rank(bar(C::BAR_CLC_FULL + q), rk) : bar(C::BAR_CLC_FULL + q), tile);
          }
        }
        __syncwarp();
        if (tile < 0) break;
      }
    }
  } else if (warp == C::RELAY_WARP) {
    // ============================================================ relay
    // Waits, for the MMA warp, on everything a unit of MMAs needs (operands landed,
    // accumulator drained by the epilogue, scale slot written) and then meets it at
    // the named barrier; both walk the same schedule of units.  After a failed wait
    // it keeps meeting the barrier without waiting, so the MMA warp always finishes
    // its schedule (on stale data; the status word reports the failure).
    ctl.role_bit = FGF8_DEVERR_ROLE_MMA;
    if (leader) {
      int unit = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      uint32_t gctr = 0u;
      bool ok = true;
      for (Seq sq = seq_begin(); sq.t != kSeqEnd; seq_next(sq)) {
        Tile tl;
        if (sq.t >= num_tiles || !get_tile(sq.t, tl)) continue;
        if constexpr (!C::kF32S) {
          if (ok) ok = pwait(bar(C::BAR_ACC_EMPTY + acc), acc_phase ^ 1u, ctl);
        }
        for (int kb0 = 0; kb0 < nkb; kb0 += C::KPU) {
          const int nk = min(C::KPU, nkb - kb0);
          if constexpr (C::kF32S) {
            // the slot of partial buffers the unit writes has been drained by the promotion
            if (ok) ok = pwait(bar(C::BAR_ACC_EMPTY + acc), acc_phase ^ 1u, ctl);
            if (++acc == C::NSLOT) { acc = 0; acc_phase ^= 1u; }
          }
          if constexpr (C::kBS) {
            if (ok && kb0 % C::GK == 0)
              ok = pwait(bar(C::BAR_SFR + gctr % C::SF_SLOTS), (gctr / C::SF_SLOTS) & 1u, ctl);
          }
          if (ok) ok = pwait(bar(C::BAR_FULL + unit), phase, ctl);
          named_bar_sync(C::HANDOFF_BAR, 64);
          const int kl = kb0 + nk - 1;
          if (C::kBS && ((kl + 1) % C::GK == 0 || kl == nkb - 1)) ++gctr;
          if (++unit == C::UNITS) { unit = 0; phase ^= 1u; }
        }
        if constexpr (!C::kF32S) {
          if (++acc == C::NACC) { acc = 0; acc_phase ^= 1u; }
        }
      }
      aborted = !ok;
    }
  } else if constexpr (!C::kF32S && C::EPI_WARPS == 4) {
    // ============================================================ epilogue
    ctl.role_bit = FGF8_DEVERR_ROLE_EPILOGUE;
    const uint32_t q = warp & 3u;
    const bool bf16 = args.out_bf16 != 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t epi_chunks = 0;   // chunks staged so far (TMA-store epilogue)
    (void)epi_chunks;
    bool ok = true;
    for (Seq sq = seq_begin(); sq.t != kSeqEnd; seq_step_epi(sq)) {
      Tile tl;
      if (sq.t >= num_tiles || !get_tile(sq.t, tl)) continue;
      if (!pwait(bar(C::BAR_ACC_FULL + acc), acc_phase, ctl)) { ok = false; break; }
      ptx::tc_fence_after();
      const int r = static_cast<int>(q * C::QROWS + lane);
      bool row_ok = lane < static_cast<uint32_t>(C::QROWS) && r < tl.row_limit;
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
      if constexpr (C::kFuseQuant) {
        {
          // 1x128 quantization of the output rows: per 128-column group, the values
          // rounded to bf16 exactly as D would be stored, their max |x|, the scale
          // and the codes.  Rows between M and the scale table's padded row count
          // get zero scales, and the last group's row fills the unused bytes of
          // its UE8M0 word with zeros, as quantize_1x128 leaves them.
          const int grow = tl.a_row0 + r;
#pragma unroll 1
          for (int g = 0; g < BN / 128; ++g) {
            uint32_t hv[64];
            float amax = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t v[32];
              ptx::tmem_ld_32x32b_x32(taddr + 128u * g + 32u * c, v);
              ptx::tmem_wait_ld();
              ptx::reg_fence(v);
              if (c == 3 && g == BN / 128 - 1) {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(lbar(C::BAR_ACC_EMPTY + acc));
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const uint32_t h = pack_2x16(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), true);
                hv[16 * c + j] = h;
                amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(h << 16)), fabsf(__uint_as_float(h & 0xFFFF0000u))));
              }
            }
            fused_group_out(args, PackedBf16{hv}, amax, (tl.n_blk * BN) / 128 + g, grow, row_ok);
          }
          if (++acc == C::NACC) { acc = 0; acc_phase ^= 1u; }
          continue;
        }
      }
      // 32-column chunks, then a 16-column tail when BN is an odd multiple of 16;
      // the accumulator is released after its last load
      constexpr int NCH = BN / 32;
      constexpr bool TAIL = (BN % 32) != 0;
      // dense: the tensor map clips rows past M; grouped: every row of the warp valid
      bool tma_rows = true;
      if constexpr (C::kTmaStore && SCHED != Sched::Dense) tma_rows = __all_sync(0xffffffffu, row_ok);
      if (C::kTmaStore && tma_rows) {
        // each chunk, rounded to 16 bits, goes to one of this warp's two staging
        // buffers (row `lane` = 64 bytes) and lane 0 stores it by TMA; the buffer
        // is rewritten only after the store issued two chunks earlier has read it
        const uint32_t stage0 = sbase + C::OFF_EPI + (warp - C::EPI_WARP0) * 2u * C::EPI_CHUNK_BYTES;
        const int y = tl.a_row0 + static_cast<int>(q) * 32;     // first row of this warp's 32
#pragma unroll 1
        for (int c = 0; c < NCH; ++c) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(taddr + 32u * c, v);
          ptx::tmem_wait_ld();
          ptx::reg_fence(v);
          if (c == NCH - 1) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(lbar(C::BAR_ACC_EMPTY + acc));
          }
          const uint32_t buf = stage0 + (epi_chunks & 1u) * C::EPI_CHUNK_BYTES;
          if (lane == 0) ptx::bulk_wait_group_read<1>();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float* f = reinterpret_cast<const float*>(v) + 8 * j;
            st_shared_v4(buf + lane * 64u + 16u * j, pack_2x16(f[0], f[1], bf16), pack_2x16(f[2], f[3], bf16),
                         pack_2x16(f[4], f[5], bf16), pack_2x16(f[6], f[7], bf16));
          }
          ptx::fence_proxy_async_smem();   // the generic writes, before the async-proxy read
          __syncwarp();
          const int x = tl.n_blk * BN + 32 * c;
          // rows of D's 2-D view: M, or G x Mmax with the experts stacked (masked)
          const int d_rows = SCHED == Sched::Masked ? G * M : M;
          if (lane == 0 && y < d_rows && x < N) {
            ptx::tma_store_2d(&tm_d, buf, x, y);
            ptx::bulk_commit_group();
          }
          ++epi_chunks;
        }
        if (++acc == C::NACC) { acc = 0; acc_phase ^= 1u; }
        continue;
      }
#pragma unroll 1
      for (int c = 0; c < NCH; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + 32u * c, v);
        ptx::tmem_wait_ld();
        ptx::reg_fence(v);
        if (!TAIL && c == NCH - 1) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lbar(C::BAR_ACC_EMPTY + acc));
        }
        if (row_ok)
          store_row32(args.D, row_off, tl.n_blk * BN + 32 * c, N, reinterpret_cast<const float*>(v), bf16);
      }
      if constexpr (TAIL) {
        uint32_t v[16];
        ptx::tmem_ld_32x32b_x16(taddr + 32u * NCH, v);
        ptx::tmem_wait_ld();
        ptx::reg_fence(v);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(lbar(C::BAR_ACC_EMPTY + acc));
        if (row_ok)
          store_row16(args.D, row_off, tl.n_blk * BN + 32 * NCH, N, reinterpret_cast<const float*>(v), bf16);
      }
      if (++acc == C::NACC) { acc = 0; acc_phase ^= 1u; }
    }
    if constexpr (C::kTmaStore) {
      // every store this warp issued has completed before the CTA may exit
      if (lane == 0) ptx::bulk_wait_group<0>();
      __syncwarp();
    }
    aborted = !ok;
  } else if constexpr (!C::kF32S) {
    // ============================================================ drain epilogue
    // One accumulator buffer: two warps per TMEM lane quarter each drain 128
    // columns into registers (rounded to 16 bits) and release the buffer at once,
    // then store them (or quantize them 1x128 when the output is quantized).
    ctl.role_bit = FGF8_DEVERR_ROLE_EPILOGUE;
    constexpr int HALF = BN / 2;
    static_assert(HALF == 128, "drain epilogue: 128 columns per warp");
    const uint32_t q = warp & 3u;
    const int h = static_cast<int>(warp - C::EPI_WARP0) >> 2;
    const bool bf16 = args.out_bf16 != 0 || C::kFuseQuant;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (Seq sq = seq_begin(); sq.t != kSeqEnd; seq_step_epi(sq)) {
      Tile tl;
      if (sq.t >= num_tiles || !get_tile(sq.t, tl)) continue;
      if (!pwait(bar(C::BAR_ACC_FULL + acc), acc_phase, ctl)) { ok = false; break; }
      ptx::tc_fence_after();
      const int r = static_cast<int>(q * C::QROWS + lane);
      bool row_ok = lane < static_cast<uint32_t>(C::QROWS) && r < tl.row_limit;
      if constexpr (SCHED == Sched::Contiguous) {
        if (row_ok) {
          const int g = __ldg(args.m_indices + tl.a_row0 + r);
          if (g != tl.group) {
            if (g >= 0) atomicOr(args.status, FGF8_DEVERR_INPUT);
            row_ok = false;
          }
        }
      }
      const uint32_t taddr =
          tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(acc * BN + h * HALF);
      const int col0 = tl.n_blk * BN + h * HALF;
      uint32_t hv[64];
      float amax = 0.0f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + 32u * c, v);
        ptx::tmem_wait_ld();
        ptx::reg_fence(v);
        if (c == 3) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lbar(C::BAR_ACC_EMPTY + acc));
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t p = pack_2x16(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), bf16);
          hv[16 * c + j] = p;
          if constexpr (C::kFuseQuant)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(p << 16)), fabsf(__uint_as_float(p & 0xFFFF0000u))));
        }
      }
      // everything after the drain works from registers only
      ptx::reg_fence(hv);
      if constexpr (C::kFuseQuant) {
        fused_group_out(args, PackedBf16{hv}, amax, col0 / 128, tl.a_row0 + r, row_ok);  // skips groups past N
      } else if (row_ok) {
        const size_t row_off = static_cast<size_t>(tl.a_row0 + r) * static_cast<size_t>(N);
#pragma unroll
        for (int c = 0; c < 4; ++c) store_row32_packed(args.D, row_off, col0 + 32 * c, N, hv + 16 * c);
      }
      if (++acc == C::NACC) { acc = 0; acc_phase ^= 1u; }
    }
    aborted = !ok;
  } else {
    // ============================================================ promotion
    // Warp (q, h): TMEM lane quarter q; h selects the column half of the partial,
    // or, on the weight-stationary tile, the 128-row sub-tile (all its columns).
    ctl.role_bit = FGF8_DEVERR_ROLE_EPILOGUE;
    constexpr int HALF = C::kWS ? BN : BN / 2;        // columns per warp
    const uint32_t q = warp & 3u;
    const int h = static_cast<int>(warp - C::EPI_WARP0) >> 2;
    const int row_off_h = C::kWS ? h * C::BM : 0;      // first row of this warp's sub-tile
    const int col_off_h = C::kWS ? 0 : h * HALF;       // first column of this warp's half
    const bool bf16 = args.out_bf16 != 0;
    const int nkb128 = K / 128;
    const int nnb = (N + 127) / 128;
    const int ld_a = (M + 3) / 4 * 4;
    const int r = static_cast<int>(q * C::QROWS + lane);
    // The scale stream walks the same tiles and units as the promotion below, one
    // unit earlier, with plain global loads into registers (the MMAs keep shared
    // memory busy, so scales do not go through it).  The loads are unconditional
    // so that nothing waits for them before the next unit: a row past the tile's
    // valid rows, or columns past N, read the table's first entries instead, and
    // those values only reach outputs that are never stored.
    Seq s_sq = seq_begin();
    int s_kb0 = 0;
    const float* s_pa = args.sfa_f32;
    const float* s_pb = args.sfb_f32;
    auto stream_seek = [&]() {  // first tile at or after the stream's cursor that this CTA works on
      s_pa = args.sfa_f32;
      s_pb = args.sfb_f32;
      Tile st;
      seq_valid(s_sq, st);
      if (s_sq.t == kSeqEnd) return;
      const int c0 = st.n_blk * BN + col_off_h;
      if (lane < static_cast<uint32_t>(C::QROWS) && row_off_h + r < st.row_limit)
        s_pa = args.sfa_f32 + (SCHED == Sched::Masked ? static_cast<size_t>(st.group) * nkb128 * ld_a : 0) +
               (st.m_blk + row_off_h + r);
      if (c0 < N) s_pb = args.sfb_f32 + (static_cast<size_t>(st.group) * nnb + c0 / 128) * nkb128;
    };
    float na[C::KPU], nb[C::KPU];  // the next unit's scales, in flight
    auto stream_fetch = [&]() {
      if (s_sq.t != kSeqEnd) {
#pragma unroll
        for (int j = 0; j < C::KPU; ++j) {
          const int kb = min(s_kb0 + j, nkb - 1);  // a short tail unit repeats its last K block
          na[j] = __ldg(s_pa + static_cast<size_t>(kb) * ld_a);
          nb[j] = __ldg(s_pb + kb);
        }
        s_kb0 += C::KPU;
        if (s_kb0 >= nkb) {
          s_kb0 = 0;
          seq_next(s_sq);
          stream_seek();
        }
      }
    };
    stream_seek();
    stream_fetch();
    int pslot = 0;
    uint32_t pphase = 0;
    bool ok = true;
    // chunks of CH columns of each partial, double-buffered across the unit: the
    // load of chunk c + 1 is in flight while chunk c is accumulated; the slot is
    // released as soon as its last chunk has landed
    constexpr int CH = (HALF >= 128 || C::KPU > 2) ? 16 : 32;
    constexpr int NCH = HALF / CH;
    float accv[HALF];
    auto promote_unit = [&](auto nk_c, const float (&sc)[C::KPU], uint32_t taddr) {
      constexpr int TOT = decltype(nk_c)::value * NCH;
      uint32_t va[CH], vb[CH];
      tmem_ld_chunk(taddr, va);
      ptx::tmem_wait_ld();
      ptx::reg_fence(va);
#pragma unroll
      for (int c = 0; c < TOT; ++c) {
        uint32_t(&cur)[CH] = (c & 1) ? vb : va;
        uint32_t(&nxt)[CH] = (c & 1) ? va : vb;
        if (c + 1 < TOT) {
          const int n1 = c + 1;
          tmem_ld_chunk(taddr + static_cast<uint32_t>((n1 / NCH) * C::PBN + CH * (n1 % NCH)), nxt);
        } else {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lbar(C::BAR_ACC_EMPTY + pslot));
        }
        const float sj = sc[c / NCH];
        float* a0 = accv + CH * (c % NCH);
#pragma unroll
        for (int j = 0; j < CH; j += 2)
          ptx::ffma2(a0[j], a0[j + 1], sj, __uint_as_float(cur[j]), __uint_as_float(cur[j + 1]));
        if (c + 1 < TOT) {
          ptx::tmem_wait_ld();
          ptx::reg_fence(nxt);
        }
      }
    };
    for (Seq sq = seq_begin(); ok && sq.t != kSeqEnd; seq_step_epi(sq)) {
      Tile tl;
      if (sq.t >= num_tiles || !get_tile(sq.t, tl)) continue;
      bool row_ok = lane < static_cast<uint32_t>(C::QROWS) && row_off_h + r < tl.row_limit;
      // a warp whose rows are all past the tile's valid rows (the last M tile of
      // a masked expert or contiguous segment, or a weight-stationary sub-tile that
      // got no MMAs) promotes nothing and only keeps the slot handshake
      const bool idle = row_off_h + static_cast<int>(q) * C::QROWS >= tl.row_limit;
      if constexpr (SCHED == Sched::Contiguous) {
        if (row_ok) {
          const int g = __ldg(args.m_indices + tl.a_row0 + r);
          if (g != tl.group) {
            if (g >= 0) atomicOr(args.status, FGF8_DEVERR_INPUT);
            row_ok = false;
          }
        }
      }
      const int col0 = tl.n_blk * BN + col_off_h;
#pragma unroll
      for (int i = 0; i < HALF; ++i) accv[i] = 0.0f;
      for (int kb0 = 0; kb0 < nkb; kb0 += C::KPU) {
        float sc[C::KPU];
#pragma unroll
        for (int j = 0; j < C::KPU; ++j) sc[j] = na[j] * nb[j];
        stream_fetch();  // the next unit's loads run during this unit's promotion
        if (!pwait(bar(C::BAR_ACC_FULL + pslot), pphase, ctl)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t taddr =
            tmem_base + ((q * 32u) << 16) + static_cast<uint32_t>(pslot * C::KPU * C::PBN + h * HALF);
        // a tile's last unit may hold fewer K blocks
        const int nk = min(C::KPU, nkb - kb0);
        if (idle) {
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(lbar(C::BAR_ACC_EMPTY + pslot));
        } else if (nk == C::KPU) promote_unit(std::integral_constant<int, C::KPU>{}, sc, taddr);
        else if (C::KPU > 3 && nk == 3) promote_unit(std::integral_constant<int, (C::KPU > 3 ? 3 : 1)>{}, sc, taddr);
        else if (C::KPU > 2 && nk == 2) promote_unit(std::integral_constant<int, (C::KPU > 2 ? 2 : 1)>{}, sc, taddr);
        else promote_unit(std::integral_constant<int, 1>{}, sc, taddr);
        if (++pslot == C::NSLOT) { pslot = 0; pphase ^= 1u; }
      }
      if (!ok) break;
      if constexpr (C::kFuseQuant) {
        {
          // 1x128 quantization of the output: this warp's 128 columns of the row
          // are one group, quantized from the accumulators rounded to bf16
          float amax = 0.0f;
#pragma unroll
          for (int j = 0; j < HALF; ++j) amax = fmaxf(amax, fabsf(bf16_round(accv[j])));
          fused_group_out(args, RoundedF32{accv}, amax, col0 / 128, tl.a_row0 + r, row_ok);
          continue;
        }
      }
      if (row_ok) {
        const size_t row_off = static_cast<size_t>(tl.a_row0 + row_off_h + r) * static_cast<size_t>(N);
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c) store_row32(args.D, row_off, col0 + 32 * c, N, accv + 32 * c, bf16);
      }
    }
    aborted = !ok;
  }

  // ---------------------------------------------------------------- teardown
  // After an abort, loads or MMAs may still be in flight toward this CTA's shared
  // memory or TMEM: give them time to land (a few microseconds suffice) before the
  // CTA may exit.  Normal completion never takes this path.
  if (__syncthreads_or(aborted ? 1 : 0) || *abort_flag) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < 200000ull) __nanosleep(1000);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if constexpr (C::CLUSTER > 1) cluster_sync_all();
  if (warp == 1) {
    ptx::tc_fence_after();
    tc_dealloc<NCTA>(tmem_base, C::TMEM_ALLOC);
  }
}

}  // namespace fgf8

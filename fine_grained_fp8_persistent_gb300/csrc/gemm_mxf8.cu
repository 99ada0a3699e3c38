// gemm_mxf8.cu -- launcher of the E4M3 GEMMs with power-of-two (UE8M0) scales:
// the block-scaled tcgen05.mma path (dense, grouped contiguous, grouped masked).
#include "gemm_launch.cuh"

namespace fgf8 {
namespace {

template <Sched S>
int launch_cfg(const TileCfg& c, const GemmArgs& a, const TensorMaps& tm, long long tiles, bool thin,
               cudaStream_t stream) {
  if constexpr (S == Sched::Dense) {
    if (a.dq != nullptr) {  // output quantized 1x128 in the epilogue
      if (c.bn == 256) return launch_persistent<Kind::MXF8, S, 2, 256, 6, 1, 128, true>(a, tm, tiles, stream);
      if (c.ncta == 2) return launch_persistent<Kind::MXF8, S, 2, 128, 8, 2, 128, true>(a, tm, tiles, stream);
      return launch_persistent<Kind::MXF8, S, 1, 128, 6, 2, 128, true>(a, tm, tiles, stream);
    }
    // one 256-wide accumulator (drained by 8 epilogue warps)
    if (c.ncta == 2 && c.bn == 256) return launch_persistent<Kind::MXF8, S, 2, 256, 6, 1>(a, tm, tiles, stream);
    if (thin) {  // at most 64 rows: 64-row A stages (boxes of M rounded to 8), A and B interleaved per 16 KB stage
      switch (c.bn) {
        case 64: return launch_persistent<Kind::MXF8, S, 1, 64, 12, 2, 64>(a, tm, tiles, stream);
        case 48: return launch_persistent<Kind::MXF8, S, 1, 48, 12, 2, 64>(a, tm, tiles, stream);
        default: return launch_persistent<Kind::MXF8, S, 1, 32, 12, 2, 64>(a, tm, tiles, stream);
      }
    }
  }
  if (c.ncta == 2) {
    if (c.bn == 224) return launch_persistent<Kind::MXF8, S, 2, 224, 6>(a, tm, tiles, stream);
    return launch_persistent<Kind::MXF8, S, 2, 128, 8>(a, tm, tiles, stream);
  }
  switch (c.bn) {
    case 224: return launch_persistent<Kind::MXF8, S, 1, 224, 4>(a, tm, tiles, stream);
    case 128: return launch_persistent<Kind::MXF8, S, 1, 128, 6>(a, tm, tiles, stream);
    case 64: return launch_persistent<Kind::MXF8, S, 1, 64, 8>(a, tm, tiles, stream);
    case 48: return launch_persistent<Kind::MXF8, S, 1, 48, 8>(a, tm, tiles, stream);
    default: return launch_persistent<Kind::MXF8, S, 1, 32, 8>(a, tm, tiles, stream);
  }
}

}  // namespace

int launch_gemm_mxf8(const GemmArgs& a, Sched sched, const void* Aq, const void* SFA,
                     const void* Bq, const void* SFB, cudaStream_t stream) {
  // relative tile times: see pick_cfg (the 64, 48 and 32 widths are extrapolated;
  // the 256-wide pair tile, measured at 4096 x 7168 x 7168, ties the 224-wide one).
  // The contiguous layout takes CTA pairs when its expert segments fit the
  // scheduler's table (pairs are then cut per segment), else one CTA per tile.
  static const TileCfg dense_cands[] = {{2, 224, 18.4}, {2, 128, 14.4}, {1, 224, 23.5},
                                        {1, 128, 14.9}, {1, 64, 9.1},   {1, 48, 8.0},
                                        {1, 32, 6.3},   {2, 256, 24.2}};
  static const TileCfg pair_cands[] = {{2, 224, 18.4}, {2, 128, 14.4}, {1, 224, 23.5},
                                       {1, 128, 14.9}, {1, 64, 9.1},   {1, 48, 8.0},
                                       {1, 32, 6.3}};
  static const TileCfg single_cands[] = {{1, 224, 23.5}, {1, 128, 14.9}, {1, 64, 9.1},
                                         {1, 48, 8.0},   {1, 32, 6.3}};
  // fused output quantization: 128-wide tiles hold whole 1x128 groups
  static const TileCfg fused_cands[] = {{2, 256, 24.2}, {2, 128, 14.4}, {1, 128, 14.9}};
  const bool pairs = sched != Sched::Contiguous || (a.M + 127) / 128 <= kMaxContiguousPairBlocks;
  const bool fused = a.dq != nullptr;
  if (fused && sched != Sched::Dense) return set_error(2, "fused output quantization: dense layout only");
  const TileCfg* cands = fused ? fused_cands : sched == Sched::Dense ? dense_cands : (pairs ? pair_cands : single_cands);
  const int n = fused ? kCount(fused_cands)
                : sched == Sched::Dense ? kCount(dense_cands) : (pairs ? kCount(pair_cands) : kCount(single_cands));
  const TileCfg c = cands[pick_cfg(a, sched, cands, n)];
  const long long a_rows = (sched == Sched::Masked) ? static_cast<long long>(a.G) * a.M : a.M;
  const long long b_rows = static_cast<long long>(a.G) * a.N;
  GemmArgs at = a;
  const bool thin = sched == Sched::Dense && a.M <= 64 && c.ncta == 1 && c.bn <= 64;
  at.a_box_rows = thin ? thin_a_box_rows(a.M) : 0;
  TensorMaps tm;
  if (make_operand_maps(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Aq, a_rows, Bq, b_rows, a.K, c.bn / c.ncta,
                        thin ? thin_a_box_rows(a.M) : 128))
    return 4;
  // Packed UE8M0 scale words: one int32 per row per four K blocks, rows padded to 4.
  const long long kq = (a.K / 128 + 3) / 4;
  const long long lda = (a.M + 3) / 4 * 4;
  const long long ldn = (a.N + 3) / 4 * 4;
  const long long sfa_rows = kq * (sched == Sched::Masked ? a.G : 1);
  if (!encode_tmap_2d(&tm.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFA, lda, sfa_rows, lda * 4, 128, 1, false))
    return 4;
  if (!encode_tmap_2d(&tm.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFB, ldn, kq * a.G, ldn * 4, c.bn, 1, false))
    return 4;
  const long long tiles = tile_count(a, sched, c);
  switch (sched) {
    case Sched::Dense: return launch_cfg<Sched::Dense>(c, at, tm, tiles, thin, stream);
    case Sched::Contiguous: return launch_cfg<Sched::Contiguous>(c, at, tm, tiles, false, stream);
    default: return launch_cfg<Sched::Masked>(c, at, tm, tiles, false, stream);
  }
}

}  // namespace fgf8

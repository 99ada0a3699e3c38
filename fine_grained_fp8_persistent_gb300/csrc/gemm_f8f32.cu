// gemm_f8f32.cu -- launcher of the E4M3 GEMMs with FP32 scales: per-128-K partials
// in TMEM promoted on the CUDA cores (dense, grouped contiguous, grouped masked).
#include "gemm_launch.cuh"

namespace fgf8 {
namespace {

template <Sched S>
int launch_cfg(const TileCfg& c, const GemmArgs& a, const TensorMaps& tm, long long tiles, bool thin,
               cudaStream_t stream) {
  if constexpr (S == Sched::Dense) {
    // output quantized 1x128 in the epilogue (the fused launcher picks the 256-wide tile)
    if (a.dq != nullptr) return launch_persistent<Kind::F8F32, S, 1, 256, 4, 2, 128, true>(a, tm, tiles, stream);
    // at most 64 rows: 64-row A stages, more stages in flight
    if (thin) return launch_persistent<Kind::F8F32, S, 1, 64, 12, 8, 64>(a, tm, tiles, stream);
  }
  // weight-stationary: 256 rows as two .ws sub-tiles sharing B (dense and masked
  // layouts; a 256-row tile could straddle two contiguous expert segments)
  if constexpr (S != Sched::Contiguous) {
    if (c.ws) return launch_persistent<Kind::F8F32, S, 1, 128, 4, 2, 256>(a, tm, tiles, stream);
  }
  // pairs: 128-wide tiles so that four partial buffers fit in TMEM
  if (c.ncta == 2) return launch_persistent<Kind::F8F32, S, 2, 128, 8, 4>(a, tm, tiles, stream);
  switch (c.bn) {
    case 256: return launch_persistent<Kind::F8F32, S, 1, 256, 4>(a, tm, tiles, stream);
    case 128: return launch_persistent<Kind::F8F32, S, 1, 128, 6, 4>(a, tm, tiles, stream);
    default: return launch_persistent<Kind::F8F32, S, 1, 64, 8, 4>(a, tm, tiles, stream);
  }
}

}  // namespace

int launch_gemm_f8f32(const GemmArgs& a, Sched sched, const void* Aq, const void* Bq,
                      cudaStream_t stream) {
  // relative tile times (see pick_cfg), measured on M=4096, N=K=7168: the
  // 128-wide tiles and the 256-wide one take the same time per output element,
  // and the 128-wide single-CTA tile is faster on the grouped layouts
  // (the weight-stationary tile is selectable by FGF8_FORCE_TILE=1x128ws; its
  // relative time keeps it out of the automatic choice, see the design notes)
  static const TileCfg pair_cands[] = {{2, 128, 17.0}, {1, 256, 34.0}, {1, 128, 16.8}, {1, 64, 16.0}};
  static const TileCfg ws_cands[] = {{2, 128, 17.0}, {1, 256, 34.0}, {1, 128, 16.8}, {1, 64, 16.0},
                                     {1, 128, 1e9, true}};
  static const TileCfg single_cands[] = {{1, 256, 34.0}, {1, 128, 16.8}, {1, 64, 16.0}};
  // the contiguous layout takes CTA pairs when its expert segments fit the
  // scheduler's table (pairs are then cut per segment)
  // fused output quantization: the 256-wide tile, whose promotion warps hold whole
  // 1x128 groups of a row
  static const TileCfg fused_cands[] = {{1, 256, 34.0}};
  const bool fused = a.dq != nullptr;
  if (fused && sched != Sched::Dense) return set_error(2, "fused output quantization: dense layout only");
  const bool pairs = sched != Sched::Contiguous || (a.M + 127) / 128 <= kMaxContiguousPairBlocks;
  const bool ws_ok = sched != Sched::Contiguous;
  const TileCfg* cands = fused ? fused_cands : ws_ok ? ws_cands : pairs ? pair_cands : single_cands;
  const int n = fused ? kCount(fused_cands) : ws_ok ? kCount(ws_cands) : pairs ? kCount(pair_cands) : kCount(single_cands);
  const TileCfg c = cands[pick_cfg(a, sched, cands, n)];
  const long long a_rows = (sched == Sched::Masked) ? static_cast<long long>(a.G) * a.M : a.M;
  const long long b_rows = static_cast<long long>(a.G) * a.N;
  GemmArgs at = a;
  const bool thin = sched == Sched::Dense && a.M <= 64 && c.ncta == 1 && c.bn == 64;
  at.a_box_rows = thin ? thin_a_box_rows(a.M) : 0;
  TensorMaps tm;
  if (make_operand_maps(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Aq, a_rows, Bq, b_rows, a.K, c.bn / c.ncta,
                        thin ? thin_a_box_rows(a.M) : c.ws ? 256 : 128))
    return 4;
  const long long tiles = tile_count(a, sched, c);
  switch (sched) {
    case Sched::Dense: return launch_cfg<Sched::Dense>(c, at, tm, tiles, thin, stream);
    case Sched::Contiguous: return launch_cfg<Sched::Contiguous>(c, at, tm, tiles, false, stream);
    default: return launch_cfg<Sched::Masked>(c, at, tm, tiles, false, stream);
  }
}

}  // namespace fgf8

// gemm_mxf8.cu -- launcher of the E4M3 GEMMs with power-of-two (UE8M0) scales:
// the block-scaled tcgen05.mma path (dense, grouped contiguous, grouped masked).
#include "gemm_launch.cuh"

namespace fgf8 {
namespace {

template <Sched S>
int launch_bn(int bn, const GemmArgs& a, const TensorMaps& tm, int grid, cudaStream_t stream) {
  switch (bn) {
    case 224: return launch_instance<Kind::MXF8, S, 224, 4>(a, tm, grid, stream);
    case 128: return launch_instance<Kind::MXF8, S, 128, 6>(a, tm, grid, stream);
    case 64: return launch_instance<Kind::MXF8, S, 64, 8>(a, tm, grid, stream);
    default: return launch_instance<Kind::MXF8, S, 32, 8>(a, tm, grid, stream);
  }
}

}  // namespace

int launch_gemm_mxf8(const GemmArgs& a, Sched sched, const void* Aq, const void* SFA,
                     const void* Bq, const void* SFB, cudaStream_t stream) {
  static const int cands[] = {224, 128, 64, 32};
  const int bn = pick_bn(a, sched, cands, 4);
  const long long a_rows = (sched == Sched::Masked) ? static_cast<long long>(a.G) * a.M : a.M;
  const long long b_rows = static_cast<long long>(a.G) * a.N;
  TensorMaps tm;
  if (make_operand_maps(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Aq, a_rows, Bq, b_rows, a.K, bn))
    return 4;
  // Packed UE8M0 scale words: one int32 per row per four K blocks, rows padded to 4.
  const long long kq = (a.K / 128 + 3) / 4;
  const long long lda = (a.M + 3) / 4 * 4;
  const long long ldn = (a.N + 3) / 4 * 4;
  const long long sfa_rows = kq * (sched == Sched::Masked ? a.G : 1);
  if (!encode_tmap_2d(&tm.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFA, lda, sfa_rows, lda * 4, 128, 1,
                      false))
    return 4;
  if (!encode_tmap_2d(&tm.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFB, ldn, kq * a.G, ldn * 4, bn, 1,
                      false))
    return 4;
  const int grid = persistent_grid(tile_count(a, sched, bn));
  switch (sched) {
    case Sched::Dense: return launch_bn<Sched::Dense>(bn, a, tm, grid, stream);
    case Sched::Contiguous: return launch_bn<Sched::Contiguous>(bn, a, tm, grid, stream);
    default: return launch_bn<Sched::Masked>(bn, a, tm, grid, stream);
  }
}

}  // namespace fgf8

// gemm_f8f32.cu -- launcher of the E4M3 GEMMs with FP32 scales: per-128-K partials
// in TMEM promoted on the CUDA cores (dense, grouped contiguous, grouped masked).
#include "gemm_launch.cuh"

namespace fgf8 {
namespace {

template <Sched S>
int launch_bn(int bn, const GemmArgs& a, const TensorMaps& tm, int grid, cudaStream_t stream) {
  switch (bn) {
    case 256: return launch_instance<Kind::F8F32, S, 256, 4>(a, tm, grid, stream);
    case 128: return launch_instance<Kind::F8F32, S, 128, 6>(a, tm, grid, stream);
    default: return launch_instance<Kind::F8F32, S, 64, 8>(a, tm, grid, stream);
  }
}

}  // namespace

int launch_gemm_f8f32(const GemmArgs& a, Sched sched, const void* Aq, const void* Bq,
                      cudaStream_t stream) {
  static const int cands[] = {256, 128, 64};
  const int bn = pick_bn(a, sched, cands, 3);
  const long long a_rows = (sched == Sched::Masked) ? static_cast<long long>(a.G) * a.M : a.M;
  const long long b_rows = static_cast<long long>(a.G) * a.N;
  TensorMaps tm;
  if (make_operand_maps(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Aq, a_rows, Bq, b_rows, a.K, bn))
    return 4;
  const int grid = persistent_grid(tile_count(a, sched, bn));
  switch (sched) {
    case Sched::Dense: return launch_bn<Sched::Dense>(bn, a, tm, grid, stream);
    case Sched::Contiguous: return launch_bn<Sched::Contiguous>(bn, a, tm, grid, stream);
    default: return launch_bn<Sched::Masked>(bn, a, tm, grid, stream);
  }
}

}  // namespace fgf8

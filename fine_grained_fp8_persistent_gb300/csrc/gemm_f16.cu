// gemm_f16.cu -- launcher of the dense 16-bit (fp16/bf16) NT GEMM.
#include "gemm_launch.cuh"

namespace fgf8 {

int launch_gemm_f16(const GemmArgs& a, const void* A, const void* B, cudaStream_t stream) {
  static const int cands[] = {256, 128};
  const int bn = pick_bn(a, Sched::Dense, cands, 2);
  TensorMaps tm;
  const CUtensorMapDataType dt =
      a.in_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (make_operand_maps(tm, dt, 2, A, a.M, B, a.N, a.K, bn)) return 4;
  const int grid = persistent_grid(tile_count(a, Sched::Dense, bn));
  if (bn == 256) return launch_instance<Kind::F16, Sched::Dense, 256, 4>(a, tm, grid, stream);
  return launch_instance<Kind::F16, Sched::Dense, 128, 6>(a, tm, grid, stream);
}

}  // namespace fgf8

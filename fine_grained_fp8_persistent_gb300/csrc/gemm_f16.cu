// gemm_f16.cu -- launcher of the dense 16-bit (fp16/bf16) NT GEMM.
#include "gemm_launch.cuh"

namespace fgf8 {

int launch_gemm_f16(const GemmArgs& a, const void* A, const void* B, cudaStream_t stream) {
  // relative tile times: see pick_cfg (the 1 x 128 tile is extrapolated)
  static const TileCfg cands[] = {{2, 256, 40.3}, {2, 224, 36.6}, {1, 128, 25.0}};
  const TileCfg c = cands[pick_cfg(a, Sched::Dense, cands, kCount(cands))];
  TensorMaps tm;
  const CUtensorMapDataType dt =
      a.in_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (make_operand_maps(tm, dt, 2, A, a.M, B, a.N, a.K, c.bn / c.ncta)) return 4;
  const long long tiles = tile_count(a, Sched::Dense, c);
  if (c.ncta == 2 && c.bn == 224) return launch_persistent<Kind::F16, Sched::Dense, 2, 224, 6>(a, tm, tiles, stream);
  if (c.ncta == 2) return launch_persistent<Kind::F16, Sched::Dense, 2, 256, 6>(a, tm, tiles, stream);
  return launch_persistent<Kind::F16, Sched::Dense, 1, 128, 6>(a, tm, tiles, stream);
}

}  // namespace fgf8

// gemm_fp4.cu -- launcher of the dense 4-bit block-scaled NT GEMM (MXFP4: E2M1 +
// E8M0 per 32 elements; NVFP4: E2M1 + E4M3 per 16) on kind::mxf4nvf4.
//
// "GPU GEMM part 4: tcgen05 & Blackwell", section 6: the scale tables are MMA
// operands read from TMEM; section 3.5: a 4-bit MMA takes K = 64 per
// instruction, so a 128-byte K block of each row holds 256 elements and four
// instructions.  Operands are the packed bytes quantize_fp4 writes (two elements
// per byte along K), loaded by TMA exactly like the 8-bit operands.
#include "gemm_launch.cuh"

namespace fgf8 {
namespace {

template <Kind KIND>
int launch_fp4_cfg(const TileCfg& c, const GemmArgs& a, const TensorMaps& tm, long long tiles, cudaStream_t stream) {
  // one 256-wide accumulator drained by 8 epilogue warps; 4 stages leave room for
  // the scale-word rings
  if (c.ncta == 2 && c.bn == 256) return launch_persistent<KIND, Sched::Dense, 2, 256, 4, 1>(a, tm, tiles, stream);
  if (c.ncta == 2) return launch_persistent<KIND, Sched::Dense, 2, 128, 8>(a, tm, tiles, stream);
  return launch_persistent<KIND, Sched::Dense, 1, 128, 6>(a, tm, tiles, stream);
}

}  // namespace

int launch_gemm_fp4(const GemmArgs& a, const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                    int fmt, cudaStream_t stream) {
  // relative tile times (see pick_cfg): the 8-bit block-scaled tiles' ratios
  static const TileCfg cands[] = {{2, 256, 24.2}, {2, 128, 14.4}, {1, 128, 14.9}};
  const TileCfg c = cands[pick_cfg(a, Sched::Dense, cands, kCount(cands))];
  TensorMaps tm;
  // packed operands: K / 2 bytes per row, a K block is 128 bytes (256 elements)
  if (make_operand_maps(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, Aq, a.M, Bq, a.N, a.K / 2, c.bn / c.ncta))
    return 4;
  // scale words: int32 [K / SV / 4][align4(rows)]; one pipeline unit (two K
  // blocks) takes 4 (MXFP4) or 8 (NVFP4) words of every row
  const int sv = fmt == 0 ? 32 : 16;
  const long long kq = (a.K / sv + 3) / 4;
  const uint32_t wg = static_cast<uint32_t>(2 * (256 / sv) / 4);
  const long long lda = (a.M + 3) / 4 * 4;
  const long long ldn = (a.N + 3) / 4 * 4;
  if (!encode_tmap_2d(&tm.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFA, lda, kq, lda * 4, 128, wg, false)) return 4;
  if (!encode_tmap_2d(&tm.sfb, CU_TENSOR_MAP_DATA_TYPE_UINT32, SFB, ldn, kq, ldn * 4, c.bn, wg, false)) return 4;
  const long long tiles = tile_count(a, Sched::Dense, c);
  return fmt == 0 ? launch_fp4_cfg<Kind::MXF4>(c, a, tm, tiles, stream)
                  : launch_fp4_cfg<Kind::NVF4>(c, a, tm, tiles, stream);
}

}  // namespace fgf8

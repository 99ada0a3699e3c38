// fgf8_internal.h -- declarations shared by the library's translation units (not
// part of the public ABI; the public header is include/fgf8.h).
#pragma once
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

// Bits of the per-device status word written by kernels.
#define FGF8_DEVERR_TIMEOUT 0x1u      // a bounded barrier wait ran out
#define FGF8_DEVERR_INPUT 0x2u        // device-side input out of contract (m_indices / masked_m)
#define FGF8_DEVERR_ROLE_PRODUCER 0x100u
#define FGF8_DEVERR_ROLE_MMA 0x200u
#define FGF8_DEVERR_ROLE_EPILOGUE 0x400u
#define FGF8_DEVERR_ROLE_SELFTEST 0x800u

#ifndef __CUDACC_RTC__
namespace fgf8 {

enum class Kind : int { F16 = 0, MXF8 = 1, F8F32 = 2, MXF4 = 3, NVF4 = 4 };
enum class Sched : int { Dense = 0, Contiguous = 1, Masked = 2 };

// Everything a GEMM launch needs besides the tensor maps.
struct GemmArgs {
  int M;              // rows of A (dense/contiguous) or Mmax (masked)
  int N;              // columns of D (per expert)
  int K;              // reduction length
  int G;              // experts (1 for dense)
  const int32_t* m_indices;   // contiguous: expert of each row, -1 = padding
  const int32_t* masked_m;    // masked: valid rows per expert (device memory)
  void* D;                    // output, row-major, leading dimension N
  int in_bf16;                // 16-bit GEMM operands: 1 bf16, 0 fp16
  int out_bf16;               // 1: bf16 output, 0: fp16 output
  const float* sfa_f32;       // FP32-scale path: activation scales
  const float* sfb_f32;       // FP32-scale path: weight block scales
  const uint32_t* sfa_ue8m0;  // UE8M0 path: packed activation scale words
  const uint32_t* sfb_ue8m0;  // UE8M0 path: packed weight scale words
  uint32_t* status;           // device status word
  uint64_t timeout_ns;        // bound on every barrier wait
  // Fused output quantization (dense block-scaled GEMM on 128-wide tiles): when
  // dq is set, D is not written; its bf16-rounded rows are quantized in 1x128
  // groups to E4M3 codes dq [M][N] and scales sfd (the quantize_1x128 layout).
  uint8_t* dq;
  void* sfd;
  int dq_ue8m0;               // 1: UE8M0 scales, 0: FP32 scales
  // Thin tiles (at most 64 rows): rows of the A box, a multiple of 8 that covers M
  // (the A tensor has only M rows; the stage rows past the box are never stored).
  // 0 = the tile's full 64.
  int a_box_rows;
  // Tile scheduling: 0 = static round robin over a persistent grid; 1 = cluster
  // launch control (a grid of one cluster per tile; running clusters cancel the
  // clusters not yet launched and take their tiles)
  int clc;
};

struct TensorMaps {
  CUtensorMap a, b, sfa, sfb;
};

// Host helpers (host.cu).
int set_error(int code, const char* fmt, ...);
// Whether kernels are launched with programmatic stream serialization (PDL).
bool pdl_enabled();
// Tile scheduler of the GEMMs (0 static, 1 cluster launch control) and whether
// the persistent grid is capped by the wave-preserving SM count.
int scheduler_mode();
bool sm_cap_enabled();
// Clusters of a static persistent grid for `tiles` cluster tiles: at most
// max_clusters; with the cap, the fewest that keep the number of waves, but not
// fewer than (sms - 8) SMs' worth, rounded to whole clusters.
long long persistent_clusters(long long tiles, int cluster, int sms, int max_clusters, bool cap);
// Launches the bounded-wait self-test (selftest.cu).
int launch_wait_selftest(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream);
// Records the configuration of the GEMM launch this thread makes (fgf8_last_tile).
void set_last_tile(const char* kind, const char* sched, int ctas, int bn, const char* suffix = "");
int device_sm_count();
int device_max_smem_optin();
uint32_t* device_status_ptr();
uint64_t wait_timeout_ns();
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                    uint32_t box_outer, bool swizzle128);

// Launchers (one translation unit each).
int launch_gemm_f16(const GemmArgs& a, const void* A, const void* B, cudaStream_t stream);
int launch_gemm_mxf8(const GemmArgs& a, Sched sched, const void* Aq, const void* SFA,
                     const void* Bq, const void* SFB, cudaStream_t stream);
int launch_gemm_f8f32(const GemmArgs& a, Sched sched, const void* Aq, const void* Bq,
                      cudaStream_t stream);
int launch_gemm_fp4(const GemmArgs& a, const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                    int fmt, cudaStream_t stream);
int launch_quantize_1x128(const void* X, void* Xq, void* SF, int M, int K, int fmt,
                          cudaStream_t stream);
int launch_quantize_128x128(const void* W, void* Wq, void* SF, int G, int N, int K, int fmt,
                            cudaStream_t stream);
int launch_quantize_fp4(const void* X, void* Xq, void* SF, int R, int K, int fmt, cudaStream_t stream);

}  // namespace fgf8
#endif

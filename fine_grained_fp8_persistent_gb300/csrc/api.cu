// api.cu -- the C ABI (include/fgf8.h): host-side validation, the per-device status
// word, tensor-map encoding and dispatch to the kernel launchers.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/fgf8.h"
#include "fgf8_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kBlockM = 128;     // rows per tile; the contiguous-layout alignment
constexpr int kMaxGroups = 1024; // masked scheduler keeps a per-expert prefix in SMEM

// Status word written by kernels (one per device that loads the library).
__device__ uint32_t g_status;

thread_local char g_errbuf[512];
int g_pdl = -1;   // -1 = not read from the environment yet
int g_sched = -1;  // tile scheduler; -1 = not read from the environment yet
int g_smcap = -1;  // wave-preserving SM cap of persistent grids; -1 = not read yet
thread_local char g_last_tile[64];

struct DevInfo {
  bool ready = false;
  int sms = 0;
  int smem_optin = 0;
  uint32_t* status = nullptr;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;

uint64_t g_timeout_ns = 0;   // 0 = not read from the environment yet
std::once_flag g_timeout_once;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int current_device(int* dev) {
  const cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fgf8::set_error(FGF8_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (*dev < 0 || *dev >= kMaxDevices) return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "device id %d", *dev);
  return FGF8_OK;
}

const DevInfo* dev_info() {
  int dev = 0;
  if (current_device(&dev) != FGF8_OK) return nullptr;
  DevInfo& d = g_dev[dev];
  if (d.ready) return &d;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (d.ready) return &d;
  cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  void* p = nullptr;
  if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, g_status);
  if (e != cudaSuccess) {
    fgf8::set_error(FGF8_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    return nullptr;
  }
  d.status = static_cast<uint32_t*>(p);
  d.ready = true;
  return &d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every tensor pointer must be device (or managed) memory of the current device:
// a pointer into another GPU's memory would put a peer's memory under the tensor
// maps, and a host pointer cannot be read by TMA.  Checked before any tensor map
// is encoded or any kernel launched.
int check_on_device(const char* who, std::initializer_list<const void*> ptrs) {
  int dev = 0;
  if (int r = current_device(&dev)) return r;
  int i = 0;
  for (const void* p : ptrs) {
    cudaPointerAttributes at;
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
      cudaGetLastError();  // the failed query also sets the runtime's last error; clear it
      return fgf8::set_error(FGF8_ERR_INVALID_ARG, "%s: pointer %d: %s", who, i, cudaGetErrorString(e));
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
      return fgf8::set_error(FGF8_ERR_INVALID_ARG, "%s: pointer %d is not device memory", who, i);
    if (at.type == cudaMemoryTypeDevice && at.device != dev)
      return fgf8::set_error(FGF8_ERR_INVALID_ARG, "%s: pointer %d is on device %d, the current device is %d",
                             who, i, at.device, dev);
    ++i;
  }
  return FGF8_OK;
}
long long align4(long long x) { return (x + 3) / 4 * 4; }

}  // namespace

namespace fgf8 {

void set_last_tile(const char* kind, const char* sched, int ctas, int bn, const char* suffix) {
  std::snprintf(g_last_tile, sizeof(g_last_tile), "%s %s %dx%d%s", kind, sched, ctas, bn, suffix);
}

bool pdl_enabled() {
  if (g_pdl < 0) {
    const char* e = std::getenv("FGF8_PDL");
    g_pdl = (e != nullptr && e[0] == '0') ? 0 : 1;
  }
  return g_pdl != 0;
}

int scheduler_mode() {
  if (g_sched < 0) {
    const char* e = std::getenv("FGF8_SCHED");
    g_sched = (e != nullptr && std::strcmp(e, "clc") == 0) ? 1 : 0;
  }
  return g_sched;
}

bool sm_cap_enabled() {
  if (g_smcap < 0) {
    const char* e = std::getenv("FGF8_SM_CAP");
    g_smcap = (e != nullptr && e[0] == '0') ? 0 : 1;
  }
  return g_smcap != 0;
}

// "DeepGEMM dissected", section on the SM count (num_min_sms): the fewest SMs that
// keep the number of waves, but never fewer than all SMs but 8, in whole clusters.
long long persistent_clusters(long long tiles, int cluster, int sms, int max_clusters, bool cap) {
  if (tiles < 1 || cluster < 1 || max_clusters < 1) return 1;
  long long clusters = tiles < max_clusters ? tiles : max_clusters;
  if (!cap) return clusters;
  const long long waves = (tiles + clusters - 1) / clusters;
  const long long wave_sms = (tiles + waves - 1) / waves * cluster;
  const long long floor_sms = sms - 8;
  const long long want_sms = wave_sms > floor_sms ? wave_sms : floor_sms;
  long long c = (want_sms + cluster - 1) / cluster;
  if (c > clusters) c = clusters;
  return c < 1 ? 1 : c;
}

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_errbuf, sizeof(g_errbuf), fmt, ap);
  va_end(ap);
  return code;
}

int device_sm_count() {
  const DevInfo* d = dev_info();
  return d ? d->sms : 1;
}

int device_max_smem_optin() {
  const DevInfo* d = dev_info();
  return d ? d->smem_optin : 0;
}

uint32_t* device_status_ptr() {
  const DevInfo* d = dev_info();
  return d ? d->status : nullptr;
}

uint64_t wait_timeout_ns() {
  std::call_once(g_timeout_once, [] {
    long ms = 2000;
    if (const char* s = std::getenv("FGF8_WAIT_TIMEOUT_MS")) {
      const long v = std::strtol(s, nullptr, 10);
      if (v > 0) ms = v;
    }
    if (g_timeout_ns == 0) g_timeout_ns = static_cast<uint64_t>(ms) * 1000000ull;
  });
  return g_timeout_ns;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                    uint32_t box_outer, bool swizzle128) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) {
    set_error(FGF8_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
    return false;
  }
  std::memset(map, 0, sizeof(*map));
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error(FGF8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d): dims %llu x %llu, box %u x %u",
              static_cast<int>(r), static_cast<unsigned long long>(inner),
              static_cast<unsigned long long>(outer), box_inner, box_outer);
    return false;
  }
  return true;
}

}  // namespace fgf8

// ============================================================================ C ABI
extern "C" {

const char* fgf8_last_error(void) { return g_errbuf; }

const char* fgf8_last_tile(void) { return g_last_tile; }

int fgf8_version(void) { return 100; }

int fgf8_mk_alignment_for_contiguous(void) { return kBlockM; }

int fgf8_selftest_wait_timeout(void* stream) {
  int dev = 0;
  if (int r = current_device(&dev)) return r;
  uint32_t* status = fgf8::device_status_ptr();
  if (status == nullptr) return FGF8_ERR_CUDA;
  return fgf8::launch_wait_selftest(status, fgf8::wait_timeout_ns(), static_cast<cudaStream_t>(stream));
}

int fgf8_set_pdl(int enable) {
  const int prev = fgf8::pdl_enabled() ? 1 : 0;
  if (enable == 0 || enable == 1) g_pdl = enable;
  return prev;
}

int fgf8_set_scheduler(int mode) {
  const int prev = fgf8::scheduler_mode();
  if (mode == 0 || mode == 1) g_sched = mode;
  return prev;
}

int fgf8_set_sm_cap(int enable) {
  const int prev = fgf8::sm_cap_enabled() ? 1 : 0;
  if (enable == 0 || enable == 1) g_smcap = enable;
  return prev;
}

long long fgf8_persistent_clusters(long long tiles, int cluster, int sms, int max_clusters, int cap) {
  return fgf8::persistent_clusters(tiles, cluster, sms, max_clusters, cap != 0);
}

int fgf8_set_wait_timeout_ms(int ms) {
  const int prev = static_cast<int>(fgf8::wait_timeout_ns() / 1000000ull);
  if (ms > 0) g_timeout_ns = static_cast<uint64_t>(ms) * 1000000ull;
  return prev;
}

long long fgf8_sfa_bytes(int rows, int K, int fmt) {
  if (rows < 0 || K <= 0 || K % 128 != 0) return -1;
  const long long nkb = K / 128;
  if (fmt == FGF8_SCALE_F32) return nkb * align4(rows) * 4;
  if (fmt == FGF8_SCALE_UE8M0) return (nkb + 3) / 4 * align4(rows) * 4;
  return -1;
}

long long fgf8_sfb_bytes(int G, int N, int K, int fmt) {
  if (G <= 0 || N <= 0 || K <= 0 || K % 128 != 0) return -1;
  const long long nkb = K / 128;
  if (fmt == FGF8_SCALE_F32) return static_cast<long long>(G) * ((N + 127) / 128) * nkb * 4;
  if (fmt == FGF8_SCALE_UE8M0) return static_cast<long long>(G) * ((nkb + 3) / 4) * align4(N) * 4;
  return -1;
}

int fgf8_check_status(void* stream, unsigned int* raw_bits) {
  if (raw_bits) *raw_bits = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fgf8::set_error(FGF8_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  if (!dev_info()) return FGF8_ERR_CUDA;
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
  if (e == cudaSuccess && v != 0) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
  }
  if (e != cudaSuccess)
    return fgf8::set_error(FGF8_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
  if (raw_bits) *raw_bits = v;
  if (v & FGF8_DEVERR_TIMEOUT)
    return fgf8::set_error(FGF8_ERR_DEVICE_TIMEOUT, "a kernel pipeline wait timed out (bits 0x%x)", v);
  if (v & FGF8_DEVERR_INPUT)
    return fgf8::set_error(FGF8_ERR_DEVICE_INPUT, "device-side input out of contract (bits 0x%x)", v);
  return FGF8_OK;
}

int quantize_1x128(const void* X, void* Xq, void* SFA, int M, int K, int fmt, void* stream) {
  if (M < 0 || K <= 0) return fgf8::set_error(FGF8_ERR_INVALID_ARG, "quantize_1x128: M=%d K=%d", M, K);
  if (K % 128 != 0) return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "quantize_1x128: K=%d not a multiple of 128", K);
  if (fmt != FGF8_SCALE_F32 && fmt != FGF8_SCALE_UE8M0)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "quantize_1x128: bad scale format %d", fmt);
  if (M == 0) return FGF8_OK;
  if (!X || !Xq || !SFA) return fgf8::set_error(FGF8_ERR_INVALID_ARG, "quantize_1x128: null pointer");
  if (!aligned16(X) || !aligned16(Xq) || !aligned16(SFA))
    return fgf8::set_error(FGF8_ERR_MISALIGNED, "quantize_1x128: pointers must be 16-byte aligned");
  if (int r = check_on_device("quantize_1x128", {X, Xq, SFA})) return r;
  return fgf8::launch_quantize_1x128(X, Xq, SFA, M, K, fmt, static_cast<cudaStream_t>(stream));
}

int quantize_128x128(const void* W, void* Wq, void* SFB, int G, int N, int K, int fmt, void* stream) {
  if (G <= 0 || N <= 0 || K <= 0)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "quantize_128x128: G=%d N=%d K=%d", G, N, K);
  if (K % 128 != 0) return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "quantize_128x128: K=%d not a multiple of 128", K);
  if (fmt != FGF8_SCALE_F32 && fmt != FGF8_SCALE_UE8M0)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "quantize_128x128: bad scale format %d", fmt);
  if (!W || !Wq || !SFB) return fgf8::set_error(FGF8_ERR_INVALID_ARG, "quantize_128x128: null pointer");
  if (!aligned16(W) || !aligned16(Wq) || !aligned16(SFB))
    return fgf8::set_error(FGF8_ERR_MISALIGNED, "quantize_128x128: pointers must be 16-byte aligned");
  if (int r = check_on_device("quantize_128x128", {W, Wq, SFB})) return r;
  return fgf8::launch_quantize_128x128(W, Wq, SFB, G, N, K, fmt, static_cast<cudaStream_t>(stream));
}

long long fgf8_fp4_sf_bytes(int R, int K, int fmt) {
  if (R < 0 || K <= 0 || K % 64 != 0 || (fmt != FGF8_FP4_MX && fmt != FGF8_FP4_NV)) return -1;
  const long long groups = K / (fmt == FGF8_FP4_MX ? 32 : 16);
  return (groups + 3) / 4 * align4(R) * 4;
}

int quantize_fp4(const void* X, void* Xq, void* SF, int R, int K, int fmt, void* stream) {
  if (R < 0 || K <= 0) return fgf8::set_error(FGF8_ERR_INVALID_ARG, "quantize_fp4: R=%d K=%d", R, K);
  if (K % 64 != 0) return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "quantize_fp4: K=%d not a multiple of 64", K);
  if (fmt != FGF8_FP4_MX && fmt != FGF8_FP4_NV)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "quantize_fp4: bad format %d", fmt);
  if (R == 0) return FGF8_OK;
  if (!X || !Xq || !SF) return fgf8::set_error(FGF8_ERR_INVALID_ARG, "quantize_fp4: null pointer");
  if (!aligned16(X) || !aligned16(Xq) || !aligned16(SF))
    return fgf8::set_error(FGF8_ERR_MISALIGNED, "quantize_fp4: pointers must be 16-byte aligned");
  if (int r = check_on_device("quantize_fp4", {X, Xq, SF})) return r;
  return fgf8::launch_quantize_fp4(X, Xq, SF, R, K, fmt, static_cast<cudaStream_t>(stream));
}

static int prepare_args(fgf8::GemmArgs& a, int M, int N, int K, int G, void* D) {
  std::memset(&a, 0, sizeof(a));
  a.M = M;
  a.N = N;
  a.K = K;
  a.G = G;
  a.D = D;
  a.out_bf16 = 1;
  a.status = fgf8::device_status_ptr();
  if (!a.status) return FGF8_ERR_CUDA;
  a.timeout_ns = fgf8::wait_timeout_ns();
  return FGF8_OK;
}

int gemm_f16(const void* A, const void* B, void* D, int M, int N, int K, int in_dtype,
             int out_dtype, void* stream) {
  if (M < 0 || N <= 0 || K <= 0)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_f16: M=%d N=%d K=%d", M, N, K);
  if ((in_dtype != FGF8_F16 && in_dtype != FGF8_BF16) || (out_dtype != FGF8_F16 && out_dtype != FGF8_BF16))
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_f16: bad dtype");
  if (K % 8 != 0 || N % 8 != 0)
    return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "gemm_f16: K=%d and N=%d must be multiples of 8", K, N);
  if (M == 0) return FGF8_OK;
  if (!A || !B || !D) return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_f16: null pointer");
  if (!aligned16(A) || !aligned16(B) || !aligned16(D))
    return fgf8::set_error(FGF8_ERR_MISALIGNED, "gemm_f16: pointers must be 16-byte aligned");
  if (int r = check_on_device("gemm_f16", {A, B, D})) return r;
  fgf8::GemmArgs a;
  if (prepare_args(a, M, N, K, 1, D) != FGF8_OK) return FGF8_ERR_CUDA;
  a.in_bf16 = in_dtype == FGF8_BF16;
  a.out_bf16 = out_dtype == FGF8_BF16;
  return fgf8::launch_gemm_f16(a, A, B, static_cast<cudaStream_t>(stream));
}

static int check_fp8_common(const char* who, int N, int K, int fmt) {
  if (N <= 0 || K <= 0) return fgf8::set_error(FGF8_ERR_INVALID_ARG, "%s: N=%d K=%d", who, N, K);
  if (K % 128 != 0) return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "%s: K=%d not a multiple of 128", who, K);
  if (N % 8 != 0) return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "%s: N=%d not a multiple of 8", who, N);
  if (fmt != FGF8_SCALE_F32 && fmt != FGF8_SCALE_UE8M0)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "%s: bad scale format %d", who, fmt);
  return FGF8_OK;
}

static int dispatch_fp8(fgf8::GemmArgs& a, fgf8::Sched sched, const void* Aq, const void* SFA,
                        const void* Bq, const void* SFB, int fmt, void* stream) {
  if (fmt == FGF8_SCALE_UE8M0) {
    a.sfa_ue8m0 = static_cast<const uint32_t*>(SFA);
    a.sfb_ue8m0 = static_cast<const uint32_t*>(SFB);
    return fgf8::launch_gemm_mxf8(a, sched, Aq, SFA, Bq, SFB, static_cast<cudaStream_t>(stream));
  }
  a.sfa_f32 = static_cast<const float*>(SFA);
  a.sfb_f32 = static_cast<const float*>(SFB);
  return fgf8::launch_gemm_f8f32(a, sched, Aq, Bq, static_cast<cudaStream_t>(stream));
}

int gemm_fp8_blockscaled(const void* Aq, const void* SFA, const void* Bq, const void* SFB, void* D,
                         int M, int N, int K, int fmt, void* stream) {
  if (M < 0) return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_fp8_blockscaled: M=%d", M);
  if (int r = check_fp8_common("gemm_fp8_blockscaled", N, K, fmt)) return r;
  if (M == 0) return FGF8_OK;
  if (!Aq || !SFA || !Bq || !SFB || !D)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_fp8_blockscaled: null pointer");
  if (!aligned16(Aq) || !aligned16(SFA) || !aligned16(Bq) || !aligned16(SFB) || !aligned16(D))
    return fgf8::set_error(FGF8_ERR_MISALIGNED, "gemm_fp8_blockscaled: pointers must be 16-byte aligned");
  if (int r = check_on_device("gemm_fp8_blockscaled", {Aq, SFA, Bq, SFB, D})) return r;
  fgf8::GemmArgs a;
  if (prepare_args(a, M, N, K, 1, D) != FGF8_OK) return FGF8_ERR_CUDA;
  return dispatch_fp8(a, fgf8::Sched::Dense, Aq, SFA, Bq, SFB, fmt, stream);
}

int gemm_fp8_blockscaled_quant(const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                               void* Dq, void* SFD, int M, int N, int K, int fmt, int out_fmt,
                               void* stream) {
  if (M < 0) return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_fp8_blockscaled_quant: M=%d", M);
  if (int r = check_fp8_common("gemm_fp8_blockscaled_quant", N, K, fmt)) return r;
  if (out_fmt != FGF8_SCALE_F32 && out_fmt != FGF8_SCALE_UE8M0)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_fp8_blockscaled_quant: bad output scale format %d", out_fmt);
  if (N % 128 != 0)
    return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "gemm_fp8_blockscaled_quant: N=%d not a multiple of 128", N);
  if (M == 0) return FGF8_OK;
  if (!Aq || !SFA || !Bq || !SFB || !Dq || !SFD)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_fp8_blockscaled_quant: null pointer");
  if (!aligned16(Aq) || !aligned16(SFA) || !aligned16(Bq) || !aligned16(SFB) || !aligned16(Dq) || !aligned16(SFD))
    return fgf8::set_error(FGF8_ERR_MISALIGNED, "gemm_fp8_blockscaled_quant: pointers must be 16-byte aligned");
  if (int r = check_on_device("gemm_fp8_blockscaled_quant", {Aq, SFA, Bq, SFB, Dq, SFD})) return r;
  fgf8::GemmArgs a;
  if (prepare_args(a, M, N, K, 1, nullptr) != FGF8_OK) return FGF8_ERR_CUDA;
  a.dq = static_cast<uint8_t*>(Dq);
  a.sfd = SFD;
  a.dq_ue8m0 = out_fmt == FGF8_SCALE_UE8M0;
  return dispatch_fp8(a, fgf8::Sched::Dense, Aq, SFA, Bq, SFB, fmt, stream);
}

int gemm_fp4_blockscaled(const void* Aq, const void* SFA, const void* Bq, const void* SFB, void* D, int M,
                         int N, int K, int fmt, void* stream) {
  if (M < 0 || N <= 0 || K <= 0)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_fp4_blockscaled: M=%d N=%d K=%d", M, N, K);
  if (K % 256 != 0) return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "gemm_fp4_blockscaled: K=%d not a multiple of 256", K);
  if (N % 32 != 0) return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "gemm_fp4_blockscaled: N=%d not a multiple of 32", N);
  if (fmt != FGF8_FP4_MX && fmt != FGF8_FP4_NV)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_fp4_blockscaled: bad format %d", fmt);
  if (M == 0) return FGF8_OK;
  if (!Aq || !SFA || !Bq || !SFB || !D)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "gemm_fp4_blockscaled: null pointer");
  if (!aligned16(Aq) || !aligned16(SFA) || !aligned16(Bq) || !aligned16(SFB) || !aligned16(D))
    return fgf8::set_error(FGF8_ERR_MISALIGNED, "gemm_fp4_blockscaled: pointers must be 16-byte aligned");
  if (int r = check_on_device("gemm_fp4_blockscaled", {Aq, SFA, Bq, SFB, D})) return r;
  fgf8::GemmArgs a;
  if (prepare_args(a, M, N, K, 1, D) != FGF8_OK) return FGF8_ERR_CUDA;
  return fgf8::launch_gemm_fp4(a, Aq, SFA, Bq, SFB, fmt, static_cast<cudaStream_t>(stream));
}

int grouped_fp8_contiguous(const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                           const int32_t* m_indices, void* D, int M, int N, int K, int G, int fmt,
                           void* stream) {
  if (M < 0 || G <= 0)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "grouped_fp8_contiguous: M=%d G=%d", M, G);
  if (int r = check_fp8_common("grouped_fp8_contiguous", N, K, fmt)) return r;
  if (M % kBlockM != 0)
    return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "grouped_fp8_contiguous: M=%d not a multiple of %d",
                           M, kBlockM);
  if (static_cast<long long>(G) * N >= (1ll << 31))
    return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "grouped_fp8_contiguous: G*N too large");
  if (M == 0) return FGF8_OK;
  if (!Aq || !SFA || !Bq || !SFB || !D || !m_indices)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "grouped_fp8_contiguous: null pointer");
  if (!aligned16(Aq) || !aligned16(SFA) || !aligned16(Bq) || !aligned16(SFB) || !aligned16(D))
    return fgf8::set_error(FGF8_ERR_MISALIGNED, "grouped_fp8_contiguous: pointers must be 16-byte aligned");
  if (int r = check_on_device("grouped_fp8_contiguous", {Aq, SFA, Bq, SFB, D, m_indices})) return r;
  fgf8::GemmArgs a;
  if (prepare_args(a, M, N, K, G, D) != FGF8_OK) return FGF8_ERR_CUDA;
  a.m_indices = m_indices;
  return dispatch_fp8(a, fgf8::Sched::Contiguous, Aq, SFA, Bq, SFB, fmt, stream);
}

int grouped_fp8_masked(const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                       const int32_t* masked_m, void* D, int G, int Mmax, int N, int K,
                       int expected_m, int fmt, void* stream) {
  (void)expected_m;
  if (G <= 0 || Mmax < 0)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "grouped_fp8_masked: G=%d Mmax=%d", G, Mmax);
  if (int r = check_fp8_common("grouped_fp8_masked", N, K, fmt)) return r;
  if (G > kMaxGroups)
    return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "grouped_fp8_masked: G=%d above %d", G, kMaxGroups);
  if (static_cast<long long>(G) * Mmax >= (1ll << 31) || static_cast<long long>(G) * N >= (1ll << 31))
    return fgf8::set_error(FGF8_ERR_UNSUPPORTED, "grouped_fp8_masked: G*Mmax or G*N too large");
  if (Mmax == 0) return FGF8_OK;
  if (!Aq || !SFA || !Bq || !SFB || !D || !masked_m)
    return fgf8::set_error(FGF8_ERR_INVALID_ARG, "grouped_fp8_masked: null pointer");
  if (!aligned16(Aq) || !aligned16(SFA) || !aligned16(Bq) || !aligned16(SFB) || !aligned16(D))
    return fgf8::set_error(FGF8_ERR_MISALIGNED, "grouped_fp8_masked: pointers must be 16-byte aligned");
  if (int r = check_on_device("grouped_fp8_masked", {Aq, SFA, Bq, SFB, D, masked_m})) return r;
  fgf8::GemmArgs a;
  if (prepare_args(a, Mmax, N, K, G, D) != FGF8_OK) return FGF8_ERR_CUDA;
  a.masked_m = masked_m;
  return dispatch_fp8(a, fgf8::Sched::Masked, Aq, SFA, Bq, SFB, fmt, stream);
}

}  // extern "C"

/*
 * fgf8.h -- C ABI of the fine-grained FP8 persistent GEMM library for GB300
 * (sm_103a).  Library file: libfgf8.so.
 *
 * What it computes: the NT GEMM D = A * B^T (the linear layer Y = X W^T) with
 * FP32 accumulation, for 16-bit operands and for E4M3 operands carrying
 * DeepSeek-V3 fine-grained scales (1x128 per token for A, 128x128 per block for
 * B), plus the contiguous and masked grouped MoE forms, the quantizers that
 * produce the E4M3 operands, and a GEMM whose epilogue quantizes its own output
 * for the next layer.  Page references name the web page and section:
 *   [DG]   "DeepGEMM dissected: a 300-line FP8 GEMM kernel" (pinghaoyang.com.cn)
 *   [TC5]  "GPU GEMM part 4: tcgen05 & Blackwell" (pinghaoyang.com.cn)
 *   [TIRx] "TIRx and high-performance GEMM (part 2)" (Tencent Cloud developer)
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or keeps them.  Each must be 16-byte aligned and
 *     must be device (or managed) memory of the current device
 *     (cudaGetDevice); host memory or another GPU's memory is refused with
 *     FGF8_ERR_INVALID_ARG before anything is launched.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and returns as soon as the work is
 *     enqueued.
 *   - Arguments are validated on the host first.  An invalid call returns a
 *     non-zero fgf8_status and launches nothing; fgf8_last_error() then gives a
 *     message.  Validation needs no GPU.
 *   - Device-side problems (a device-side input out of contract, or a bounded
 *     pipeline wait that ran out) set bits in a per-device status word read by
 *     fgf8_check_status().  After such an error the output is undefined.
 *   - Row-major layouts; "NT": A is (M, K) with K contiguous, B is (N, K) with K
 *     contiguous ([DG] "why only the NT layout").
 *   - Empty problems (M == 0, or every masked row count 0) are valid no-ops.
 *
 * Scale-table layouts (fmt = FGF8_SCALE_F32 or FGF8_SCALE_UE8M0), with
 * nkb = K / 128 (K must be a multiple of 128, [DG] "thread organisation":
 * BLOCK_K is fixed at 128, the scale granularity):
 *   activation scales SFA for R rows (the 1x128 groups of [DG] "fine-grained
 *   quantization", stored TMA-aligned and transposed, [DG] "why only the NT
 *   layout"):
 *     F32   : float  [nkb][align4(R)]   entry (kb, r) = scale of row r, K block kb
 *     UE8M0 : int32  [ceil(nkb/4)][align4(R)]; byte (kb % 4) of word (kb / 4, r)
 *             is the biased exponent e + 127 of the power-of-two scale 2^e;
 *             bytes of K blocks >= nkb and rows >= R are 0.
 *   weight scales SFB for G experts of N rows (128x128 blocks):
 *     F32   : float  [G][ceil(N/128)][nkb]   one scale per 128x128 block
 *     UE8M0 : int32  [G][ceil(nkb/4)][align4(N)]; the block exponent is stored
 *             for every row n of its block (the MMA reads one scale per B row,
 *             [TC5] section 6 block-scaling formula with SFB(N, SFK)).
 *   align4(x) = ceil(x / 4) * 4.
 * F32 scales are s = amax / 448 (FP32); UE8M0 scales are 2^e with
 * e = ceil(log2(amax / 448)) clamped to [-127, 127]; an all-zero group has
 * scale 1.  E4M3 codes are round-to-nearest-even, saturating at +-448.
 */
#ifndef FGF8_H
#define FGF8_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FGF8_API __attribute__((visibility("default")))
#else
#define FGF8_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FGF8_OK = 0,
  FGF8_ERR_INVALID_ARG = 1,   /* null pointer, negative or inconsistent size */
  FGF8_ERR_UNSUPPORTED = 2,   /* shape or option outside what the kernels support */
  FGF8_ERR_MISALIGNED = 3,    /* pointer or leading dimension not 16-byte aligned */
  FGF8_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  FGF8_ERR_DEVICE_TIMEOUT = 5,/* fgf8_check_status: a kernel's bounded wait ran out */
  FGF8_ERR_DEVICE_INPUT = 6   /* fgf8_check_status: m_indices / masked_m out of contract */
} fgf8_status;

typedef enum { FGF8_F16 = 0, FGF8_BF16 = 1 } fgf8_dtype;
typedef enum { FGF8_SCALE_F32 = 0, FGF8_SCALE_UE8M0 = 1 } fgf8_scale_fmt;
/* 4-bit block-scaled formats ([TC5] section 6.3): E2M1 elements with an E8M0
 * scale per 32 elements along K (MXFP4) or an E4M3 scale per 16 (NVFP4). */
typedef enum { FGF8_FP4_MX = 0, FGF8_FP4_NV = 1 } fgf8_fp4_fmt;

/*
 * quantize_1x128 -- activation quantization, 1x128 groups ([DG] "fine-grained
 * quantization": one scale per token per 128 channels, computed online from the
 * group's max |x|).
 *   X   : bf16 [M][K]              input
 *   Xq  : uint8 [M][K]             E4M3 codes (output)
 *   SFA : activation scale table for M rows in format fmt (output; layout above)
 * Requires K % 128 == 0, M >= 0.
 */
FGF8_API int quantize_1x128(const void* X, void* Xq, void* SFA, int M, int K, int fmt, void* stream);

/*
 * quantize_128x128 -- weight quantization, 128x128 blocks per expert ([DG]
 * "fine-grained quantization": one scale per 128 input x 128 output channels).
 *   W   : bf16 [G][N][K]           input
 *   Wq  : uint8 [G][N][K]          E4M3 codes (output)
 *   SFB : weight scale table (output; layout above)
 * Requires K % 128 == 0, G >= 1, N >= 1.  A partial last block along N takes
 * its max over its valid rows.
 */
FGF8_API int quantize_128x128(const void* W, void* Wq, void* SFB, int G, int N, int K, int fmt,
                     void* stream);

/*
 * gemm_f16 -- dense 16-bit NT GEMM, D[M][N] = A[M][K] * B[N][K]^T, FP32
 * accumulation, 16-bit output rounded to nearest even ([TIRx] Step 7/8: the
 * persistent warp-specialised fp16 GEMM; [TC5] section 3: kind::f16 MMA).
 *   A, B : fp16 or bf16 (in_dtype), D : fp16 or bf16 (out_dtype)
 * Requires K % 8 == 0, N % 8 == 0, M >= 0, N, K >= 1.
 */
FGF8_API int gemm_f16(const void* A, const void* B, void* D, int M, int N, int K, int in_dtype,
             int out_dtype, void* stream);

/*
 * gemm_fp8_blockscaled -- dense E4M3 NT GEMM with fine-grained scales:
 *   D[m,n] = sum_kb SFA(m,kb) * SFB(n,kb) * sum_{k in kb} Aq[m,k] * Bq[n,k]
 * ([TC5] section 6 block-scaling formula with scale-vector length 128 along K;
 * [DG] main loop: per-128-K promotion).  FP32 scales run as FP32 partials per
 * K block promoted on the CUDA cores; UE8M0 scales run on the block-scaled MMA.
 *   Aq : uint8 [M][K], SFA : activation table (M rows), Bq : uint8 [N][K],
 *   SFB : weight table (G = 1), D : bf16 [M][N]
 * Requires K % 128 == 0, N % 8 == 0.
 */
FGF8_API int gemm_fp8_blockscaled(const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                         void* D, int M, int N, int K, int fmt, void* stream);

/*
 * gemm_fp8_blockscaled_quant -- gemm_fp8_blockscaled with the next layer's
 * activation quantization fused into its epilogue ([DG] "fine-grained
 * quantization": activation quantization belongs in the kernel that produces
 * the activations).  D is computed as gemm_fp8_blockscaled computes it and
 * rounded to bf16, but instead of D the kernel writes its 1x128 quantization:
 *   Dq  : uint8 [M][N]             E4M3 codes (output)
 *   SFD : scale table for M rows and N columns in format out_fmt (output; the
 *         layout quantize_1x128 writes for an M x N input, padding rows zero)
 * The outputs are bit-identical to quantize_1x128(gemm_fp8_blockscaled(...)).
 * Requires everything gemm_fp8_blockscaled requires, and N % 128 == 0 (other
 * N return FGF8_ERR_UNSUPPORTED with nothing launched).  Either input scale
 * format: UE8M0 runs on the block-scaled MMA, FP32 on the promoted partials.
 */
FGF8_API int gemm_fp8_blockscaled_quant(const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                               void* Dq, void* SFD, int M, int N, int K, int fmt, int out_fmt,
                               void* stream);

/*
 * grouped_fp8_contiguous -- MoE grouped GEMM, contiguous layout ([DG] "two
 * grouped layouts": the tokens of one expert are concatenated along M; N and K
 * are shared by all experts; every expert segment is padded to a multiple of
 * fgf8_mk_alignment_for_contiguous() rows).
 *   Aq : uint8 [M][K] (all segments), SFA : activation table for M rows
 *   Bq : uint8 [G][N][K], SFB : weight table for G experts
 *   m_indices : int32 [M] on the device: expert of each row, -1 = padding row
 *   D : bf16 [M][N]; padding rows are not written.
 * Each aligned block of rows must hold one expert's rows followed by padding;
 * a row naming another expert sets FGF8_ERR_DEVICE_INPUT and is not written.
 * Requires K % 128 == 0, N % 8 == 0, M % alignment == 0, G >= 1.
 */
FGF8_API int grouped_fp8_contiguous(const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                           const int32_t* m_indices, void* D, int M, int N, int K, int G, int fmt,
                           void* stream);

/*
 * grouped_fp8_masked -- MoE grouped GEMM, masked layout ([DG] "two grouped
 * layouts": each expert owns a fixed slot of Mmax rows and a mask says how many
 * are valid; only valid rows are computed, so the call needs no host knowledge
 * of the counts and can be captured in a CUDA graph).
 *   Aq : uint8 [G][Mmax][K], SFA : per expert an activation table for Mmax rows
 *        (G tables back to back)
 *   Bq : uint8 [G][N][K], SFB : weight table for G experts
 *   masked_m : int32 [G] on the device, valid rows per expert (0..Mmax)
 *   D : bf16 [G][Mmax][N]; rows >= masked_m[g] are not written.
 *   expected_m : a hint of the typical masked_m (may be 0); unused at present.
 * Requires K % 128 == 0, N % 8 == 0, 1 <= G <= 1024.
 */
FGF8_API int grouped_fp8_masked(const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                       const int32_t* masked_m, void* D, int G, int Mmax, int N, int K,
                       int expected_m, int fmt, void* stream);

/*
 * quantize_fp4 -- 4-bit block quantization of the rows of X along K, for either
 * GEMM operand ([TC5] section 6.1: every SV consecutive K elements of a row
 * share one scale; section 6.3: SV = 32 with an E8M0 scale for MXFP4, SV = 16
 * with an E4M3 scale for NVFP4; section 7.1: two elements per byte along K).
 *   X  : bf16 [R][K]               input
 *   Xq : uint8 [R][K/2]            E2M1 codes, element 2j in the low nibble of
 *                                  byte j, element 2j+1 in the high nibble (output)
 *   SF : int32 [ceil(K/SV/4)][align4(R)] (output): byte j of word (w, r) is the
 *        scale of group 4w+j of row r; unused bytes and rows R..align4(R)-1 are 0.
 * MXFP4 scale 2^e, e = ceil(log2(amax/6)) (FP32 quotient) clamped to
 * [-127, 127], stored as e + 127, codes E2M1(x * 2^-e).  NVFP4 scale
 * s = E4M3(amax/6) (nearest even, saturating), codes E2M1(x / s) (FP32
 * division; all codes 0 when s is 0).  An all-zero group has scale 1.  E2M1
 * rounds to nearest even and saturates at +-6.
 * Requires K % 64 == 0, R >= 0; fmt is an fgf8_fp4_fmt.
 */
FGF8_API int quantize_fp4(const void* X, void* Xq, void* SF, int R, int K, int fmt, void* stream);

/*
 * gemm_fp4_blockscaled -- dense 4-bit block-scaled NT GEMM ([TC5] section 6.1):
 *   D[m,n] = sum_k (A[m,k] * SFA[m, k/SV]) * (B[n,k] * SFB[n, k/SV])
 * on the block-scaled tensor-core MMA (kind::mxf4nvf4, scale_vec 2X for MXFP4,
 * 4X for NVFP4), FP32 accumulation, bf16 output.
 *   Aq : uint8 [M][K/2], SFA : scale table of M rows (quantize_fp4 layouts)
 *   Bq : uint8 [N][K/2], SFB : scale table of N rows
 *   D  : bf16 [M][N]
 * Requires K % 256 == 0, N % 32 == 0, M >= 0.
 */
FGF8_API int gemm_fp4_blockscaled(const void* Aq, const void* SFA, const void* Bq, const void* SFB,
                                  void* D, int M, int N, int K, int fmt, void* stream);

/* Bytes of a quantize_fp4 scale table for R rows; -1 on invalid arguments. */
FGF8_API long long fgf8_fp4_sf_bytes(int R, int K, int fmt);

/* Row alignment of expert segments in the contiguous layout (the BLOCK_M of the
 * kernel; [DG] mentions a query of this name for the contiguous layout). */
FGF8_API int fgf8_mk_alignment_for_contiguous(void);

/* Bytes of an activation scale table for `rows` rows, or of a weight scale
 * table for G experts of N rows.  Return -1 on invalid arguments. */
FGF8_API long long fgf8_sfa_bytes(int rows, int K, int fmt);
FGF8_API long long fgf8_sfb_bytes(int G, int N, int K, int fmt);

/*
 * fgf8_check_status -- synchronises `stream`, then reads and clears the status
 * word of the current device.  Returns FGF8_OK, FGF8_ERR_DEVICE_TIMEOUT,
 * FGF8_ERR_DEVICE_INPUT or FGF8_ERR_CUDA.  *raw_bits (if not NULL) receives the
 * raw word (bit 0 timeout, bit 1 input; bits 8-11 the role that timed out:
 * 0x100 producer, 0x200 MMA issue / relay, 0x400 epilogue or promotion, 0x800
 * the wait self-test).
 */
FGF8_API int fgf8_check_status(void* stream, unsigned int* raw_bits);

/* Message for the last non-OK return on this thread ("" if none). */
FGF8_API const char* fgf8_last_error(void);

/* Kernel configuration of the last GEMM this thread launched, as text
 * ("<kind> <schedule> <CTAs per cluster>x<tile width>", e.g. "mxf8 dense 2x224");
 * "" before the first launch.  The pointer stays valid until this thread's next
 * GEMM call. */
FGF8_API const char* fgf8_last_tile(void);

/*
 * fgf8_selftest_wait_timeout -- diagnostic of the device-side failure path (no
 * counterpart on the pages).  Launches one warp that waits, through the same
 * bounded wait routine every GEMM role uses, on a barrier that nothing ever
 * signals.  After the current wait limit (fgf8_set_wait_timeout_ms) the wait
 * gives up and the kernel returns; the next fgf8_check_status() then reports
 * FGF8_ERR_DEVICE_TIMEOUT with raw bits 0x801.  Nothing else is touched and the
 * CUDA context stays usable.  Returns FGF8_OK once the kernel is enqueued.
 */
FGF8_API int fgf8_selftest_wait_timeout(void* stream);

/* Programmatic dependent launch (on by default; the environment variable
 * FGF8_PDL=0 turns it off at first use).  When on, every kernel is launched with
 * programmatic stream serialization: its set-up (barriers, TMEM, descriptor
 * prefetch) overlaps the end of the previous kernel on the stream, and it reads no
 * global data before that kernel has completed.  enable: 1 on, 0 off, anything
 * else leaves it unchanged.  Returns the previous setting. */
FGF8_API int fgf8_set_pdl(int enable);

/* Tile scheduler of the GEMM kernels ("Dissecting NVIDIA Blackwell" (EEPW), the
 * feature list: cluster launch control).  0 (default; FGF8_SCHED unset): a
 * persistent grid of at most one CTA (or CTA pair) per SM walks the tiles in a
 * static round robin.  1 (FGF8_SCHED=clc at first use): the grid holds one
 * cluster per tile; each running cluster, as it drains its tiles, cancels clusters
 * that have not launched yet (clusterlaunchcontrol.try_cancel) and takes their
 * tiles, so the work is handed out dynamically.  Results are identical either way
 * up to the order of tiles.  mode: 0 or 1, anything else leaves it unchanged.
 * Returns the previous mode. */
FGF8_API int fgf8_set_scheduler(int mode);

/* Wave-preserving SM cap of the static persistent grid of dense GEMMs
 * ("DeepGEMM dissected", section on the number of SMs launched: num_min_sms =
 * ceil(max(SMs the waves need, SMs - 8) / cluster) * cluster, leaving SMs idle
 * where that keeps the wave count, for less L2 pressure and power).  On by default
 * (FGF8_SM_CAP=0 turns it off at first use); grouped layouts, whose tile count the
 * host only bounds, always use the full grid.  enable: 1 on, 0 off, anything else
 * leaves it unchanged.  Returns the previous setting. */
FGF8_API int fgf8_set_sm_cap(int enable);

/* The cluster count of a static persistent grid for `tiles` cluster tiles of
 * `cluster` CTAs on `sms` SMs where at most `max_clusters` clusters fit, with the
 * SM cap on (cap = 1) or off.  Pure host arithmetic (no device needed); it is the
 * rule every GEMM launch applies. */
FGF8_API long long fgf8_persistent_clusters(long long tiles, int cluster, int sms, int max_clusters, int cap);

/* Upper bound, in milliseconds, on any single pipeline wait inside a kernel
 * (default 2000; also read from the environment variable FGF8_WAIT_TIMEOUT_MS
 * at first use).  Returns the previous value. */
FGF8_API int fgf8_set_wait_timeout_ms(int ms);

/* Library version as an integer (major * 10000 + minor * 100 + patch). */
FGF8_API int fgf8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FGF8_H */

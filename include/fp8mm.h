/*
 * fp8mm.h -- C ABI of libfp8mm, the GB300 (sm_103a) FP8 linear-layer hot path.
 *
 * Two operations and their variants, all asynchronous on the caller's CUDA
 * stream:
 *
 *  1. per_token_group_quant_fp8: bf16/fp16 activations -> E4M3FN codes +
 *     fp32 / UE8M0 scales, the producer of the GEMM's A operand; variants:
 *     topk scatter, the masked expert-major layout with fused SiLU*up, int8
 *     output, row-padded outputs.  Defined by sglang PR #33533 "[JIT]
 *     per_token_group_quant: fix the fp16 UE8M0 multiplier overflow, 1.23x on
 *     the fused EP-MoE path, unify the scale allocation" (Motivation;
 *     Modifications 1-3; commit notes for the scatter and the entry points).
 *     Static per-tensor activation quant and the requantization of a fused
 *     weight's per-shard scales to their maximum follow the prhub summary of
 *     sglang PR #33148 (Key source snippets).
 *
 *  2. fp8_scaled_mm: D = out_dtype(a_scale * b_scale * A B^T (+ bias)) with
 *     E4M3FN A [M,K] and B [N,K] (both K-major) and fp32 scales.
 *     Defined by sglang PR #34318 "[Kernel] Route large SM90 row/column-scaled
 *     FP8 GEMMs to Torch" (Summary: E4M3FN inputs, fp32 row/column scales,
 *     bf16 out), the prhub summary of sglang PR #33148 (per-tensor scalar
 *     scales passed through unbroadcast; weight stored [K,N] column-major =
 *     [N,K] K-major; K%16 / N%16 alignment; the bias argument) and sglang
 *     PR #44861 (deterministic, batch-invariant mode; zero-filled K tails).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library allocates no memory per call and never synchronizes the host.
 *  - Arguments are validated on the host before anything is launched; on any
 *    error a negative fp8mm_status is returned and nothing is launched (no
 *    fallback path exists).  M == 0 (or an empty problem) returns FP8MM_OK
 *    without a launch.
 *  - Launch failures return FP8MM_ECUDA; the CUDA error is left for the
 *    caller's next runtime call to observe as usual.
 *  - Kernels never trap.  Every wait inside a kernel is bounded; if one runs
 *    out the kernel records FP8MM_ETIMEOUT in a per-device status word, frees
 *    what it holds and returns.  fp8mm_get_device_status() reads that word.
 *  - `stream` is a cudaStream_t (0 = legacy default stream).
 *  - fp8_scaled_mm and the group / per-token quant entry points
 *    (per_token_group_quant_fp8 and its scatter, masked, int8 and row-padded
 *    forms) launch their kernels as programmatic dependents of the work before
 *    them on the stream: when that work lets its dependents start early, their
 *    CTAs launch and set up while it finishes, and read or write anything only
 *    once it has completed (griddepcontrol.wait).  The quant kernels, the
 *    static quant and the small-M (M <= 128) and deterministic cluster GEMMs
 *    let their own dependents start when they start, so in a decode step each
 *    kernel's launch and set-up overlap the end of the one before.  After any
 *    other work the kernel starts when that work ends, as usual.
 */
#ifndef FP8MM_H_
#define FP8MM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FP8MM_API __attribute__((visibility("default")))
#else
#define FP8MM_API
#endif

typedef struct CUstream_st* fp8mm_stream_t; /* same type as cudaStream_t */

typedef enum {
  FP8MM_OK = 0,
  FP8MM_EINVAL = -1,       /* bad shape, null pointer, bad mode */
  FP8MM_EALIGN = -2,       /* pointer / stride / size alignment violated */
  FP8MM_EUNSUPPORTED = -3, /* valid request this build does not implement */
  FP8MM_ECUDA = -4,        /* a CUDA runtime / driver call failed */
  FP8MM_ETIMEOUT = -5      /* a kernel-side bounded wait ran out */
} fp8mm_status;

/* Input / output element types. */
enum { FP8MM_DTYPE_BF16 = 0, FP8MM_DTYPE_FP16 = 1 };

/* Scale storage formats of the group quant (the `ue8m0` argument). */
enum {
  FP8MM_SCALE_FP32 = 0,          /* fp32 s = max(amax, 1e-10) / 448 */
  FP8MM_SCALE_FP32_POW2 = 1,     /* fp32 s = 2^(e-127), the UE8M0 value */
  FP8MM_SCALE_UE8M0_PACKED = 2   /* UE8M0 byte e, four groups per int32 */
};

/* GEMM scale modes: A side in bits 0-3, B side in bits 4-7. */
enum {
  FP8MM_SCALE_A_TENSOR = 0x0,          /* a_scale[0] */
  FP8MM_SCALE_A_ROW = 0x1,             /* a_scale[m], [M] */
  FP8MM_SCALE_A_GROUP128 = 0x2,        /* a_scale[m*(K/128) + g], [M, K/128] row-major */
  FP8MM_SCALE_A_GROUP128_COLMAJOR = 0x3, /* a_scale[g*pad4(M) + m], [K/128, pad4(M)] */
  FP8MM_SCALE_A_GROUP128_UE8M0 = 0x4,  /* UE8M0 bytes packed four per int32, column-major
                                          [ceil(K/512), pad4(M)] (the group quant's output):
                                          a_s(m, g) = 2^(e - 127), e = byte g%4 of word
                                          (g/4, m), as an fp32 value: e = 0 is the subnormal
                                          2^-127 and e = 255 is +inf (2^128 overflows fp32),
                                          the value the quant's FP32_POW2 format gives for
                                          the same group (finite inputs give 85 <= e <= 254,
                                          a group holding an infinity e = 255) */
  FP8MM_SCALE_B_TENSOR = 0x00,         /* b_scale[0] */
  FP8MM_SCALE_B_COL = 0x10,            /* b_scale[n], [N] */
  FP8MM_SCALE_B_BLOCK128 = 0x20        /* b_scale[(n/128)*(K/128) + g], [ceil(N/128), K/128];
                                          requires a per-group A mode */
};

/*
 * fp8_scaled_mm
 *   out[m, n] = round_out( a_s(m, .) * b_s(n) * sum_k A[m,k] * B[n,k]  (+ bias[n]) )
 *
 *   A        E4M3FN codes, row-major [M, lda] (first K columns used), device.
 *   B        E4M3FN codes, row-major [N, ldb] (first K columns used), device;
 *            i.e. the weight [K, N] stored column-major.
 *   a_scale  fp32, layout by scale_mode (see FP8MM_SCALE_A_*), device.
 *   b_scale  fp32, layout by scale_mode (see FP8MM_SCALE_B_*), device.
 *   bias     NULL or bf16 [N], device; added in fp32 after scaling.
 *   out      out_dtype (FP8MM_DTYPE_BF16 / _FP16) row-major [M, N], device;
 *            must not overlap A, B, the scales or the bias.
 *   Per-group A scales (FP8MM_SCALE_A_GROUP128*): the sum is formed per
 *   128-wide K block and promoted in fp32 as sum_g a_s[m,g] * partial_g; with
 *   128 x 128 block B scales (FP8MM_SCALE_B_BLOCK128) as
 *   sum_g a_s[m,g] * b_s[n/128,g] * partial_g (the block-scaled GEMM).
 *   deterministic != 0: batch-invariant mode -- one fixed tile shape and
 *   K-block order for every M, no split of K, zero-filled K tail; row m of
 *   the result is bit-identical for any M and any prefix / suffix split of
 *   the rows (sglang PR #44861, Modifications).
 *   Requirements (else FP8MM_EINVAL / FP8MM_EALIGN): M, N, K >= 0;
 *   K % 16 == 0; lda >= K, ldb >= K, lda % 16 == 0, ldb % 16 == 0;
 *   N % 8 == 0 (16-byte output rows); A, B, out 16-byte aligned; group
 *   modes need K % 128 == 0; K >= 16.  Returns FP8MM_OK or a negative status.
 */
FP8MM_API int fp8_scaled_mm(const void* A, const void* B, const float* a_scale, const float* b_scale,
                  int scale_mode, const void* bias, void* out, int out_dtype, int64_t M, int64_t N,
                  int64_t K, int64_t lda, int64_t ldb, int deterministic, fp8mm_stream_t stream);

/*
 * per_token_group_quant_fp8
 *   For each row m and group g of `group` consecutive columns:
 *     v      = x[m, k]                       (fuse_silu_mul == 0)
 *            = silu(x[m, k]) * x[m, K + k]   (fuse_silu_mul != 0; x is [M, 2K],
 *              gate first; silu(t) = t / (1 + exp(-t)), IEEE divide)
 *     a      = max(max_k |v|, 1e-10)
 *     s      = a / 448,  mult = 448 / a      (IEEE fp32 division)
 *     UE8M0 (ue8m0 != 0): e = exponent of s rounded up, s = 2^(e-127),
 *            mult = 2^(127-e)
 *     q[m,k] = E4M3FN_rne_satfinite(v * mult)   (fp32 multiply)
 *
 *   x        bf16 / fp16 (x_dtype) row-major [M, K] or [M, 2K], device, 16-byte aligned.
 *   q        uint8 E4M3FN codes, row-major [M, K], device, 16-byte aligned.
 *   s        scales, device (G = K / group):
 *              FP32 / FP32_POW2, row-major      : float [M, G]
 *              FP32 / FP32_POW2, column-major   : float [G, pad4(M)]
 *              UE8M0_PACKED, row-major          : int32 [M, ceil(G/4)]
 *              UE8M0_PACKED, column-major       : int32 [ceil(G/4), pad4(M)]
 *            pad4(M) = M rounded up to a multiple of 4.  Group 4j+b sits in
 *            byte b of word j; unused bytes of the last word are written as 0;
 *            padding columns are not written.
 *   group    32, 64 or 128, or group == K (one scale per row).
 *   Requirements: K % 16 == 0, K % group == 0; else FP8MM_EINVAL.
 */
FP8MM_API int per_token_group_quant_fp8(const void* x, int x_dtype, uint8_t* q, void* s, int64_t M, int64_t K,
                              int group, int ue8m0, int scale_colmajor, int fuse_silu_mul,
                              fp8mm_stream_t stream);

/*
 * per_token_group_quant_fp8_scatter
 *   The same quant of x [M, K] (no SiLU), each token quantized once and its
 *   codes and scales written to every destination row dst_row[m*topk + t]
 *   (entries < 0 are skipped) -- the MoE gate/up input layout of sglang PR
 *   #33533's second commit note.  Destination rows must be distinct.
 *   q is [num_dst_rows, K]; s is laid out as for per_token_group_quant_fp8
 *   with num_dst_rows in place of M (column-major = the MN-major grouped-GEMM
 *   scale buffer).  Rows not named by dst_row are not written.
 *   dst_row  int32 [M, topk], device.  Entries must be < num_dst_rows (checked
 *            on the device: out-of-range entries are skipped and recorded as
 *            FP8MM_EINVAL in the device status word).
 */
FP8MM_API int per_token_group_quant_fp8_scatter(const void* x, int x_dtype, const int32_t* dst_row, int topk,
                                      int64_t num_dst_rows, uint8_t* q, void* s, int64_t M,
                                      int64_t K, int group, int ue8m0, int scale_colmajor,
                                      fp8mm_stream_t stream);

/*
 * silu_and_mul_masked_post_quant_fp8
 *   The fused SiLU(gate)*up group quant on the expert-major layout that an
 *   expert-parallel MoE dispatch produces (sglang PR #33533, Speed Tests: the
 *   fused, masked, column-packed UE8M0 path of EP-MoE decode):
 *   x [E, T, 2K] (gate = x[e, t, :K], up = x[e, t, K:]), of which only the
 *   first masked_m[e] rows of expert e hold tokens.  For those rows the result
 *   is exactly per_token_group_quant_fp8 with fuse_silu_mul on x viewed as
 *   [E*T, 2K]; all other rows of q and s are left untouched.
 *   q        uint8 [E, T, K], device.
 *   s        row-major: as per_token_group_quant_fp8 with E*T rows;
 *            column-major: per expert, float [E, G, pad4(T)] or packed
 *            int32 [E, ceil(G/4), pad4(T)].
 *   masked_m int32 [E], device; values outside [0, T] are clamped and
 *            recorded as FP8MM_EINVAL in the device status word.
 *   E        at most 1024 (each CTA stages masked_m in shared memory).
 *   group    32, 64 or 128.  Requirements as per_token_group_quant_fp8.
 */
FP8MM_API int silu_and_mul_masked_post_quant_fp8(const void* x, int x_dtype, const int32_t* masked_m, int64_t E,
                                                 int64_t T, int64_t K, uint8_t* q, void* s, int group, int ue8m0,
                                                 int scale_colmajor, fp8mm_stream_t stream);

/*
 * per_token_group_quant_int8
 *   The int8 output format of the same group quant (sglang PR #33533,
 *   "Verified": fp32 / ue8m0 / int8 formats; the entry-point notes name
 *   sglang_per_token_group_quant_int8): per group, a = max(absmax, 1e-10),
 *   s = fl32(a / 127), q = int8 of fl32(v * fl32(127 / a)) after min(., 127)
 *   (NaN -> +127), rounded to nearest even, saturating at -128.
 *   q      int8 [M, K], device, 16-byte aligned.
 *   s      fp32, row-major [M, K/group] or column-major [K/group, pad4(M)].
 *   Other arguments as per_token_group_quant_fp8 (no scatter, no masked layout).
 */
FP8MM_API int per_token_group_quant_int8(const void* x, int x_dtype, int8_t* q, float* s, int64_t M, int64_t K,
                                         int group, int scale_colmajor, int fuse_silu_mul, fp8mm_stream_t stream);

/*
 * per_token_group_quant_fp8_row_padded
 *   The group quant into outputs sized for M_pad >= M rows, rows M .. M_pad-1
 *   zeroed (codes 0, scale entries 0): the row padding plus tail zeroing that
 *   the plain entry cannot express (sglang PR #33533, entry-point dedup notes).
 *   q  uint8 [M_pad, K].  s  as per_token_group_quant_fp8 with M_pad rows:
 *   row-major [M_pad, cols] or column-major [cols, pad4(M_pad)], cols = K/group
 *   (fp32) or ceil(K/group/4) (packed UE8M0).  Columns M_pad .. pad4(M_pad)-1
 *   of a column-major buffer are not written.  Two launches on `stream`.
 */
FP8MM_API int per_token_group_quant_fp8_row_padded(const void* x, int x_dtype, uint8_t* q, void* s, int64_t M,
                                                   int64_t M_pad, int64_t K, int group, int ue8m0,
                                                   int scale_colmajor, fp8mm_stream_t stream);

/*
 * static_per_tensor_quant_fp8
 *   Static per-tensor activation quant with a given scale (the checkpoint's
 *   activation scale, prhub summary of sglang PR #33148, Key source snippets):
 *   q[i] = E4M3FN_rne_satfinite(fl32(x[i] / scale[0])), IEEE division; a NaN
 *   quotient encodes as +448.
 *   x      bf16 / fp16 [numel], device, 16-byte aligned; numel % 16 == 0.
 *   scale  fp32 [1], device.   q  uint8 [numel], device, 16-byte aligned.
 */
FP8MM_API int static_per_tensor_quant_fp8(const void* x, int x_dtype, const float* scale, uint8_t* q, int64_t numel,
                                          fp8mm_stream_t stream);

/*
 * requantize_with_max_scale_fp8
 *   A fused weight (e.g. QKV or gate/up) whose logical shards carry their own
 *   per-tensor scales is brought to one scale, the largest (same snippets,
 *   process_weights_after_loading): s_max = max_i shard_scales[i]; every row of
 *   shard i becomes E4M3(fl32(fl32(decode(w) * s_i) / s_max)); rows past the
 *   last shard are copied.  s_max is written to max_scale_out[0].
 *   w, w_out        uint8 E4M3 codes [N, K], device, 16-byte aligned (w_out may be w).
 *   shard_scales    fp32 [num_shards], device.
 *   logical_widths  int64 [num_shards], HOST; rows of each shard in order, sum <= N.
 *   max_scale_out   fp32 [1], device; must not overlap shard_scales (FP8MM_EINVAL).
 *   num_shards      1 .. 16.   K % 16 == 0.
 */
FP8MM_API int requantize_with_max_scale_fp8(const uint8_t* w, uint8_t* w_out, const float* shard_scales,
                                            const int64_t* logical_widths, int num_shards, int64_t N, int64_t K,
                                            float* max_scale_out, fp8mm_stream_t stream);

/*
 * Device status word of `device` (the current device if device < 0):
 * FP8MM_OK, or the first error a kernel recorded there (FP8MM_ETIMEOUT,
 * FP8MM_EINVAL).  Reading synchronizes with the device.  clear != 0 resets
 * it to FP8MM_OK after reading.  Returns FP8MM_ECUDA if the word cannot be
 * read.
 */
FP8MM_API int fp8mm_get_device_status(int device, int clear);

/*
 * Diagnostic: launch one kernel that waits on a barrier nothing ever arrives
 * on, through the same bounded wait the GEMM uses.  After `timeout_ns`
 * (1 .. 1e10) the wait gives up, records FP8MM_ETIMEOUT in the device status
 * word and the kernel returns; the context stays usable.  Returns FP8MM_OK
 * when the kernel was launched.
 */
FP8MM_API int fp8mm_selftest_bounded_wait(int64_t timeout_ns, fp8mm_stream_t stream);

/*
 * Diagnostic: the limit, in ns, of the waits inside the pipelines of the GEMM
 * kernels (stage, accumulator and cluster hand-offs) and of the group-quant
 * kernel (stage hand-offs) for every launch after this call, process-wide; 0
 * restores the default (2 s, also the most allowed).  A short limit makes real
 * waits give up mid-run: the kernel then records FP8MM_ETIMEOUT, leaves every
 * output it had not finished unwritten (GEMM tiles; the quant's items of up to
 * 32 rows x 512 columns), waits with the full limit for its own copies and MMAs
 * in flight, frees its TMEM and returns -- the path a fault in production would
 * take, exercised without one.  Returns FP8MM_EINVAL for a negative or larger
 * value; not for use while other host threads launch kernels that expect the
 * default.
 */
FP8MM_API int fp8mm_set_wait_timeout_ns(int64_t timeout_ns);

/*
 * Diagnostic: evaluate the quant kernels' per-group scale arithmetic for every
 * fp32 value whose bit pattern lies in [bits_lo, bits_hi) (bits_hi <=
 * 0x7F800000) and compare it with IEEE division: adds to device counters
 * mismatches[0] (a/448), mismatches[1] (448/a) and mismatches[2] (the UE8M0
 * exponent byte), for a = max(value, 1e-10).  `mismatches` is a device array of
 * three unsigned 64-bit counters owned by the caller.
 */
FP8MM_API int fp8mm_selftest_scale_math(uint32_t bits_lo, uint32_t bits_hi, unsigned long long* mismatches,
                                        fp8mm_stream_t stream);

/* Human-readable name of a status code (static string). */
FP8MM_API const char* fp8mm_status_string(int status);

/* Library ABI version, (major << 16) | minor. */
FP8MM_API int fp8mm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8MM_H_ */

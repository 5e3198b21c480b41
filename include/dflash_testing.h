/*
 * dflash_testing.h -- test hooks of libdflash.so (not part of the DFlash operations).
 *
 * They expose single kernels of the library so tests can check them in isolation.  The
 * four operations of dflash.h never depend on these hooks.
 */
#ifndef DFLASH_TESTING_H_
#define DFLASH_TESTING_H_

#include <stdint.h>

#include "dflash.h"

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_TESTING_ENGINE_TC 0   /* tcgen05 / TMEM / TMA kernel (bf16 or fp16) */
#define DFLASH_TESTING_ENGINE_SIMT 1 /* CUDA-core kernel (fp32 accumulation, no TF32) */

/* C[z] (float32, [splits][M][ldc]) = A[:, Kz] * B[:, Kz]^T, A [M, K] (row stride lda) and
 * B [N, K] (row stride ldb) both of type dtype (tensor cores: DFLASH_DTYPE_BF16 or _F16;
 * CUDA cores: _BF16 or _F32), device pointers.  The K range is cut into `splits`
 * contiguous slices of 64-element steps; slice z goes to C + z*M*ldc.  Asynchronous on
 * `stream`.  Returns a DFLASH_* status. */
DFLASH_API int dflash_testing_gemm(int engine, int dtype, const void* A, long lda, const void* B,
                                   long ldb, float* C, long ldc, long M, int N, int K, int splits,
                                   void* stream);

/* Weight-streaming projection GEMM of the draft layers (tcgen05 with the weight rows as the
 * MMA's M operand, converted to fp16 in tensor memory): C[z] (float32, [splits][M][ldc]) =
 * X[:, Kz] * W[:, Kz]^T for the token rows of the 128-row tiles in tile_list (device int32
 * array: [0] = count, then tile indices; NULL = every tile).  X fp16 [M, K] (row stride ldx),
 * W [N, K] of type w_dtype (DFLASH_DTYPE_BF16 or _F16; row stride ldw), strides multiples
 * of 8 elements.  The device picks the split count (<= max_splits) and writes it to
 * *splits_out (device int32).  Rows of unlisted tiles are left unwritten. */
DFLASH_API int dflash_testing_gemm_ws(const void* X, long ldx, const void* W, int w_dtype,
                                      long ldw, float* C, long ldc, long M, int N, int K,
                                      int max_splits, const int32_t* tile_list,
                                      int32_t* splits_out, void* stream);

/* Failure detection of the tensor-core kernels: the bf16 GEMM of dflash_testing_gemm
 * (one K slice) with its TMA producer withholding every copy and every arrival, and every
 * bounded device wait limited to wait_ns (1 us .. 100 ms).  Nothing ever fills the first
 * shared-memory stage, so the MMA thread's wait runs out: each CTA raises its abort flag,
 * reports DFLASH_ERR_TIMEOUT in the device status word, waits (bounded) for its own work in
 * flight, frees its tensor memory and exits.  C is left unwritten; the device stays usable.
 * No GPU fault, trap or endless wait is involved. */
DFLASH_API int dflash_testing_gemm_withheld(const void* A, long lda, const void* B, long ldb,
                                            float* C, long ldc, long M, int N, int K,
                                            long wait_ns, void* stream);

/* The K-split the library picks for an M x N x K projection on the current device. */
DFLASH_API int dflash_testing_gemm_splits(long M, int N, int K);

/* How the 128 x 256-tile tensor-core GEMM behind every 16-bit projection runs, for the
 * calls that follow: 0 (default) as pairs of CTAs (a thread-block cluster of two computing a
 * 256 x 256 tile with tcgen05 cta_group::2 MMAs, each CTA loading its 128 rows of A and
 * half of the B tile) whenever the GEMM has at least two 128-row M tiles, else one CTA per
 * 128 x 256 tile; 1: one CTA per tile everywhere.  Results are bit-identical between the
 * two (same MMA shapes per output element and K order).  Process-wide; returns a DFLASH_*
 * status. */
DFLASH_API int dflash_testing_gemm_pairs(int mode);

/* Which body projections of the bf16 configuration use the fused epilogues of the
 * 128 x 256-tile GEMM (Q/K RoPE and the attention layouts written by the QKV projection's
 * epilogue; the residual add done by the O and down projections' epilogues), for the calls
 * of dflash_body_forward that follow:
 *   0 (default) where the projection's output tiles fill three waves of the SMs without a
 *     K-split; 1 on every call that runs on the 128 x 256-tile GEMM; 2 never.
 * The results agree with the unfused path within fp32 rounding of the RoPE products.
 * Process-wide; returns a DFLASH_* status. */
DFLASH_API int dflash_testing_fused_epilogues(int mode);

/* The chunk plan of greedy verification, computed on the host (no device needed): each of
 * the B*(gamma+1) logits rows of length V is cut into *chunks column ranges of *chunk_len
 * elements (a multiple of 8), sized for `resident_ctas` resident argmax CTAs.  With
 * static_entries > 0 the plan is then capped as dflash_verify_greedy_static caps it: at
 * most static_entries partials in all.  Returns a DFLASH_* status. */
DFLASH_API int dflash_testing_verify_plan(int B, int gamma, int V, long resident_ctas,
                                          long static_entries, int* chunks, int* chunk_len);

/* The RoPE table the draft body and the context projection build on the device ("DFlash",
 * Configuration: rotary position embedding with base rope_theta): cos_t[p][i] and
 * sin_t[p][i] of the angle (p0 + p) * theta^(-2i / head_dim) for p < P, i < head_dim / 2,
 * float32, row-major [P][head_dim / 2], device pointers 16-byte aligned.  Needs head_dim even
 * and <= 256, P >= 1, 0 <= p0 and p0 + P <= 2^24 (positions exact in float32).  Enqueued on
 * `stream`; returns a DFLASH_* status. */
DFLASH_API int dflash_testing_rope_table(float* cos_t, float* sin_t, int p0, int P, int head_dim,
                                         double theta, void* stream);

/* ---- live kernel timing ----------------------------------------------------------------
 * While enabled, every kernel launch of the four operations is bracketed by two CUDA events
 * recorded on the launch stream, grouped by kind.  Enabling clears earlier records. */
#define DFLASH_PROF_GEMM 0       /* tensor-core / CUDA-core projection GEMMs */
#define DFLASH_PROF_ATTENTION 1  /* block-sparse attention */
#define DFLASH_PROF_ROWS 2       /* norms, RoPE table, GEMM epilogues */
#define DFLASH_PROF_PLAN 3       /* anchor plan */
#define DFLASH_PROF_VERIFY 4     /* argmax + accepted-prefix scan */
#define DFLASH_PROF_CONVERT 5    /* bf16 -> fp16 weight conversion */
#define DFLASH_PROF_KINDS 6

DFLASH_API int dflash_profile_enable(int on);

/* Synchronizes the current device, then returns the summed event time (ms) and the number
 * of launches of one kind recorded since profiling was enabled. */
DFLASH_API int dflash_profile_read(int kind, double* total_ms, long* launches);

/* Kernel launches issued by the library in this process (always counted). */
DFLASH_API long dflash_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_TESTING_H_ */

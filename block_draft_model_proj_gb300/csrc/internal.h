// Internal launch interfaces between the C ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace dflash {

// Launch with programmatic stream serialization (the kernel must call pdl_wait() before its
// first global-memory access).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same, launched as thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                      size_t smem, cudaStream_t stream, int cluster_x,
                                      Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- api.cu ----
// Records the thread-local message returned by dflash_last_error(); returns `code`.
int set_error(int code, const char* fmt, ...);

// ---- plan.cu ----
cudaError_t launch_plan(const uint8_t* mask, const int64_t* sids, int B, int L, uint64_t step,
                        uint64_t seed, int N, int S, int32_t* anchors, uint8_t* block_valid,
                        uint8_t* loss_mask, int32_t* position_ids, int32_t* ctx_len,
                        cudaStream_t stream);

// ---- verify.cu ----
struct VerifyPlan {
  int chunks = 1;
  int chunk_len = 0;
  size_t ws_bytes = 0;
};
// Chunks per row for `rows` rows of V logits: about three waves of the resident CTAs,
// chunks of at least 4096 elements, chunk_len a multiple of 8.
VerifyPlan plan_verify_for(long rows, int V, long resident_ctas);
VerifyPlan plan_verify(int B, int gamma, int V, int num_sms);
// At most max_entries partials in all: fewer, longer chunks when rows * chunks exceeds it
// (rows <= max_entries).  Keeps chunk_len % 8 == 0 and chunks * chunk_len >= V.
VerifyPlan cap_verify_chunks(VerifyPlan vp, long rows, int V, long max_entries);
// Dynamic shared memory of the prefix-scan kernel: (gamma + 1) ints per warp, up to four
// warps; above the default 48 KB the launch raises the kernel's limit, up to kScanSmemMax.
constexpr size_t kScanSmemDefault = 48 * 1024;
constexpr size_t kScanSmemMax = 227 * 1024;
// Logits rows (B * (gamma + 1)) a verification call takes: one grid row of CTAs per logits row.
constexpr long kMaxVerifyRows = 65535;
// Largest gamma the verification calls accept: one warp's (gamma + 1) choices in shared memory.
constexpr int kMaxVerifyGamma = (int)(kScanSmemMax / sizeof(int)) - 1;
cudaError_t launch_verify(const void* logits, int dtype, const int32_t* draft, int B, int gamma,
                          int V, int32_t eos, int32_t* emitted, int32_t* num_emitted,
                          int32_t* accepted, int32_t* choices, float* part_v, int* part_i,
                          const VerifyPlan& vp, cudaStream_t stream);

// ---- verify_sampling.cu: speculative-sampling verification ----
struct SamplingPlan {
  int chunks = 1, chunk_len = 0;            // softmax statistics: chunks per logits row
  int race_chunks = 1, race_chunk_len = 0;  // the sampled row of each request
  size_t ws_bytes = 0;
};
SamplingPlan plan_sampling(int B, int gamma, int V, int num_sms);
// logits [B][gamma+1][V] (bf16 or fp32), q [B][gamma][V] fp32 (the actual proposal
// distributions), draft [B][gamma]; ws holds plan.ws_bytes.  y_scale = log2(e) / temperature:
// the softmax runs in base 2 on y = logit * y_scale.  A draft token outside [0, V)
// reports a device check and counts as rejected.
cudaError_t launch_verify_sampling(const void* logits, int dtype, float y_scale, const float* q,
                                   const int32_t* draft, int B, int gamma, int V, uint64_t seed,
                                   int32_t eos, int32_t* emitted, int32_t* num_emitted,
                                   int32_t* accepted, void* ws, const SamplingPlan& sp,
                                   unsigned* status, cudaStream_t stream);

// ---- loss.cu: decayed cross-entropy of the lm_head over the drafted blocks ----
struct CeLayout {
  int n_tiles = 0;                     // vocab tiles of 256 columns
  __nv_bfloat16* hidden16 = nullptr;   // [T][D] bf16 GEMM operand
  float* part = nullptr;               // [T][n_tiles][2]
  float* tlogit = nullptr;             // [T]
  int32_t* tile_list = nullptr;        // 128-row tiles with a masked slot
  size_t bytes = 0;
};
CeLayout ce_layout(long T, int D, int V, void* ws);
cudaError_t launch_decayed_ce(const float* hidden, const void* lm_head, const int32_t* targets,
                              const uint8_t* mask, long T, int S, int D, int V, double decay,
                              float* ce, float* loss, const CeLayout& l, unsigned* status,
                              cudaStream_t stream);

// ---- rows.cu: row-wise kernels (norms, RoPE table, GEMM epilogues) ----
// RoPE table: cos/sin [P, dh/2] fp32 for positions p0 .. p0+P-1, angles formed and
// range-reduced in fp64 (inverse frequencies computed on the host in fp64; dh <= 256).
// Active 128-row tiles, built by one extra block of the RoPE-table launch: list[0] = count,
// list[1..] = the tiles in order.  kContext: context rows m = b*L + c with c < ctx_len[b];
// kSlots: slots t < T with valid[t] != 0.
struct TileJob {
  enum : int { kNone = 0, kContext = 1, kSlots = 2 };
  int kind = kNone;
  const int32_t* ctx_len = nullptr;
  const uint8_t* valid = nullptr;
  int B = 0, L = 0;
  long T = 0;
  long tiles = 0;  // set by the launcher
  int32_t* list = nullptr;
};
cudaError_t launch_rope_table(float* cos_t, float* sin_t, int p0, int P, int head_dim,
                              double theta, cudaStream_t stream, const TileJob& job = TileJob());

enum NormMode { kNormInit = 0, kNormAdd = 1, kNormFinal = 2 };
// Residual-stream step on rows of width D:
//  kNormInit : x = emb; h = RMSNorm(x) * g
//  kNormAdd  : x += sum_s y[s]; h = RMSNorm(x) * g
//  kNormFinal: x += sum_s y[s]; out = valid ? (final_norm ? RMSNorm(x) * g : x) : 0
// y: nsplit partial results [nsplit][rows][D] (fp32; the count read from *nsplit_dev when
// that is given); emb and g have type `dtype`.  With `valid`, a row of an invalid slot
// writes zeros (h, or out) and reads nothing.  nsplit = 0 without nsplit_dev: x already
// holds the sum (the GEMM epilogue added into it) and is only read.
cudaError_t launch_residual_norm(int mode, int dtype, float* x, const void* emb, const float* y,
                                 int nsplit, const int* nsplit_dev, const void* g, double eps,
                                 ActOut h, float* out, const uint8_t* valid, bool final_norm,
                                 long rows, int D, cudaStream_t stream);

// Plain RMSNorm of fp32 rows (the context norm); with_norm=false copies.  Rows r = b*L + c
// with c >= ctx_len[b] are skipped when ctx_len is given (vectorised path).
cudaError_t launch_rows_norm(int dtype, const float* y, int nsplit, const void* g, double eps,
                             bool with_norm, ActOut out, long rows, int D,
                             const int32_t* ctx_len, int L, cudaStream_t stream);

// QKV epilogue: y [nsplit][T][(Hq+2Hkv)*dh] fp32 -> attention-ready operands (fp16 when
// f16, else fp32) q [B][Hkv][N][S][grp][dh], kb [B][Hkv][N*S][dh], vbt [B][Hkv][dh][ns_pad];
// RoPE on q and k at position pos[t] (table of P positions; out-of-range valid slots report
// a device check and use position 0).  nsplit_dev (optional) overrides nsplit.
cudaError_t launch_qkv_rope(const float* y, int nsplit, const int* nsplit_dev, const int32_t* pos,
                            const uint8_t* valid,
                            const float* cos_t, const float* sin_t, int P, void* q, void* kb,
                            void* vbt, int ns_pad, long T, int N, int S, int Hq, int Hkv, int dh,
                            bool f16, unsigned* status, cudaStream_t stream);

// Zeroes what the fused QKV epilogue (launch_gemm_tc_qkv) never writes: q, kb and vbt of
// every slot of a 128-slot tile without a valid slot, and the pad columns N*S .. ns_pad-1 of
// vbt (fp16 operands, head_dim dh).  Run once per call, before the first layer.
cudaError_t launch_qkv_clear(const uint8_t* valid, __half* q, __half* kb, __half* vbt, int ns_pad,
                             long T, int N, int S, int Hq, int Hkv, int dh, cudaStream_t stream);

// Context K/V epilogue (fp32 configuration): y [nsplit][B*L][2*Hkv*dh] fp32 -> the fp32
// cache planes of one layer [B][2][Hkv]: K as [L_cache][dh] (RoPE'd; table row c = position
// pos_offset + c) and V^T as [dh][L_cache], at positions pos_offset + c.
// Rows c >= ctx_len[b] (when ctx_len is given) are not written.
// row_pos0 (optional [B]): as in KvCacheEpilogue.
cudaError_t launch_ctx_kv_scatter(const float* y, int nsplit, const float* cos_t,
                                  const float* sin_t, float* kv_layer, int B, int L,
                                  int pos_offset, int L_cache, int Hkv, int dh,
                                  const int32_t* ctx_len, const int32_t* row_pos0,
                                  cudaStream_t stream);

// Cache append after verification: for each row b, n[b] = accepted ? clamp(accepted[b] + 1,
// 0, P) : P positions commit at start[b] = cache_len[b]; cache_len[b] += n[b].  A row whose
// start is negative or whose new length would pass L_cache reports a device check and
// commits nothing (n[b] = 0, cache_len unchanged).
cudaError_t launch_append_plan(const int32_t* accepted, int32_t* cache_len, int B, int P,
                               int L_cache, int32_t* n, int32_t* start, unsigned* status,
                               cudaStream_t stream);

// SwiGLU epilogue: y [nsplit][T][2I] fp32 (gate | up) -> act [T][I] = SiLU(gate) * up.
// nsplit_dev (optional) overrides nsplit; valid (optional): invalid slots' rows get zeros.
cudaError_t launch_swiglu(const float* y, int nsplit, const int* nsplit_dev, ActOut act, long T,
                          int I, const uint8_t* valid, cudaStream_t stream);

// ---- gemm_simt.cu: C[z][M][N] (fp32) = A[M][K] * B[N][K]^T over K-split z ----
cudaError_t launch_gemm_simt(int dtype, const void* A, long lda, const void* Bm, long ldb,
                             float* C, long ldc, long M, int N, int K, int splits,
                             cudaStream_t stream);

// K-split for `units1` output tiles of `kb` K-steps each, at most max_splits: the fewest
// waves over `sms` SMs, weighing each tile's fixed cost as 6 K-steps; at least 8 K-steps
// per slice; never an empty slice.  The GEMMs that choose on the device and the kernels
// that sum their slices call it with the same arguments.
__host__ __device__ inline int choose_splits(long units1, int kb, int max_splits, int sms) {
  int best = 1;
  long best_cost = -1;
  for (int s = 1; s <= max_splits; ++s) {
    const int per = (kb + s - 1) / s;
    if ((kb + per - 1) / per != s) continue;
    if (s > 1 && per < 8) break;
    const long waves = (units1 * s + sms - 1) / sms;
    const long cost = waves * (per + 6);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// ---- gemm_tc.cu: tcgen05 16-bit GEMM, fp32 output, optional K-split ----
// elem = DFLASH_DTYPE_BF16 (A and B bf16) or DFLASH_DTYPE_F16 (A and B fp16).
// tile_list (optional, device): [0] = count, [1..] = the 128-row M tiles to compute, in
// order; tiles not listed are skipped entirely (their C rows are left unwritten).
constexpr int kGemmTileM = 128;
bool gemm_tc_supported(long M, int N, int K, long lda, long ldb);

// Destination of the context K/V projection written straight from the GEMM epilogue
// (head_dim 128): rows m = b*L + c of the GEMM are cache positions pos_offset + c.
struct KvCacheEpilogue {
  __half* kv = nullptr;          // first layer: [B][2][Hkv] fp16 planes, K [L_cache][128], V^T [128][L_cache]
  const float* cos_t = nullptr;  // [L][64], row c = position pos_offset + c
  const float* sin_t = nullptr;
  const int32_t* ctx_len = nullptr;  // optional [B]: rows c >= ctx_len[b] are not written
  // optional [B]: row b's context index c is cache position row_pos0[b] + c and its RoPE
  // angle is the table row of that absolute position (the table then starts at position 0);
  // without it the position is pos_offset + c and the table row c
  const int32_t* row_pos0 = nullptr;
  int L = 0, pos_offset = 0, L_cache = 0, Hkv = 0;
  // `layers` consecutive layers in one GEMM: columns [l * 2*Hkv*128, (l+1) * 2*Hkv*128) are
  // layer l's K then V heads, written to the planes at kv + l * layer_elems
  int layers = 1;
  long layer_elems = 0;
};
// Attention-ready Q / K / V of the draft body's QKV projection written straight from the
// GEMM epilogue (head_dim 128, no K-split): GEMM row t is slot t = (b, k, j) of the blocks,
// columns are the Q heads, then the K heads, then the V heads.  Q and K get RoPE at
// position pos[t] (table rows [P][64]) and land in q [B][Hkv][N][S][grp][128] and
// kb [B][Hkv][N*S][128]; V lands transposed in vbt [B][Hkv][128][ns_pad].  Invalid slots
// are written as zeros.  Slots of 128-row tiles the GEMM skips and the pad columns
// N*S .. ns_pad-1 of vbt are not written (launch_qkv_clear zeroes them once per call).
struct QkvEpilogue {
  const int32_t* pos = nullptr;
  const uint8_t* valid = nullptr;
  const float* cos_t = nullptr;
  const float* sin_t = nullptr;
  __half* q = nullptr;
  __half* kb = nullptr;
  __half* vbt = nullptr;
  int P = 0, ns_pad = 0, NS = 0, S = 0, Hq = 0, Hkv = 0;
};
cudaError_t launch_gemm_tc_qkv(const void* A, long lda, const void* Bm, long ldb, long M, int N,
                               int K, const int32_t* tile_list, const QkvEpilogue& e,
                               unsigned* status, cudaStream_t stream);
// x[t][:] += (A Bm^T)[t][:] for the valid rows t (fp16 operands, fp32 residual stream of
// width N = ldx, no K-split): the O and down projections add into the residual stream.
cudaError_t launch_gemm_tc_residual(const void* A, long lda, const void* Bm, long ldb, float* x,
                                    long ldx, long M, int N, int K, const int32_t* tile_list,
                                    const uint8_t* valid, unsigned* status, cudaStream_t stream);
// Cross-entropy statistics of lm_head logits, computed in the GEMM epilogue (the logits are
// never stored): for row m and vocab tile n_t (columns n_t*256 .. +255 below V),
// part[(m * n_tiles + n_t) * 2 + {0, 1}] = (max, sum of exp(logit - max)); the tile holding
// targets[m] writes that logit to target_logit[m].
struct CrossEntropyEpilogue {
  const int32_t* targets = nullptr;  // [M]
  float* part = nullptr;             // [M][n_tiles][2]
  float* target_logit = nullptr;     // [M]
  int V = 0;
};
// A bf16 [M][K] (hidden states), Bm bf16 [V][K] (lm_head); tile_list as for launch_gemm_tc.
cudaError_t launch_gemm_tc_cross_entropy(const void* A, long lda, const void* Bm, long ldb,
                                         long M, int V, int K, const int32_t* tile_list,
                                         const CrossEntropyEpilogue& ce, unsigned* status,
                                         cudaStream_t stream);
// act = SiLU(gate) * up with [gate | up] = A W_gate_up^T (W_gate_up [2I][K]: gate rows then
// up rows), written by the epilogue (no K-split).
cudaError_t launch_gemm_tc_swiglu(int elem, const void* A, long lda, const void* Bm, long ldb,
                                  long M, int I, int K, const int32_t* tile_list,
                                  const ActOut& act, unsigned* status, cudaStream_t stream);
// C = A B^T with N = kv.layers * 2*Hkv*128, written to the cache by the epilogue (no K-split).
cudaError_t launch_gemm_tc_kv_cache(int elem, const void* A, long lda, const void* Bm, long ldb,
                                    long M, int N, int K, const int32_t* tile_list,
                                    const KvCacheEpilogue& kv, unsigned* status,
                                    cudaStream_t stream);
// splits_out == nullptr: exactly `splits` K-slices.  Otherwise at most `splits`, the count
// chosen on the device from the active M tiles (choose_splits) and written to *splits_out.
cudaError_t launch_gemm_tc(int elem, const void* A, long lda, const void* Bm, long ldb, float* C,
                           long ldc, long M, int N, int K, int splits, const int32_t* tile_list,
                           unsigned* status, cudaStream_t stream, int* splits_out = nullptr);

// 0 (default): the 128 x 256-tile GEMMs run as CTA pairs (256 x 256 per pair) from two M
// tiles up; 1: one CTA per 128 x 256 tile everywhere.  Process-wide.
void set_gemm_tc_pairs(int mode);

// Testing only: the bf16 GEMM with its TMA producer withholding every copy and arrival and
// every bounded wait limited to wait_ns, so the MMA thread's first wait runs out: the CTAs
// report kStatusTimeout, drain, free their tensor memory and exit without writing C.
cudaError_t launch_gemm_tc_withheld(const void* A, long lda, const void* Bm, long ldb, float* C,
                                    long ldc, long M, int N, int K, uint64_t wait_ns,
                                    unsigned* status, cudaStream_t stream);

// ---- gemm_ws.cu: weight-streaming tcgen05 GEMM of the draft layers ----
// C[z][t][n] = X[t, Kz] W[n, Kz]^T over the active 128-row token tiles: X fp16 [M][K] (row
// stride ldx), W bf16 or fp16 [Nw][K] (row stride ldw; converted to fp16 on the fly).  The
// fp32 variant cuts K into up to max_splits slices (count chosen on the device, written to
// *splits_out); the SwiGLU and K/V-cache variants never split.
struct WsArgs {
  const void* X = nullptr;
  long ldx = 0;
  long M = 0;
  const void* W = nullptr;
  int w_dtype = DFLASH_DTYPE_BF16;
  long ldw = 0;
  int Nw = 0;
  int K = 0;
  const int32_t* tile_list = nullptr;
  float* C = nullptr;
  long ldc = 0;
  int max_splits = 1;
  int* splits_out = nullptr;
  unsigned* status = nullptr;
};
// Split count the device picks for units1 (weight tile, token tile) units and K.
int gemm_ws_splits(long units1, int K, int max_splits);
cudaError_t launch_gemm_ws(const WsArgs& a, cudaStream_t stream);
// act[t][i] = SiLU(gate) * up, W = W_gate_up [2I][K] (gate rows, then up rows); Nw = 2I.
cudaError_t launch_gemm_ws_swiglu(const WsArgs& a, const ActOut& act, cudaStream_t stream);

// ---- rows.cu: bf16 -> fp16 conversion (weights) ----
// dst[i] = fp16(src[i]), round to nearest even; exact for bf16 values of magnitude in
// [2^-14, 65504] and zero.  Non-finite results report kStatusRange.  16-byte aligned.
cudaError_t launch_convert_bf16_f16(const void* src, void* dst, size_t n, unsigned* status,
                                    cudaStream_t stream);

// ---- rows.cu: compacted lists of active 128-row M tiles for the GEMMs ----
// list[0] = count, list[1..] = tile indices in increasing order; list holds 1 + tiles ints.
// Rows t: tile active iff some row is a valid slot (the body builds its list inside the
// RoPE-table launch, TileJob).
cudaError_t launch_slot_tile_list(const uint8_t* valid, long T, int32_t* list,
                                  cudaStream_t stream);

// ---- attention.cu ----
struct AttnArgs {
  const float* q;           // [B][Hkv][N][S][grp][dh]
  const float* kb;          // [B][Hkv][N*S][dh]
  const float* vbt;         // [B][Hkv][dh][ns_pad]
  int ns_pad;
  const float* kv_layer;    // [B][2][Hkv] planes: K [L][dh], V^T [dh][L]
  const int32_t* anchors;   // [B][N]
  const uint8_t* valid;     // [B][N][S]
  const uint8_t* mask;      // [B][L]
  ActOut out;               // [T][Hq*dh]
  int B, N, S, L, Hq, Hkv, dh;
  unsigned* status;
};
cudaError_t launch_attention_simt(int dtype, const AttnArgs& a, cudaStream_t stream);

// ---- attention_tc.cu: tcgen05 (kind::f16) attention over attention-ready fp16 layouts ----
struct AttnTcArgs {
  const __half* q;          // [B][Hkv][N][S][grp][dh]
  const __half* kb;         // [B][Hkv][N*S][dh] block keys
  const __half* vbt;        // [B][Hkv][dh][ns_pad] block values transposed
  int ns_pad;               // row stride of vbt (>= N*S, multiple of 8)
  const __half* kv_layer;   // [B][2][Hkv] planes: K [L][dh], V^T [dh][L] (fp16)
  const int32_t* anchors;
  const uint8_t* valid;
  const uint8_t* mask;
  float* partials;          // attention_tc_layout(...).part_floats floats
  ActOut out;               // [T][Hq*dh]
  int B, N, S, L, Hq, Hkv;
  int num_sms;
  unsigned* status;
};
struct AttnTcLayout {
  int grp, R, bpt, tiles, chunk, max_chunks;
  long units;
  long part_floats;
};
AttnTcLayout attention_tc_layout(int B, int N, int S, int L, int Hq, int Hkv, int num_sms);
bool attention_tc_supported(int S, int Hq, int Hkv, int dh);
cudaError_t launch_attention_tc(const AttnTcArgs& a, cudaStream_t stream);

}  // namespace dflash

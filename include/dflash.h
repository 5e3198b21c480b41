/*
 * dflash.h -- C ABI of libdflash.so: the DFlash draft-body forward pass and greedy block
 * verification on one NVIDIA GB300 (sm_103a).
 *
 * The operations come from three public pages about DFlash:
 *   [P1] "DFlash" (angelspec docs): "How it works" (block-parallel prediction with a
 *        block-causal mask, dual-source KV context through W_proj, anchor sampling) and
 *        "Configuration" (the JSON fields mirrored by dflash_config_t).
 *   [P2] "DFlash Draft Body" (NeMo RL design doc): "How It Works" steps 1-4 (anchor plan,
 *        draft blocks, block update, loss mask) and "Scope".
 *   [P3] "DFlash: drafting, verification, and speed": "One DFlash generation cycle"
 *        (greedy verification of a drafted block, the bonus token, EOS).
 *
 * Conventions shared by every call
 *  - Every tensor pointer is a DEVICE pointer owned by the caller, unless a parameter
 *    says "host".  Weight, embedding, hidden-state, cache, mask and output pointers of the
 *    body and projection calls must be 16-byte aligned (cudaMalloc gives 256).  The library allocates no device memory: scratch space comes from a
 *    caller-provided workspace `ws` of at least the size the matching *_workspace_size
 *    query returns, aligned to 256 bytes (cudaMalloc alignment).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns a status code.  Host-side argument checks return
 *    DFLASH_ERR_INVALID_ARG before anything is launched.  Device-side checks (an index
 *    outside its documented range, a bounded wait that ran out) do not stop the stream:
 *    they set a sticky per-device status word read by dflash_device_status().
 *  - Dense matrices are row-major; weight matrices are stored [out_features, in_features]
 *    (y = x W^T).  Row strides are exactly the row widths given below.
 *  - Floating-point storage type is cfg->dtype for weights, inputs and embeddings:
 *    DFLASH_DTYPE_BF16 or DFLASH_DTYPE_F32 (fp32 throughout, no TF32).  In the bf16
 *    configuration W_proj runs bf16 x bf16 on the tensor cores (the target hidden states
 *    are exact bf16); the draft layers' projections run fp16 x fp16 on the tensor cores:
 *    their weights are fp16 copies of the bf16 matrices (see DFLASH_FLAG_F16_LAYERS and
 *    dflash_convert_bf16_to_f16) and the activations feeding them (norm outputs, attention
 *    output, SwiGLU product) are rounded to fp16, whose 11 significant bits keep the body
 *    within its error bound; accumulation is fp32, the residual stream fp32.  Attention
 *    runs fp16 x fp16 on the tensor cores (fp16 Q, K, V and probabilities; fp32 softmax
 *    and accumulation) over an fp16 context K/V cache.  A value outside the fp16 range
 *    (an activation or a cache entry) sets DFLASH_ERR_RANGE.  The fp32 configuration keeps
 *    an fp32 cache.
 *  - The thread-local message of the last failing call: dflash_last_error().
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------ */
#define DFLASH_OK 0
#define DFLASH_ERR_INVALID_ARG 1   /* bad shape, null pointer, misalignment, too small ws */
#define DFLASH_ERR_UNSUPPORTED 2   /* valid request this build does not handle */
#define DFLASH_ERR_CUDA 3          /* a CUDA runtime call failed */
#define DFLASH_ERR_TIMEOUT 4       /* device status: a bounded device-side wait ran out */
#define DFLASH_ERR_DEVICE_CHECK 5  /* device status: a device-side index check failed */
#define DFLASH_ERR_RANGE 6         /* device status: a value outside the fp16 range (or a
                                      NaN) was stored as fp16 */

#define DFLASH_DTYPE_F32 0
#define DFLASH_DTYPE_BF16 1
#define DFLASH_DTYPE_F16 2         /* IEEE binary16: prepared layer weights only */

#define DFLASH_FLAG_FINAL_NORM 1u  /* output = RMSNorm(x; g_final) (else the raw residual) */
#define DFLASH_FLAG_CTX_NORM 2u    /* context = RMSNorm(H_cat W_proj^T; g_ctx) (else raw) */
/* bf16 configuration only: the layer matrices w_qkv, w_o, w_gate_up and w_down are given
 * as fp16 (made once per weight update with dflash_convert_bf16_to_f16).  Without it they
 * are bf16 and every projection or body call first converts the matrices it uses into its
 * workspace (one extra read and write of them per call). */
#define DFLASH_FLAG_F16_LAYERS 4u

/* Draft model shape ([P1] "Configuration"; the attention/MLP sizes of the draft layers).
 * num_heads % num_kv_heads == 0; head_dim a multiple of 8.  The bf16 configuration also needs
 * head_dim == 128, block_size * num_heads / num_kv_heads dividing 128, num_heads /
 * num_kv_heads dividing 16, and every matrix row width a multiple of 8
 * (DFLASH_ERR_UNSUPPORTED otherwise). */
typedef struct dflash_config {
  int32_t target_hidden;      /* D_t: width of one selected target layer */
  int32_t num_target_layers;  /* n_tl: number of selected target layers (concat width n_tl*D_t) */
  int32_t hidden;             /* D: draft hidden size */
  int32_t num_layers;         /* NL: draft decoder layers */
  int32_t num_heads;          /* Hq */
  int32_t num_kv_heads;       /* Hkv */
  int32_t head_dim;           /* dh */
  int32_t intermediate;       /* I: SwiGLU width */
  int32_t block_size;         /* S = gamma + 1: anchor plus gamma draft positions */
  int32_t dtype;              /* DFLASH_DTYPE_* */
  uint32_t flags;             /* DFLASH_FLAG_* */
  int32_t reserved;
  double rope_theta;          /* RoPE base ([P1] "Configuration": rope_theta) */
  double rms_eps;             /* RMSNorm epsilon */
} dflash_config_t;

/* One draft decoder layer (pre-norm attention + SwiGLU MLP), device pointers, dtype cfg->dtype
 * (the four matrices fp16 under DFLASH_FLAG_F16_LAYERS; the gains stay cfg->dtype). */
typedef struct dflash_layer_weights {
  const void* g_in;       /* [D] input RMSNorm gain */
  const void* w_qkv;      /* [(Hq + 2*Hkv)*dh, D]: rows = Q heads, then K heads, then V heads */
  const void* w_o;        /* [D, Hq*dh] */
  const void* g_post;     /* [D] post-attention RMSNorm gain */
  const void* w_gate_up;  /* [2*I, D]: rows 0..I-1 gate, rows I..2I-1 up */
  const void* w_down;     /* [D, I] */
} dflash_layer_weights_t;

typedef struct dflash_weights {
  const void* w_proj;                    /* [D, n_tl*D_t] context projection W_proj */
  const void* g_ctx;                     /* [D] context RMSNorm gain */
  const void* g_final;                   /* [D] output RMSNorm gain */
  const dflash_layer_weights_t* layers;  /* HOST array of num_layers entries */
  int32_t num_layers;                    /* must equal cfg->num_layers */
} dflash_weights_t;

/* ---- housekeeping ------------------------------------------------------------------ */

/* Message of the last non-OK status returned on this host thread ("" if none). */
DFLASH_API const char* dflash_last_error(void);

/* Library ABI version (major*10000 + minor*100 + patch). */
DFLASH_API int dflash_version(void);

/* Synchronizes the current device, then returns its sticky device-side status:
 * DFLASH_OK, DFLASH_ERR_TIMEOUT, DFLASH_ERR_DEVICE_CHECK or DFLASH_ERR_RANGE
 * (DFLASH_ERR_CUDA if the synchronization itself fails).  reset != 0 clears the word
 * afterwards. */
DFLASH_API int dflash_device_status(int reset);

/* dst[i] = fp16(src[i]) for n bf16 values, round to nearest even (device pointers, 16-byte
 * aligned, asynchronous on stream).  Exact for zero and for magnitudes in [2^-14, 65504];
 * smaller magnitudes land on the fp16 subnormal grid (error <= 2^-25); a result that is not
 * finite sets DFLASH_ERR_RANGE.  Prepares the layer matrices for DFLASH_FLAG_F16_LAYERS. */
DFLASH_API int dflash_convert_bf16_to_f16(const void* src, void* dst, size_t n, void* stream);

/* ---- 1. anchor plan ([P2] How It Works, steps 1, 2 and 4) ---------------------------- */

DFLASH_API size_t dflash_plan_workspace_size(int B, int L, int num_anchors, int block_size);

/* Deterministic anchor plan for B rows of L target positions.
 *   mask        [B, L] uint8, nonzero = valid target position
 *   sample_ids  [B] int64; rows sharing an id get the anchors of the lowest such row
 *   step, seed  optimizer step and seed (taken as uint64)
 * Candidate anchor a: mask[a] and mask[a+1] valid (a+1 < L).  The num_anchors candidates
 * with the smallest (key, a), key = SplitMix64 chain of (seed, step, sample id, a), sorted
 * by position; missing anchors are -1 and come last.
 * Outputs (device, caller-owned, fully written):
 *   anchors      [B, N] int32
 *   block_valid  [B, N, S] uint8: anchor != -1, position a valid, position a+j valid
 *   loss_mask    [B, N, S] uint8: block_valid and j >= 1 (the anchor never counts)
 *   position_ids [B, N, S] int32: a + j, or -1 in an empty slot
 *   ctx_len      [B] int32, optional (NULL = not written): the largest anchor of a block of
 *                row b with at least one valid slot (0 if none) -- the number of context
 *                positions any block of the row reads; dflash_project_context takes it to
 *                skip the rest
 * Errors: INVALID_ARG for B, L, N or S < 1, null pointers, ws too small. */
DFLASH_API int dflash_plan(const uint8_t* mask, const int64_t* sample_ids, int B, int L, int64_t step,
                uint64_t seed, int num_anchors, int block_size, int32_t* anchors,
                uint8_t* block_valid, uint8_t* loss_mask, int32_t* position_ids,
                int32_t* ctx_len, void* ws, size_t ws_bytes, void* stream);

/* ---- 2. context projection ([P1] How it works: dual-source KV context) ---------------- */

DFLASH_API size_t dflash_project_context_workspace_size(const dflash_config_t* cfg, int B, int L);

/* Projects the target's selected hidden states into every draft layer's K/V space.
 *   target_hidden [B, L, n_tl*D_t]: the selected target layers concatenated in
 *                 target_layer_ids order, for context positions pos_offset .. pos_offset+L-1
 *   kv_cache      fp16 (bf16 configuration) or float32 (fp32 configuration), NL x B x 2 x Hkv
 *                 planes of L_cache*dh elements: for layer l,
 *                 row b, head g, plane (l, b, 0, g) = K as [L_cache][dh] with
 *                 K = RoPE(ctx W_k^T), and plane (l, b, 1, g) = V transposed, [dh][L_cache],
 *                 V = ctx W_v^T; ctx = RMSNorm(target_hidden W_proj^T; g_ctx), W_k / W_v =
 *                 the K / V rows of layer l's w_qkv.  Written at positions
 *                 pos_offset .. pos_offset+L-1 only; 16-byte aligned; in the bf16
 *                 configuration L_cache must be a multiple of 8.
 *   ctx_len       optional [B] int32 (NULL = L): positions c >= ctx_len[b] of row b may be
 *                 left unwritten (no block of that row reads them); values are clamped to [0, L].
 * Requires 0 <= pos_offset, pos_offset + L <= L_cache.  RoPE positions are the absolute
 * positions pos_offset + c.
 * Range: in the bf16 configuration the context and the cache are fp16.  A value outside
 * the fp16 range (or a NaN) sets DFLASH_ERR_RANGE in the sticky device status and is
 * stored as inf/NaN: the call itself still returns DFLASH_OK, so a caller that needs to
 * know polls dflash_device_status (which synchronizes the device).
 * Streams: with bf16 layer weights and few context rows (a per-layer K/V GEMM under eight
 * waves of CTA pairs) the K/V rows of every layer are converted to fp16 on a library-owned
 * stream of the calling host thread, beside the W_proj GEMM; events order that work after
 * what `stream` already holds and join it back before the call's last kernel, on every
 * return path, so every result is ordered on `stream` as for any other call. */
DFLASH_API int dflash_project_context(const dflash_config_t* cfg, const dflash_weights_t* w,
                           const void* target_hidden, int B, int L, int pos_offset, int L_cache,
                           const int32_t* ctx_len, void* kv_cache, void* ws, size_t ws_bytes,
                           void* stream);

/* ---- 2b. cache append after verification ([P3] One DFlash generation cycle: cache
 *      rollback) --------------------------------------------------------------------- */

DFLASH_API size_t dflash_append_context_workspace_size(const dflash_config_t* cfg, int B, int P,
                                                       int L_cache);

/* One inference cycle's cache update.  The target has verified one drafted block per
 * request and computed hidden states for its P positions (the anchor and the P - 1
 * proposals).  Only the verified prefix may stay in a cache: for request b the first
 *   n_b = accepted[b] + 1   (the anchor and the accepted proposals; accepted as written by
 *                            dflash_verify_greedy, clamped to [0, P - 1])
 * positions commit -- all P when accepted is NULL.  The rejected proposal and its suffix
 * never enter the cache; the target's replacement (or bonus) token has had no forward pass
 * and anchors the next block at position cache_len[b] + n_b.
 *   target_hidden [B, P, n_tl*D_t]: the verified block's selected target hidden states
 *   accepted      [B] int32 (device) or NULL
 *   cache_len     [B] int32 (device, in/out): committed length of each request's cache;
 *                 the n_b positions are projected exactly as dflash_project_context projects
 *                 a context (W_proj, RMSNorm, each layer's K/V with RoPE at the absolute
 *                 position) and written at cache positions cache_len[b] .. cache_len[b] +
 *                 n_b - 1; then cache_len[b] += n_b.  All on the device: no host round trip.
 *   kv_cache      the planes of dflash_project_context with L_cache positions per plane.
 * Positions at or past the new length keep what they held; a block anchored at
 * cache_len[b] never reads them.  A row whose cache_len is negative or would pass L_cache
 * commits nothing, keeps its length and sets DFLASH_ERR_DEVICE_CHECK.  The body then runs
 * with L = L_cache and a mask [B, L_cache] (positions below each request's length valid).
 * Range and streams: as for dflash_project_context. */
DFLASH_API int dflash_append_context(const dflash_config_t* cfg, const dflash_weights_t* w,
                                     const void* target_hidden, int B, int P,
                                     const int32_t* accepted, int32_t* cache_len, int L_cache,
                                     void* kv_cache, void* ws, size_t ws_bytes, void* stream);

/* ---- 3. draft body ([P2] How It Works, step 3; [P1] block-parallel prediction) -------- */

DFLASH_API size_t dflash_body_workspace_size(const dflash_config_t* cfg, int B, int L, int N);

/* Runs the draft decoder layers over B*N blocks of S slots.
 *   block_emb    [B, N, S, D] (dtype cfg->dtype): caller-supplied slot embeddings
 *   anchors      [B, N] int32 in [-1, L] (-1 = empty block)
 *   block_valid  [B, N, S] uint8
 *   position_ids [B, N, S] int32: RoPE position of each slot, in [0, L + S) for valid slots
 *   mask         [B, L] uint8: context validity
 *   kv_cache     the planes from dflash_project_context (L = its L_cache, a multiple of 8
 *                in the bf16 configuration); the
 *                positions a block reads (c < its anchor) must have been written; what the
 *                other positions hold never reaches an output
 *   out          [B, N, S, D] float32: one hidden state per slot; exactly 0 where
 *                block_valid == 0.
 * Attention of a valid slot of block (b, k) reads exactly: context positions c < anchors[b,k]
 * (c < L) with mask[b,c] != 0, and the valid slots of the same block (all of them, in both
 * directions).  It never reads another block and never writes kv_cache.
 * Layer: x += W_o Attn(RMSNorm(x; g_in)); x += W_down(SiLU(h W_gate^T) * h W_up^T),
 * h = RMSNorm(x; g_post); out = RMSNorm(x; g_final) when DFLASH_FLAG_FINAL_NORM.
 * A valid slot whose position id is out of range sets DFLASH_ERR_DEVICE_CHECK.
 * Range: in the bf16 configuration the layer projections' inputs, Q/K/V and the attention
 * output are fp16; a value outside the fp16 range sets DFLASH_ERR_RANGE in the sticky device
 * status while the call returns DFLASH_OK: poll dflash_device_status to learn of it.
 * Streams: with bf16 layer weights and more than 512 draft slots the fp16 copies of the layer
 * matrices are made in the workspace on a library-owned stream of the calling host thread,
 * one layer ahead of the layer that reads them; events order that work after what `stream`
 * already holds and before the layer that reads it (and joins it back on every return
 * path), so every result is ordered on `stream` as for any other call. */
DFLASH_API int dflash_body_forward(const dflash_config_t* cfg, const dflash_weights_t* w,
                        const void* block_emb, const int32_t* anchors,
                        const uint8_t* block_valid, const int32_t* position_ids,
                        const uint8_t* mask, const void* kv_cache, int B, int L, int N,
                        float* out, void* ws, size_t ws_bytes, void* stream);

/* ---- 3b. draft loss over the blocks ([P1] How it works: Loss; [P2] How It Works step 4;
 *      [P3] One DFlash generation cycle: greater weight on early positions) ------------- */

DFLASH_API size_t dflash_decayed_ce_workspace_size(int T, int D, int V);

/* The draft's training loss over T = B*N*S block slots: per slot t (slot j = t mod
 * block_size of its block), CE_t = logsumexp(logits_t) - logits_t[targets[t]] with
 * logits_t = hidden[t] lm_head^T over the V vocab entries; weights w_j = exp(-(j-1)/decay)
 * for j >= 1 (the pages fix the exponential decay toward later positions, not its scale:
 * decay is the caller's), 0 for the anchor; loss = sum(mask w CE) / sum(mask w), 0 when no
 * slot is weighted.
 *   hidden     [T, D] float32: dflash_body_forward's output (rounded to bf16 for the GEMM)
 *   lm_head    [V, D] bf16: the frozen target lm_head
 *   targets    [T] int32: the ground-truth token of each slot (read where the mask is set;
 *              outside [0, V) sets DFLASH_ERR_DEVICE_CHECK and the slot counts 0)
 *   loss_mask  [T] uint8: dflash_plan's loss_mask
 * Outputs: ce [T] float32 (0 outside the mask) and loss [1] float32, device.  The logits
 * are never stored: the lm_head GEMM's epilogue reduces each 128 x 256 tile to softmax
 * statistics.  Deterministic (fixed reduction orders).
 * Errors: INVALID_ARG for sizes < 1, T not a multiple of block_size, decay <= 0, null or
 * misaligned pointers; UNSUPPORTED for D not a multiple of 8. */
DFLASH_API int dflash_decayed_ce_loss(const float* hidden, const void* lm_head,
                                      const int32_t* targets, const uint8_t* loss_mask, int T,
                                      int block_size, int D, int V, double decay, float* ce,
                                      float* loss, void* ws, size_t ws_bytes, void* stream);

/* ---- 4. greedy verification ([P3] One DFlash generation cycle) ----------------------- */

DFLASH_API size_t dflash_verify_workspace_size(int B, int gamma, int V);

/* Greedy block verification of B drafted blocks.
 *   logits  [B, gamma+1, V] of type logits_dtype (DFLASH_DTYPE_BF16 or _F32): row i is the
 *           target's distribution after the anchor and draft[0..i-1]; row gamma gives the bonus
 *   draft   [B, gamma] int32 proposed tokens
 *   eos     EOS token id, or -1 for none: a matching EOS proposal ends the block (no bonus)
 * target choice i = argmax over V of logits row i (exact comparison, lowest index on ties).
 * Outputs: emitted [B, gamma+1] int32 (the accepted proposals, then the target's choice at
 * the first mismatch or the bonus, padded with -1); num_emitted [B]; accepted [B];
 * target_choices [B, gamma+1] (optional, may be NULL).
 * Errors: INVALID_ARG for gamma < 0, V < 1, B < 1 (the length rule of the page's
 * verification: one target choice per draft token plus the bonus). */
DFLASH_API int dflash_verify_greedy(const void* logits, int logits_dtype, const int32_t* draft, int B,
                         int gamma, int V, int32_t eos, int32_t* emitted, int32_t* num_emitted,
                         int32_t* accepted, int32_t* target_choices, void* ws, size_t ws_bytes,
                         void* stream);

/* ---- 4b. speculative-sampling verification ([P3] Sampling with temperature is not argmax
 *      matching) ------------------------------------------------------------------------ */

DFLASH_API size_t dflash_verify_sampling_workspace_size(int B, int gamma, int V);

/* Speculative-sampling verification of B drafted blocks: the target distribution of row i is
 * p_i = softmax(logits[b, i] / temperature); q_i = draft_probs[b, i] is the ACTUAL proposal
 * distribution draft[b, i] was drawn from (after any top-k, temperature or selector on the
 * draft side).  In block order, proposal y = draft[b, i] is accepted when
 * U(seed, b, i, 0) < p_i(y) / q_i(y) -- probability min(1, p/q); at the first rejection the
 * block ends with a sample of the normalised residual [p_i - q_i]_+.  If every proposal is
 * accepted the block ends with a sample of p_gamma.  A matched EOS proposal ends the block
 * (no sample).  The output tokens are distributed as the target's own samples.
 *   logits       [B, gamma+1, V] of type logits_dtype (DFLASH_DTYPE_BF16 or _F32)
 *   temperature  > 0 (host double)
 *   draft_probs  [B, gamma, V] float32, rows summing to 1 (only the entries of the draft
 *                tokens and the rejected row are read)
 *   draft        [B, gamma] int32 in [0, V) (an entry outside sets DFLASH_ERR_DEVICE_CHECK)
 *   seed         the sampling stream: U(seed, counters...) is the SplitMix64 finaliser
 *                chained over the seed and the counters, top 23 bits + 1/2 times 2^-23;
 *                samples use the exponential race (index v arrives at -ln U(seed, b, i, 1,
 *                v) / w_v; the first arrival wins, lowest index on a tie), an exact draw
 *                from w / sum(w).  Same seed, same inputs: same outputs.
 * Outputs as dflash_verify_greedy: emitted [B, gamma+1] (accepted proposals, then the
 * sample; -1 padded), num_emitted [B], accepted [B].  The probabilities are fp32; a
 * decision within fp32 rounding of its threshold may come out either way.
 * Errors: INVALID_ARG for B < 1, gamma < 0, V < 1, temperature <= 0, null pointers. */
DFLASH_API int dflash_verify_sampling(const void* logits, int logits_dtype, double temperature,
                                      const float* draft_probs, const int32_t* draft, int B,
                                      int gamma, int V, uint64_t seed, int32_t eos,
                                      int32_t* emitted, int32_t* num_emitted, int32_t* accepted,
                                      void* ws, size_t ws_bytes, void* stream);

/* ---- greedy verification without a workspace ----------------------------------------
 * The pages have no counterpart for this call: it is a deployment variant of
 * dflash_verify_greedy for callers that cannot allocate device memory -- code embedded in
 * a host framework that owns the whole device memory pool and forbids side allocations,
 * or a latency-critical loop that must never call cudaMalloc/cudaFree (both may
 * synchronize the device).  Same arguments, outputs and errors as dflash_verify_greedy,
 * minus the workspace: the scratch lives in a fixed 128 KiB array inside this library's
 * device memory, held by every GPU that loads the library until the process exits.
 *  - Limit: B * (gamma + 1) <= 16384; larger requests return DFLASH_ERR_INVALID_ARG with a
 *    message (use dflash_verify_greedy with a workspace instead).
 *  - The first call on each device (with that device current) looks up the array's device
 *    address; make that first call before any stream capture on that device.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *  - Every call on a device shares the one array and no call needs it zeroed (each call
 *    writes every entry it reads).  Calls whose kernels overlap on the GPU (different
 *    streams, or host threads racing on one device) race on the array: serialize them. */
DFLASH_API int dflash_verify_greedy_static(const void* logits, int logits_dtype,
                                           const int32_t* draft, int B, int gamma, int V,
                                           int32_t eos, int32_t* emitted, int32_t* num_emitted,
                                           int32_t* accepted, int32_t* target_choices,
                                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H_ */

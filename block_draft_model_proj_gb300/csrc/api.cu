// C ABI of libdflash: argument checks, workspace layout and the launch sequence of each call.
// The operations and their sources are documented in include/dflash.h.
#include <math.h>
#include <stdarg.h>

#include <atomic>
#include <mutex>
#include <vector>
#include <stdio.h>
#include <string.h>

#include "../../include/dflash.h"
#include "../../include/dflash_testing.h"
#include "common.cuh"
#include "internal.h"

namespace dflash {

__device__ unsigned g_device_status;

namespace {

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(DFLASH_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define DF_CUDA(expr)                                   \
  do {                                                  \
    cudaError_t e_ = (expr);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #expr); \
  } while (0)

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};

// Address of this device's status word (looked up once per device).
unsigned* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

// ---- launch counting and optional event timing ----------------------------------------
std::atomic<long> g_launches{0};
std::mutex g_prof_mu;
bool g_prof_on = false;
struct ProfRec {
  int kind;
  int count;
  cudaEvent_t a, b;
};
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Brackets the kernel launches of one step; `count` = kernels launched inside.
class Prof {
 public:
  Prof(int kind, int count, cudaStream_t s) : kind_(kind), count_(count), s_(s) {
    g_launches += count;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (g_prof_on) {
      a_ = take_event();
      b_ = take_event();
      cudaEventRecord(a_, s_);
    }
  }
  ~Prof() {
    if (!a_) return;
    cudaEventRecord(b_, s_);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back({kind_, count_, a_, b_});
  }

 private:
  int kind_, count_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

int num_sms() {
  static int cached[kMaxDevices] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

// A side stream of the calling host thread on the current device, with the events that fork
// work onto it and join it back (per thread, so concurrent callers never share events).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr;
  cudaEvent_t done[2] = {nullptr, nullptr};
};

cudaError_t side_stream(SideStream** out) {
  thread_local SideStream per_dev[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  SideStream& ss = per_dev[dev];
  if (!ss.s) {
    if ((e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
    for (int i = 0; i < 2; ++i)
      if ((e = cudaEventCreateWithFlags(&ss.done[i], cudaEventDisableTiming)) != cudaSuccess)
        return e;
  }
  *out = &ss;
  return cudaSuccess;
}

// Joins the side stream back into `s` when the scope ends on a path that has not joined it
// itself (an early error return): no work of the call is left behind on the side stream
// unordered with the caller's stream.  The normal paths join explicitly and set `joined`, so
// no extra cross-stream wait sits between two kernels of `s` (it would stop the next kernel's
// programmatic early launch).
struct SideJoin {
  cudaStream_t s;
  SideStream* const* side;
  bool joined = false;
  ~SideJoin() {
    if (*side && !joined) {
      cudaEventRecord((*side)->done[0], (*side)->s);
      cudaStreamWaitEvent(s, (*side)->done[0], 0);
    }
  }
};

// ---- workspace carving -----------------------------------------------------------------
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    off = (off + 255) & ~(size_t)255;
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

size_t esize(int dtype) { return dtype == DFLASH_DTYPE_BF16 ? 2 : 4; }

struct Act;

// K-split used for a GEMM of this shape: enough tiles to cover the SMs, at least 4 K-steps
// of 64 per split, at most 8 splits; never an empty split.
int gemm_splits(long M, int N, int K) {
  const long tiles = ((M + 127) / 128) * ((N + 255) / 256);
  const int sms = num_sms();
  const int kb = (K + 63) / 64;
  int s = 1;
  while (s < 8 && tiles * s < sms && kb / (2 * s) >= 4) s *= 2;
  const int per = (kb + s - 1) / s;
  return (kb + per - 1) / per;
}

int check_cfg(const dflash_config_t* c) {
  if (!c) return fail(DFLASH_ERR_INVALID_ARG, "cfg is null");
  if (c->dtype != DFLASH_DTYPE_BF16 && c->dtype != DFLASH_DTYPE_F32)
    return fail(DFLASH_ERR_INVALID_ARG, "cfg->dtype must be DFLASH_DTYPE_BF16 or DFLASH_DTYPE_F32");
  if (c->target_hidden < 1 || c->num_target_layers < 1 || c->hidden < 1 || c->num_layers < 1 ||
      c->num_heads < 1 || c->num_kv_heads < 1 || c->head_dim < 2 || c->intermediate < 1 ||
      c->block_size < 1)
    return fail(DFLASH_ERR_INVALID_ARG, "cfg sizes must be positive");
  if (c->num_heads % c->num_kv_heads != 0)
    return fail(DFLASH_ERR_INVALID_ARG, "num_heads (%d) must be a multiple of num_kv_heads (%d)",
                c->num_heads, c->num_kv_heads);
  if (c->head_dim % 2 != 0) return fail(DFLASH_ERR_INVALID_ARG, "head_dim must be even");
  if (c->head_dim % 8 != 0)
    return fail(DFLASH_ERR_UNSUPPORTED, "head_dim must be a multiple of 8 (vectorised RoPE)");
  if (!(c->rope_theta > 0.0) || !(c->rms_eps >= 0.0))
    return fail(DFLASH_ERR_INVALID_ARG, "rope_theta must be > 0 and rms_eps >= 0");
  if ((c->flags & ~(DFLASH_FLAG_FINAL_NORM | DFLASH_FLAG_CTX_NORM | DFLASH_FLAG_F16_LAYERS)) != 0)
    return fail(DFLASH_ERR_INVALID_ARG, "unknown bits in cfg->flags");
  if ((c->flags & DFLASH_FLAG_F16_LAYERS) && c->dtype != DFLASH_DTYPE_BF16)
    return fail(DFLASH_ERR_INVALID_ARG, "DFLASH_FLAG_F16_LAYERS needs the bf16 configuration");
  if (c->dtype == DFLASH_DTYPE_BF16) {
    const long widths[] = {(long)c->target_hidden * c->num_target_layers, c->hidden,
                           (long)c->num_heads * c->head_dim, c->intermediate};
    for (long w : widths)
      if (w % 8 != 0)
        return fail(DFLASH_ERR_UNSUPPORTED,
                    "bf16 path needs every matrix row width to be a multiple of 8 elements "
                    "(16-byte rows for TMA); got %ld", w);
  }
  const int grp = c->num_heads / c->num_kv_heads;
  if ((long)c->block_size * grp > 128 || c->head_dim > 256)
    return fail(DFLASH_ERR_UNSUPPORTED, "block_size * num_heads/num_kv_heads must be <= 128 and "
                "head_dim <= 256");
  if (c->dtype == DFLASH_DTYPE_BF16 &&
      !attention_tc_supported(c->block_size, c->num_heads, c->num_kv_heads, c->head_dim))
    return fail(DFLASH_ERR_UNSUPPORTED, "bf16 attention needs head_dim == 128, "
                "block_size * num_heads/num_kv_heads dividing 128 and num_heads/num_kv_heads "
                "dividing 16");
  return DFLASH_OK;
}

// Tensor arguments are read and written with 16-byte vector accesses (and TMA).
int check_ptr16(const void* p, const char* what, int dtype) {
  (void)dtype;
  if (!p) return fail(DFLASH_ERR_INVALID_ARG, "%s is null", what);
  if (((uintptr_t)p % 16) != 0)
    return fail(DFLASH_ERR_INVALID_ARG, "%s must be 16-byte aligned", what);
  return DFLASH_OK;
}

int check_weights(const dflash_config_t* c, const dflash_weights_t* w, bool need_layers_body) {
  if (!w) return fail(DFLASH_ERR_INVALID_ARG, "weights is null");
  if (w->num_layers != c->num_layers || !w->layers)
    return fail(DFLASH_ERR_INVALID_ARG, "weights->layers must hold cfg->num_layers entries");
  int r;
  if ((r = check_ptr16(w->w_proj, "w_proj", c->dtype))) return r;
  if ((r = check_ptr16(w->g_ctx, "g_ctx", DFLASH_DTYPE_F32))) return r;
  if ((r = check_ptr16(w->g_final, "g_final", DFLASH_DTYPE_F32))) return r;
  for (int l = 0; l < c->num_layers; ++l) {
    const dflash_layer_weights_t& lw = w->layers[l];
    if ((r = check_ptr16(lw.w_qkv, "w_qkv", c->dtype))) return r;
    if (need_layers_body) {
      if ((r = check_ptr16(lw.w_o, "w_o", c->dtype))) return r;
      if ((r = check_ptr16(lw.w_gate_up, "w_gate_up", c->dtype))) return r;
      if ((r = check_ptr16(lw.w_down, "w_down", c->dtype))) return r;
      if ((r = check_ptr16(lw.g_in, "g_in", DFLASH_DTYPE_F32))) return r;
      if ((r = check_ptr16(lw.g_post, "g_post", DFLASH_DTYPE_F32))) return r;
    }
  }
  return DFLASH_OK;
}

int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (need > ws_bytes) return fail(DFLASH_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  if (need > 0 && !ws) return fail(DFLASH_ERR_INVALID_ARG, "workspace is null");
  if ((uintptr_t)ws % 256 != 0) return fail(DFLASH_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  return DFLASH_OK;
}

// C[z] = A * B^T (fp32 out): tcgen05 for 16-bit operands (elem bf16 or fp16), CUDA cores
// for the fp32 configuration.
cudaError_t gemm(int dtype, int elem, const void* A, long lda, const void* Bm, long ldb, float* C,
                 long ldc, long M, int N, int K, int splits, cudaStream_t s,
                 const int32_t* tile_list = nullptr, int* splits_out = nullptr) {
  if (dtype == DFLASH_DTYPE_BF16)
    return launch_gemm_tc(elem, A, lda, Bm, ldb, C, ldc, M, N, K, splits, tile_list,
                          status_ptr(), s, splits_out);
  return launch_gemm_simt(dtype, A, lda, Bm, ldb, C, ldc, M, N, K, splits, s);
}

// A computed activation buffer: fp32 (fp32 configuration) or fp16 (bf16 configuration).
struct Act {
  void* p = nullptr;
  int dtype = DFLASH_DTYPE_F32;
  ActOut out() const {
    ActOut o;
    o.p = p;
    o.dtype = dtype;
    o.status = status_ptr();
    return o;
  }
};

Act take_act(Carver& cv, size_t n, int dtype) {
  Act a;
  a.dtype = dtype;
  if (dtype == DFLASH_DTYPE_BF16)
    a.p = cv.take<__half>(n);
  else
    a.p = cv.take<float>(n);
  return a;
}

// Element type of the draft layers' projection matrices in the bf16 configuration, as the
// caller gives them: bf16, or fp16 under DFLASH_FLAG_F16_LAYERS.
int layer_wdtype(const dflash_config_t* c) {
  return (c->flags & DFLASH_FLAG_F16_LAYERS) ? DFLASH_DTYPE_F16 : DFLASH_DTYPE_BF16;
}

// Which GEMM runs the layer projections of a call with `tokens` rows.  The weight-streaming
// GEMM reads the weights as given (bf16 tiles converted on chip); the 128 x 256-tile GEMM
// is faster per FLOP from a few hundred tokens up but takes fp16 weights (the caller's,
// or copies converted at the start of the call, one extra read and write of every matrix).
// Up to 128 tokens the weight-streaming GEMM is faster outright; up to 512 it is cheaper
// than converting bf16 weights; above that the conversion pays for itself.
bool layer_gemm_ws(const dflash_config_t* c, long tokens) {
  if (c->dtype != DFLASH_DTYPE_BF16) return false;
  if (tokens <= 128) return true;
  return layer_wdtype(c) == DFLASH_DTYPE_BF16 && tokens <= 512;
}

// fp16 copies of the layer matrices are made inside the call (bf16 weights, large calls)
bool convert_layers(const dflash_config_t* c, long tokens) {
  return c->dtype == DFLASH_DTYPE_BF16 && layer_wdtype(c) == DFLASH_DTYPE_BF16 &&
         !layer_gemm_ws(c, tokens);
}

// The context K/V projection (dflash_project_context) reads fp16 layer weights: bf16 ones
// are converted inside the call, independently of how the body dispatches its projections.
bool context_kv_needs_convert(const dflash_config_t* c) {
  return c->dtype == DFLASH_DTYPE_BF16 && layer_wdtype(c) == DFLASH_DTYPE_BF16;
}

// Upper bound for a device-chosen K-split: about three waves of output tiles (tile_n
// columns x 128 rows) when every row tile is active, at most 8.
int ws_max_splits(int Nw, long T, int tile_n = 128) {
  const long units = (long)((Nw + tile_n - 1) / tile_n) * ((T + 127) / 128);
  long s = (3L * num_sms() + units - 1) / units;
  return (int)(s < 1 ? 1 : (s > 8 ? 8 : s));
}

struct ProjLayout {
  float* y;
  Act ctx;
  __half* wkv16;  // the K/V rows of w_qkv as fp16 (converted in the call), or null: every
                  // layer's, stacked, when kv_merged, else one layer's
  bool kv_merged;  // one K/V GEMM over all layers (N = NL * 2*Hkv*dh) instead of one per layer
  float* cos_t;
  float* sin_t;
  int32_t* tile_list;
  int32_t* n_commit;  // append: positions each row commits
  int32_t* start;     // append: each row's first cache position
  int split_proj, split_kv;
  size_t bytes;
};

// rope_rows: positions of the RoPE table (L for a projection at one offset; the cache
// length for an append at per-row offsets, whose table starts at position 0).
// append: also carve the per-row commit counts and start positions.
ProjLayout proj_layout(const dflash_config_t* c, int B, int L, void* ws, int rope_rows = -1,
                       bool append = false) {
  ProjLayout p;
  if (rope_rows < 0) rope_rows = L;
  const long M = (long)B * L;
  const int D = c->hidden, Kc = c->target_hidden * c->num_target_layers;
  const int kvw = 2 * c->num_kv_heads * c->head_dim;
  p.split_proj = gemm_splits(M, D, Kc);
  p.split_kv = c->dtype == DFLASH_DTYPE_BF16 ? 1 : gemm_splits(M, kvw, D);
  const long ycols = (long)p.split_proj * D > (long)p.split_kv * kvw ? (long)p.split_proj * D
                                                                       : (long)p.split_kv * kvw;
  Carver cv(ws);
  p.y = cv.take<float>((size_t)M * ycols);
  p.ctx = take_act(cv, (size_t)M * D, c->dtype);
  p.cos_t = cv.take<float>((size_t)rope_rows * (c->head_dim / 2));
  p.sin_t = cv.take<float>((size_t)rope_rows * (c->head_dim / 2));
  p.tile_list = cv.take<int32_t>(1 + (size_t)(M + kGemmTileM - 1) / kGemmTileM);
  p.n_commit = append ? cv.take<int32_t>(B) : nullptr;
  p.start = append ? cv.take<int32_t>(B) : nullptr;
  // the context K/V projection always runs on the 128 x 256-tile GEMM with fp16 operands:
  // bf16 layer weights are converted into the workspace whatever the row count.  When one
  // layer's GEMM would fill fewer than eight waves of CTA pairs, the converted rows of every
  // layer are stacked and projected by one GEMM: the context rows are read once and the
  // waves come out even.
  const long pair_units = ((M + 255) / 256) * ((kvw + 255) / 256);
  p.kv_merged = context_kv_needs_convert(c) && c->num_layers > 1 &&
                pair_units < 8L * (num_sms() / 2);
  p.wkv16 = context_kv_needs_convert(c)
                ? cv.take<__half>((size_t)kvw * D * (p.kv_merged ? c->num_layers : 1))
                : nullptr;
  p.bytes = cv.off;
  return p;
}

// The projection of rows m = b*L + c of target_hidden into every layer's cache planes at
// positions (row_pos0 ? row_pos0[b] : pos_offset) + c, rows c >= ctx_len[b] skipped (the
// RoPE table of `lay` is already built, and with it the list of 128-row tiles holding a row
// c < ctx_len[b], `flags`, or null: every tile).
int project_rows(const dflash_config_t* cfg, const dflash_weights_t* w, const void* target_hidden,
                 int B, int L, int pos_offset, int L_cache, const int32_t* ctx_len,
                 const int32_t* row_pos0, void* kv_cache, const ProjLayout& lay, cudaStream_t s,
                 const int32_t* flags) {
  const long M = (long)B * L;
  const int D = cfg->hidden, Kc = cfg->target_hidden * cfg->num_target_layers;
  const int dh = cfg->head_dim, Hkv = cfg->num_kv_heads, qw = cfg->num_heads * dh;
  const int kvw = 2 * Hkv * dh;
  const size_t es = esize(cfg->dtype);
  // Stacked K/V rows: their conversion (HBM-bound, independent of the context) runs on a side
  // stream of this thread beside the tensor-bound W_proj GEMM; it starts after everything
  // already on `s` (the previous reader of the buffer) and is joined before the K/V GEMM.
  SideStream* side = nullptr;
  SideJoin join{s, &side};
  if (lay.kv_merged) {
    DF_CUDA(side_stream(&side));
    DF_CUDA(cudaEventRecord(side->fork, s));
    DF_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
    {
      Prof pc(DFLASH_PROF_CONVERT, cfg->num_layers, side->s);
      for (int l = 0; l < cfg->num_layers; ++l) {
        const void* wkv = static_cast<const uint8_t*>(w->layers[l].w_qkv) + (size_t)qw * D * es;
        DF_CUDA(launch_convert_bf16_f16(wkv, lay.wkv16 + (size_t)l * kvw * D, (size_t)kvw * D,
                                        status_ptr(), side->s));
      }
    }
    DF_CUDA(cudaEventRecord(side->done[0], side->s));
  }
  {
    Prof pr(DFLASH_PROF_GEMM, 1, s);
    DF_CUDA(gemm(cfg->dtype, DFLASH_DTYPE_BF16, target_hidden, Kc, w->w_proj, Kc, lay.y, D, M, D,
                 Kc, lay.split_proj, s, flags));
  }
  {
    Prof pr(DFLASH_PROF_ROWS, 1, s);
    DF_CUDA(launch_rows_norm(cfg->dtype, lay.y, lay.split_proj, w->g_ctx, cfg->rms_eps,
                             (cfg->flags & DFLASH_FLAG_CTX_NORM) != 0, lay.ctx.out(), M, D,
                             ctx_len, L, s));
  }
  const size_t layer_elems = (size_t)B * 2 * Hkv * L_cache * dh;
  auto kv_epilogue = [&](int l0, int layers) {
    KvCacheEpilogue kv;
    kv.kv = static_cast<__half*>(kv_cache) + (size_t)l0 * layer_elems;
    kv.cos_t = lay.cos_t;
    kv.sin_t = lay.sin_t;
    kv.ctx_len = ctx_len;
    kv.row_pos0 = row_pos0;
    kv.L = L;
    kv.pos_offset = pos_offset;
    kv.L_cache = L_cache;
    kv.Hkv = Hkv;
    kv.layers = layers;
    kv.layer_elems = (long)layer_elems;
    return kv;
  };
  if (lay.kv_merged) {
    // every layer's K/V rows, converted and stacked (joined from the side stream): one GEMM,
    // RoPE and the fp16 cache layout in its epilogue
    DF_CUDA(cudaStreamWaitEvent(s, side->done[0], 0));
    join.joined = true;
    Prof pr(DFLASH_PROF_GEMM, 1, s);
    DF_CUDA(launch_gemm_tc_kv_cache(DFLASH_DTYPE_F16, lay.ctx.p, D, lay.wkv16, D, M,
                                    cfg->num_layers * kvw, D, flags,
                                    kv_epilogue(0, cfg->num_layers), status_ptr(), s));
    return DFLASH_OK;
  }
  for (int l = 0; l < cfg->num_layers; ++l) {
    const void* wkv = static_cast<const uint8_t*>(w->layers[l].w_qkv) + (size_t)qw * D * es;
    if (cfg->dtype == DFLASH_DTYPE_BF16) {
      // RoPE and the fp16 cache layout are applied in the GEMM epilogue
      const KvCacheEpilogue kv = kv_epilogue(l, 1);
      const void* wkv16 = wkv;
      if (lay.wkv16) {
        Prof pc(DFLASH_PROF_CONVERT, 1, s);
        DF_CUDA(launch_convert_bf16_f16(wkv, lay.wkv16, (size_t)kvw * D, status_ptr(), s));
        wkv16 = lay.wkv16;
      }
      Prof pr(DFLASH_PROF_GEMM, 1, s);
      DF_CUDA(launch_gemm_tc_kv_cache(DFLASH_DTYPE_F16, lay.ctx.p, D, wkv16, D, M, kvw, D, flags,
                                      kv, status_ptr(), s));
      continue;
    }
    {
      Prof pr(DFLASH_PROF_GEMM, 1, s);
      DF_CUDA(gemm(cfg->dtype, DFLASH_DTYPE_F16, lay.ctx.p, D, wkv, D, lay.y, kvw, M, kvw, D,
                   lay.split_kv, s, flags));
    }
    Prof pr(DFLASH_PROF_ROWS, 2, s);
    DF_CUDA(launch_ctx_kv_scatter(lay.y, lay.split_kv, lay.cos_t, lay.sin_t,
                                  static_cast<float*>(kv_cache) + (size_t)l * layer_elems, B, L,
                                  pos_offset, L_cache, Hkv, dh, ctx_len, row_pos0, s));
  }
  return DFLASH_OK;
}

struct BodyLayout {
  float* x;
  Act h, attn, act;
  void *q, *kb, *vbt;   // attention-ready operands (fp16 in the bf16 configuration, else fp32)
  int ns_pad;
  float* partials;      // tensor-core attention partials (bf16 configuration)
  int32_t* tile_list;   // 128-slot tiles holding at least one valid slot (count first)
  float* y;
  float* cos_t;
  float* sin_t;
  bool ws;              // layer projections on the weight-streaming GEMM (few tokens)
  int* nsplit;          // weight-streaming GEMM: K-splits chosen on the device (QKV, O, down)
  __half* wl16;         // fp16 copies of the layer matrices converted in the call, or null:
                        // two layers' buffers (layer l in buffer l % 2) when NL > 1
  size_t wl16_layer;    // elements of one layer's four matrices
  int sp_qkv, sp_o, sp_gu, sp_down;  // host K-splits, or the device upper bounds
  // 128 x 256 GEMM without a K-split: Q/K RoPE and the attention layouts in the QKV
  // epilogue, the residual add in the O and down epilogues
  bool fuse_qkv, fuse_o, fuse_down;
  int P;
  size_t bytes;
};

// Testing override of the fused-epilogue choice: 0 = by the split bound, 1 = always (on the
// 128 x 256 GEMM), 2 = never.
std::atomic<int> g_fused_mode{0};

BodyLayout body_layout(const dflash_config_t* c, int B, int L, int N, void* ws) {
  BodyLayout b;
  const long T = (long)B * N * c->block_size;
  const int D = c->hidden, qw = c->num_heads * c->head_dim, kw = c->num_kv_heads * c->head_dim;
  const int qkvw = qw + 2 * kw, I = c->intermediate;
  b.ws = layer_gemm_ws(c, T);
  if (b.ws) {
    b.sp_qkv = ws_max_splits(qkvw, T);
    b.sp_o = ws_max_splits(D, T);
    // up to 128 tokens gate/up is K-split (fp32 slices + the SwiGLU row kernel); above that
    // SiLU(gate) * up is formed in the GEMM epilogue
    b.sp_gu = T <= 128 ? ws_max_splits(2 * I, T) : 0;
    b.sp_down = ws_max_splits(D, T);
  } else if (c->dtype == DFLASH_DTYPE_BF16) {  // splits chosen on the device, these bound them
    b.sp_qkv = ws_max_splits(qkvw, T, 256);
    b.sp_o = ws_max_splits(D, T, 256);
    b.sp_gu = 0;
    b.sp_down = ws_max_splits(D, T, 256);
  } else {
    b.sp_qkv = gemm_splits(T, qkvw, D);
    b.sp_o = gemm_splits(T, D, qw);
    b.sp_gu = gemm_splits(T, 2 * I, D);
    b.sp_down = gemm_splits(T, D, I);
  }
  // Enough output tiles for three waves without a K-split (bound 1): the epilogues write
  // the attention operands / add into the residual stream directly, and the row passes that
  // would read fp32 slices drop out.
  const int fm = g_fused_mode.load();
  const bool tc_path = c->dtype == DFLASH_DTYPE_BF16 && !b.ws && fm != 2;
  b.fuse_qkv = tc_path && (fm == 1 || b.sp_qkv == 1);
  b.fuse_o = tc_path && (fm == 1 || b.sp_o == 1);
  b.fuse_down = tc_path && (fm == 1 || b.sp_down == 1);
  long ycols = (long)b.sp_qkv * qkvw;
  if ((long)b.sp_o * D > ycols) ycols = (long)b.sp_o * D;
  if ((long)b.sp_gu * 2 * I > ycols) ycols = (long)b.sp_gu * 2 * I;
  if ((long)b.sp_down * D > ycols) ycols = (long)b.sp_down * D;
  Carver cv(ws);
  b.x = cv.take<float>((size_t)T * D);
  b.h = take_act(cv, (size_t)T * D, c->dtype);
  b.ns_pad = (N * c->block_size + 7) / 8 * 8;
  const size_t nvbt = (size_t)B * c->num_kv_heads * c->head_dim * b.ns_pad;
  if (c->dtype == DFLASH_DTYPE_BF16) {
    b.q = cv.take<__half>((size_t)T * qw);
    b.kb = cv.take<__half>((size_t)T * kw);
    b.vbt = cv.take<__half>(nvbt);
  } else {
    b.q = cv.take<float>((size_t)T * qw);
    b.kb = cv.take<float>((size_t)T * kw);
    b.vbt = cv.take<float>(nvbt);
  }
  b.partials = nullptr;
  if (c->dtype == DFLASH_DTYPE_BF16)
    b.partials = cv.take<float>((size_t)attention_tc_layout(B, N, c->block_size, L, c->num_heads,
                                                            c->num_kv_heads, num_sms())
                                    .part_floats);
  b.attn = take_act(cv, (size_t)T * qw, c->dtype);
  b.act = take_act(cv, (size_t)T * I, c->dtype);
  b.y = cv.take<float>((size_t)T * ycols);
  b.tile_list = cv.take<int32_t>(1 + (size_t)(T + kGemmTileM - 1) / kGemmTileM);
  b.P = L + c->block_size;
  b.cos_t = cv.take<float>((size_t)b.P * (c->head_dim / 2));
  b.sin_t = cv.take<float>((size_t)b.P * (c->head_dim / 2));
  b.nsplit = cv.take<int>(4);
  b.wl16_layer = (size_t)qkvw * D + (size_t)D * qw + (size_t)2 * I * D + (size_t)D * I;
  b.wl16 = convert_layers(c, T)
               ? cv.take<__half>(b.wl16_layer * (c->num_layers > 1 ? 2 : 1))
               : nullptr;
  b.bytes = cv.off;
  return b;
}

}  // namespace

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

}  // namespace dflash

using namespace dflash;

extern "C" {

const char* dflash_last_error(void) { return g_msg; }

int dflash_version(void) { return 200; }

int dflash_convert_bf16_to_f16(const void* src, void* dst, size_t n, void* stream) {
  if (n == 0) return DFLASH_OK;
  int r;
  if ((r = check_ptr16(src, "src", DFLASH_DTYPE_BF16))) return r;
  if ((r = check_ptr16(dst, "dst", DFLASH_DTYPE_F16))) return r;
  Prof pr(DFLASH_PROF_CONVERT, 1, (cudaStream_t)stream);
  DF_CUDA(launch_convert_bf16_f16(src, dst, n, status_ptr(), (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_device_status(int reset) {
  unsigned* p = status_ptr();
  if (!p) return fail(DFLASH_ERR_CUDA, "no CUDA device");
  DF_CUDA(cudaDeviceSynchronize());
  unsigned v = 0;
  DF_CUDA(cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost));
  if (reset) DF_CUDA(cudaMemset(p, 0, sizeof(unsigned)));
  if (v & kStatusTimeout) return fail(DFLASH_ERR_TIMEOUT, "device wait timed out (kernel id %u)", (v >> 8) & 0xFF);
  if (v & kStatusCheck) return fail(DFLASH_ERR_DEVICE_CHECK, "device index check failed (kernel id %u)", (v >> 8) & 0xFF);
  if (v & kStatusRange)
    return fail(DFLASH_ERR_RANGE, "a value outside the fp16 range was stored as fp16 (kernel id %u)",
                (v >> 8) & 0xFF);
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------------------
size_t dflash_plan_workspace_size(int, int, int, int) { return 0; }

int dflash_plan(const uint8_t* mask, const int64_t* sample_ids, int B, int L, int64_t step,
                uint64_t seed, int num_anchors, int block_size, int32_t* anchors,
                uint8_t* block_valid, uint8_t* loss_mask, int32_t* position_ids,
                int32_t* ctx_len, void* ws, size_t ws_bytes, void* stream) {
  if (B < 1 || L < 1 || num_anchors < 1 || block_size < 1)
    return fail(DFLASH_ERR_INVALID_ARG, "B, L, num_anchors and block_size must be >= 1");
  if (num_anchors > 1024) return fail(DFLASH_ERR_UNSUPPORTED, "num_anchors must be <= 1024");
  if (!mask || !sample_ids || !anchors || !block_valid || !loss_mask || !position_ids)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  (void)ws;
  (void)ws_bytes;
  {
    Prof pr(DFLASH_PROF_PLAN, 1, (cudaStream_t)stream);
    DF_CUDA(launch_plan(mask, sample_ids, B, L, (uint64_t)step, seed, num_anchors, block_size,
                        anchors, block_valid, loss_mask, position_ids, ctx_len,
                        (cudaStream_t)stream));
  }
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------------------
size_t dflash_project_context_workspace_size(const dflash_config_t* cfg, int B, int L) {
  if (check_cfg(cfg) != DFLASH_OK || B < 1 || L < 1) return 0;
  return proj_layout(cfg, B, L, nullptr).bytes;
}

int dflash_project_context(const dflash_config_t* cfg, const dflash_weights_t* w,
                           const void* target_hidden, int B, int L, int pos_offset, int L_cache,
                           const int32_t* ctx_len, void* kv_cache, void* ws, size_t ws_bytes,
                           void* stream) {
  int r;
  if ((r = check_cfg(cfg))) return r;
  if ((r = check_weights(cfg, w, false))) return r;
  if (B < 1 || L < 1 || pos_offset < 0 || (long)pos_offset + L > L_cache)
    return fail(DFLASH_ERR_INVALID_ARG, "need B, L >= 1 and 0 <= pos_offset, pos_offset + L <= L_cache");
  if ((r = check_ptr16(target_hidden, "target_hidden", cfg->dtype))) return r;
  if ((r = check_ptr16(kv_cache, "kv_cache", DFLASH_DTYPE_BF16))) return r;
  if (cfg->dtype == DFLASH_DTYPE_BF16 && L_cache % 8 != 0)
    return fail(DFLASH_ERR_INVALID_ARG, "L_cache must be a multiple of 8 (16-byte fp16 cache rows)");
  const ProjLayout lay = proj_layout(cfg, B, L, ws);
  if ((r = check_ws(ws, ws_bytes, lay.bytes))) return r;
  cudaStream_t s = (cudaStream_t)stream;
  // 128-row tiles no block reads (all c >= ctx_len[b]) are skipped by every projection; their
  // list is built by one block of the RoPE-table launch
  TileJob tj;
  if (ctx_len && cfg->dtype == DFLASH_DTYPE_BF16) {
    tj.kind = TileJob::kContext;
    tj.ctx_len = ctx_len;
    tj.B = B;
    tj.L = L;
    tj.list = lay.tile_list;
  }
  {
    Prof pr(DFLASH_PROF_ROWS, 1, s);
    DF_CUDA(launch_rope_table(lay.cos_t, lay.sin_t, pos_offset, L, cfg->head_dim,
                              cfg->rope_theta, s, tj));
  }
  return project_rows(cfg, w, target_hidden, B, L, pos_offset, L_cache, ctx_len, nullptr,
                      kv_cache, lay, s, tj.kind != TileJob::kNone ? lay.tile_list : nullptr);
}

size_t dflash_append_context_workspace_size(const dflash_config_t* cfg, int B, int P,
                                            int L_cache) {
  if (check_cfg(cfg) != DFLASH_OK || B < 1 || P < 1 || L_cache < P) return 0;
  return proj_layout(cfg, B, P, nullptr, L_cache, true).bytes;
}

int dflash_append_context(const dflash_config_t* cfg, const dflash_weights_t* w,
                          const void* target_hidden, int B, int P, const int32_t* accepted,
                          int32_t* cache_len, int L_cache, void* kv_cache, void* ws,
                          size_t ws_bytes, void* stream) {
  int r;
  if ((r = check_cfg(cfg))) return r;
  if ((r = check_weights(cfg, w, false))) return r;
  if (B < 1 || P < 1 || L_cache < P)
    return fail(DFLASH_ERR_INVALID_ARG, "need B, P >= 1 and L_cache >= P");
  if (!cache_len) return fail(DFLASH_ERR_INVALID_ARG, "cache_len is null");
  if ((r = check_ptr16(target_hidden, "target_hidden", cfg->dtype))) return r;
  if ((r = check_ptr16(kv_cache, "kv_cache", DFLASH_DTYPE_BF16))) return r;
  if (cfg->dtype == DFLASH_DTYPE_BF16 && L_cache % 8 != 0)
    return fail(DFLASH_ERR_INVALID_ARG, "L_cache must be a multiple of 8 (16-byte fp16 cache rows)");
  const ProjLayout lay = proj_layout(cfg, B, P, ws, L_cache, true);
  if ((r = check_ws(ws, ws_bytes, lay.bytes))) return r;
  cudaStream_t s = (cudaStream_t)stream;
  // the rows each request commits (n_commit, from the plan kernel) decide the active tiles
  TileJob tj;
  if (cfg->dtype == DFLASH_DTYPE_BF16) {
    tj.kind = TileJob::kContext;
    tj.ctx_len = lay.n_commit;
    tj.B = B;
    tj.L = P;
    tj.list = lay.tile_list;
  }
  {
    Prof pr(DFLASH_PROF_ROWS, 2, s);
    DF_CUDA(launch_append_plan(accepted, cache_len, B, P, L_cache, lay.n_commit, lay.start,
                               status_ptr(), s));
    DF_CUDA(launch_rope_table(lay.cos_t, lay.sin_t, 0, L_cache, cfg->head_dim, cfg->rope_theta,
                              s, tj));
  }
  return project_rows(cfg, w, target_hidden, B, P, 0, L_cache, lay.n_commit, lay.start,
                      kv_cache, lay, s, tj.kind != TileJob::kNone ? lay.tile_list : nullptr);
}

// ---------------------------------------------------------------------------------------
size_t dflash_body_workspace_size(const dflash_config_t* cfg, int B, int L, int N) {
  if (check_cfg(cfg) != DFLASH_OK || B < 1 || L < 1 || N < 1) return 0;
  return body_layout(cfg, B, L, N, nullptr).bytes;
}

int dflash_body_forward(const dflash_config_t* cfg, const dflash_weights_t* w,
                        const void* block_emb, const int32_t* anchors,
                        const uint8_t* block_valid, const int32_t* position_ids,
                        const uint8_t* mask, const void* kv_cache, int B, int L, int N,
                        float* out, void* ws, size_t ws_bytes, void* stream) {
  int r;
  if ((r = check_cfg(cfg))) return r;
  if ((r = check_weights(cfg, w, true))) return r;
  if (B < 1 || L < 1 || N < 1) return fail(DFLASH_ERR_INVALID_ARG, "B, L and N must be >= 1");
  if (!anchors || !block_valid || !position_ids || !mask || !out)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  if ((r = check_ptr16(out, "out", cfg->dtype))) return r;
  if ((r = check_ptr16(mask, "mask", cfg->dtype))) return r;
  if ((r = check_ptr16(block_emb, "block_emb", cfg->dtype))) return r;
  if ((r = check_ptr16(kv_cache, "kv_cache", DFLASH_DTYPE_BF16))) return r;
  if (cfg->dtype == DFLASH_DTYPE_BF16 && L % 8 != 0)
    return fail(DFLASH_ERR_INVALID_ARG, "L must be a multiple of 8 (16-byte fp16 cache rows)");
  const BodyLayout lay = body_layout(cfg, B, L, N, ws);
  if ((r = check_ws(ws, ws_bytes, lay.bytes))) return r;
  cudaStream_t s = (cudaStream_t)stream;
  const int S = cfg->block_size;
  const long T = (long)B * N * S;
  const int D = cfg->hidden, dh = cfg->head_dim, Hq = cfg->num_heads, Hkv = cfg->num_kv_heads;
  const int qw = Hq * dh, kw = Hkv * dh, qkvw = qw + 2 * kw, I = cfg->intermediate;
  const int dt = cfg->dtype;
  const size_t es = esize(dt);
  unsigned* st = status_ptr();
  const size_t layer_elems = (size_t)B * 2 * Hkv * L * dh;

  // 128-slot tiles without a valid slot are skipped by every projection; their list is built
  // by one block of the RoPE-table launch
  const int32_t* flags = nullptr;
  TileJob tj;
  if (dt == DFLASH_DTYPE_BF16) {
    tj.kind = TileJob::kSlots;
    tj.valid = block_valid;
    tj.T = T;
    tj.list = lay.tile_list;
    flags = lay.tile_list;
  }
  {
    Prof pr(DFLASH_PROF_ROWS, 2, s);
    DF_CUDA(launch_rope_table(lay.cos_t, lay.sin_t, 0, lay.P, dh, cfg->rope_theta, s, tj));
    DF_CUDA(launch_residual_norm(kNormInit, dt, lay.x, block_emb, nullptr, 0, nullptr,
                                 w->layers[0].g_in, cfg->rms_eps, lay.h.out(), nullptr,
                                 block_valid, false, T, D, s));
  }
  const bool tc = dt == DFLASH_DTYPE_BF16;
  if (lay.fuse_qkv) {
    // the fused QKV epilogue writes active tiles only: zero the rest (and the V^T pad) once
    Prof pr(DFLASH_PROF_ROWS, 1, s);
    DF_CUDA(launch_qkv_clear(block_valid, static_cast<__half*>(lay.q), static_cast<__half*>(lay.kb),
                             static_cast<__half*>(lay.vbt), lay.ns_pad, T, N, S, Hq, Hkv, dh, s));
  }
  // weight-streaming GEMM of one layer projection: X (fp16) [T][K] x W [Nw][K]^T
  auto ws_args = [&](const void* X, int K, const void* W, int Nw, int max_splits, int* nsplit) {
    WsArgs a;
    a.X = X;
    a.ldx = K;
    a.M = T;
    a.W = W;
    a.w_dtype = layer_wdtype(cfg);
    a.ldw = K;
    a.Nw = Nw;
    a.K = K;
    a.tile_list = flags;
    a.C = lay.y;
    a.ldc = Nw;
    a.max_splits = max_splits;
    a.splits_out = nsplit;
    a.status = st;
    return a;
  };
  const bool use_ws = lay.ws;
  // fp16 copies of the layer matrices (exact for bf16 values in the fp16 range) are made on
  // a side stream, one layer ahead: the conversion (HBM-bound) of layer l + 1 runs beside
  // layer l's tensor-core work, into the buffer layer l - 1 used.
  const size_t sizes[4] = {(size_t)qkvw * D, (size_t)D * qw, (size_t)2 * I * D, (size_t)D * I};
  SideStream* side = nullptr;
  SideJoin join{s, &side};
  auto convert_layer = [&](int l) -> int {
    // after everything already on the caller's stream (layer l - 2's use of this buffer)
    join.joined = false;
    DF_CUDA(cudaEventRecord(side->fork, s));
    DF_CUDA(cudaStreamWaitEvent(side->s, side->fork, 0));
    const dflash_layer_weights_t& src = w->layers[l];
    const void* mats[4] = {src.w_qkv, src.w_o, src.w_gate_up, src.w_down};
    __half* dst = lay.wl16 + (size_t)(l % 2) * lay.wl16_layer;
    Prof pc(DFLASH_PROF_CONVERT, 4, side->s);
    for (int m = 0; m < 4; ++m) {
      DF_CUDA(launch_convert_bf16_f16(mats[m], dst, sizes[m], st, side->s));
      dst += sizes[m];
    }
    DF_CUDA(cudaEventRecord(side->done[l % 2], side->s));
    return DFLASH_OK;
  };
  if (lay.wl16) {
    DF_CUDA(side_stream(&side));
    if ((r = convert_layer(0)) != DFLASH_OK) return r;
  }
  for (int l = 0; l < cfg->num_layers; ++l) {
    dflash_layer_weights_t lw = w->layers[l];
    if (lay.wl16) {
      // this layer's fp16 matrices are ready; then the next layer's conversion starts
      DF_CUDA(cudaStreamWaitEvent(s, side->done[l % 2], 0));
      join.joined = true;  // every conversion forked so far is ordered before this layer
      if (l + 1 < cfg->num_layers && (r = convert_layer(l + 1)) != DFLASH_OK) return r;
      __half* buf = lay.wl16 + (size_t)(l % 2) * lay.wl16_layer;
      const void** mats[4] = {&lw.w_qkv, &lw.w_o, &lw.w_gate_up, &lw.w_down};
      for (int m = 0; m < 4; ++m) {
        *mats[m] = buf;
        buf += sizes[m];
      }
    }
    if (lay.fuse_qkv) {
      QkvEpilogue qe;
      qe.pos = position_ids;
      qe.valid = block_valid;
      qe.cos_t = lay.cos_t;
      qe.sin_t = lay.sin_t;
      qe.q = static_cast<__half*>(lay.q);
      qe.kb = static_cast<__half*>(lay.kb);
      qe.vbt = static_cast<__half*>(lay.vbt);
      qe.P = lay.P;
      qe.ns_pad = lay.ns_pad;
      qe.NS = N * S;
      qe.S = S;
      qe.Hq = Hq;
      qe.Hkv = Hkv;
      Prof pr(DFLASH_PROF_GEMM, 1, s);
      DF_CUDA(launch_gemm_tc_qkv(lay.h.p, D, lw.w_qkv, D, T, qkvw, D, flags, qe, st, s));
    } else {
      {
        Prof pr(DFLASH_PROF_GEMM, 1, s);
        if (use_ws)
          DF_CUDA(launch_gemm_ws(ws_args(lay.h.p, D, lw.w_qkv, qkvw, lay.sp_qkv, lay.nsplit), s));
        else
          DF_CUDA(gemm(dt, DFLASH_DTYPE_F16, lay.h.p, D, lw.w_qkv, D, lay.y, qkvw, T, qkvw, D,
                       lay.sp_qkv, s, flags, tc ? lay.nsplit : nullptr));
      }
      Prof pr(DFLASH_PROF_ROWS, 1, s);
      DF_CUDA(launch_qkv_rope(lay.y, lay.sp_qkv, tc ? lay.nsplit : nullptr, position_ids,
                              block_valid, lay.cos_t, lay.sin_t,
                              lay.P, lay.q, lay.kb, lay.vbt, lay.ns_pad, T, N, S, Hq, Hkv, dh,
                              dt == DFLASH_DTYPE_BF16, st, s));
    }
    if (dt == DFLASH_DTYPE_BF16) {
      AttnTcArgs aa;
      aa.q = static_cast<const __half*>(lay.q);
      aa.kb = static_cast<const __half*>(lay.kb);
      aa.vbt = static_cast<const __half*>(lay.vbt);
      aa.ns_pad = lay.ns_pad;
      aa.kv_layer = static_cast<const __half*>(kv_cache) + (size_t)l * layer_elems;
      aa.anchors = anchors;
      aa.valid = block_valid;
      aa.mask = mask;
      aa.partials = lay.partials;
      aa.out = lay.attn.out();
      aa.B = B;
      aa.N = N;
      aa.S = S;
      aa.L = L;
      aa.Hq = Hq;
      aa.Hkv = Hkv;
      aa.num_sms = num_sms();
      aa.status = st;
      const AttnTcLayout al = attention_tc_layout(B, N, S, L, Hq, Hkv, num_sms());
      Prof pr(DFLASH_PROF_ATTENTION, al.max_chunks == 1 ? 1 : 2, s);  // + combine pass
      DF_CUDA(launch_attention_tc(aa, s));
    } else {
      AttnArgs aa;
      aa.q = static_cast<const float*>(lay.q);
      aa.kb = static_cast<const float*>(lay.kb);
      aa.vbt = static_cast<const float*>(lay.vbt);
      aa.ns_pad = lay.ns_pad;
      aa.kv_layer = static_cast<const float*>(kv_cache) + (size_t)l * layer_elems;
      aa.anchors = anchors;
      aa.valid = block_valid;
      aa.mask = mask;
      aa.out = lay.attn.out();
      aa.B = B;
      aa.N = N;
      aa.S = S;
      aa.L = L;
      aa.Hq = Hq;
      aa.Hkv = Hkv;
      aa.dh = dh;
      aa.status = st;
      Prof pr(DFLASH_PROF_ATTENTION, 1, s);
      DF_CUDA(launch_attention_simt(dt, aa, s));
    }
    {
      Prof pr(DFLASH_PROF_GEMM, 1, s);
      if (lay.fuse_o)
        DF_CUDA(launch_gemm_tc_residual(lay.attn.p, qw, lw.w_o, qw, lay.x, D, T, D, qw, flags,
                                        block_valid, st, s));
      else if (use_ws)
        DF_CUDA(launch_gemm_ws(ws_args(lay.attn.p, qw, lw.w_o, D, lay.sp_o, lay.nsplit + 1), s));
      else
        DF_CUDA(gemm(dt, DFLASH_DTYPE_F16, lay.attn.p, qw, lw.w_o, qw, lay.y, D, T, D, qw, lay.sp_o,
                     s, flags, tc ? lay.nsplit + 1 : nullptr));
    }
    {
      Prof pr(DFLASH_PROF_ROWS, 1, s);
      if (lay.fuse_o)  // x already holds the sum: the norm only
        DF_CUDA(launch_residual_norm(kNormAdd, dt, lay.x, nullptr, nullptr, 0, nullptr, lw.g_post,
                                     cfg->rms_eps, lay.h.out(), nullptr, block_valid, false, T, D,
                                     s));
      else
        DF_CUDA(launch_residual_norm(kNormAdd, dt, lay.x, nullptr, lay.y, lay.sp_o,
                                     tc ? lay.nsplit + 1 : nullptr, lw.g_post, cfg->rms_eps,
                                     lay.h.out(), nullptr, block_valid, false, T, D, s));
    }
    if (use_ws && lay.sp_gu > 0) {
      // few tokens: K-split gate/up into fp32 slices (the fused epilogue would leave SMs
      // idle), SiLU(gate) * up by the row kernel
      {
        Prof pr(DFLASH_PROF_GEMM, 1, s);
        DF_CUDA(launch_gemm_ws(ws_args(lay.h.p, D, lw.w_gate_up, 2 * I, lay.sp_gu, lay.nsplit + 3),
                               s));
      }
      Prof pr(DFLASH_PROF_ROWS, 1, s);
      DF_CUDA(launch_swiglu(lay.y, lay.sp_gu, lay.nsplit + 3, lay.act.out(), T, I, block_valid, s));
    } else if (use_ws) {
      // SiLU(gate) * up is formed in the GEMM epilogue
      Prof pr(DFLASH_PROF_GEMM, 1, s);
      DF_CUDA(launch_gemm_ws_swiglu(ws_args(lay.h.p, D, lw.w_gate_up, 2 * I, 1, nullptr),
                                    lay.act.out(), s));
    } else if (tc) {
      Prof pr(DFLASH_PROF_GEMM, 1, s);
      DF_CUDA(launch_gemm_tc_swiglu(DFLASH_DTYPE_F16, lay.h.p, D, lw.w_gate_up, D, T, I, D, flags,
                                    lay.act.out(), st, s));
    } else {
      {
        Prof pr(DFLASH_PROF_GEMM, 1, s);
        DF_CUDA(gemm(dt, dt, lay.h.p, D, lw.w_gate_up, D, lay.y, 2 * I, T, 2 * I, D, lay.sp_gu, s));
      }
      Prof pr(DFLASH_PROF_ROWS, 1, s);
      DF_CUDA(launch_swiglu(lay.y, lay.sp_gu, nullptr, lay.act.out(), T, I, block_valid, s));
    }
    {
      Prof pr(DFLASH_PROF_GEMM, 1, s);
      if (lay.fuse_down)
        DF_CUDA(launch_gemm_tc_residual(lay.act.p, I, lw.w_down, I, lay.x, D, T, D, I, flags,
                                        block_valid, st, s));
      else if (use_ws)
        DF_CUDA(launch_gemm_ws(ws_args(lay.act.p, I, lw.w_down, D, lay.sp_down, lay.nsplit + 2), s));
      else
        DF_CUDA(gemm(dt, DFLASH_DTYPE_F16, lay.act.p, I, lw.w_down, I, lay.y, D, T, D, I,
                     lay.sp_down, s, flags, tc ? lay.nsplit + 2 : nullptr));
    }
    Prof pr(DFLASH_PROF_ROWS, 1, s);
    // fused: x already holds the sum (no slices to add)
    const float* yd = lay.fuse_down ? nullptr : lay.y;
    const int nsd = lay.fuse_down ? 0 : lay.sp_down;
    const int* nsd_dev = lay.fuse_down || !tc ? nullptr : lay.nsplit + 2;
    if (l + 1 < cfg->num_layers) {
      DF_CUDA(launch_residual_norm(kNormAdd, dt, lay.x, nullptr, yd, nsd, nsd_dev,
                                   w->layers[l + 1].g_in, cfg->rms_eps, lay.h.out(), nullptr,
                                   block_valid, false, T, D, s));
    } else {
      DF_CUDA(launch_residual_norm(kNormFinal, dt, lay.x, nullptr, yd, nsd, nsd_dev, w->g_final,
                                   cfg->rms_eps, ActOut(), out, block_valid,
                                   (cfg->flags & DFLASH_FLAG_FINAL_NORM) != 0, T, D, s));
    }
  }
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------------------
size_t dflash_verify_workspace_size(int B, int gamma, int V) {
  if (B < 1 || gamma < 0 || V < 1) return 0;
  return plan_verify(B, gamma, V, num_sms()).ws_bytes + 256;
}

int dflash_verify_greedy(const void* logits, int logits_dtype, const int32_t* draft, int B,
                         int gamma, int V, int32_t eos, int32_t* emitted, int32_t* num_emitted,
                         int32_t* accepted, int32_t* target_choices, void* ws, size_t ws_bytes,
                         void* stream) {
  if (B < 1 || gamma < 0 || V < 1)
    return fail(DFLASH_ERR_INVALID_ARG,
                "need B >= 1, gamma >= 0, V >= 1 (one target choice per draft token plus a bonus)");
  if (gamma > kMaxVerifyGamma)
    return fail(DFLASH_ERR_INVALID_ARG, "gamma (%d) must be <= %d", gamma, kMaxVerifyGamma);
  if ((long)B * (gamma + 1) > kMaxVerifyRows)
    return fail(DFLASH_ERR_UNSUPPORTED, "B * (gamma + 1) must be <= %ld", kMaxVerifyRows);
  if (logits_dtype != DFLASH_DTYPE_BF16 && logits_dtype != DFLASH_DTYPE_F32)
    return fail(DFLASH_ERR_INVALID_ARG, "logits_dtype must be DFLASH_DTYPE_BF16 or _F32");
  if (!logits || (!draft && gamma > 0) || !emitted || !num_emitted || !accepted)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  const VerifyPlan vp = plan_verify(B, gamma, V, num_sms());
  Carver cv(ws);
  const size_t rows = (size_t)B * (gamma + 1);
  float* pv = cv.take<float>(rows * vp.chunks);
  int* pi = cv.take<int>(rows * vp.chunks);
  int r;
  if ((r = check_ws(ws, ws_bytes, cv.off))) return r;
  Prof pr(DFLASH_PROF_VERIFY, 2, (cudaStream_t)stream);
  DF_CUDA(launch_verify(logits, logits_dtype, draft, B, gamma, V, eos, emitted, num_emitted,
                        accepted, target_choices, pv, pi, vp, (cudaStream_t)stream));
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------------------
size_t dflash_verify_sampling_workspace_size(int B, int gamma, int V) {
  if (B < 1 || gamma < 0 || V < 1) return 0;
  return plan_sampling(B, gamma, V, num_sms()).ws_bytes + 256;
}

int dflash_verify_sampling(const void* logits, int logits_dtype, double temperature,
                           const float* draft_probs, const int32_t* draft, int B, int gamma,
                           int V, uint64_t seed, int32_t eos, int32_t* emitted,
                           int32_t* num_emitted, int32_t* accepted, void* ws, size_t ws_bytes,
                           void* stream) {
  if (B < 1 || gamma < 0 || V < 1)
    return fail(DFLASH_ERR_INVALID_ARG,
                "need B >= 1, gamma >= 0, V >= 1 (one target distribution per draft token "
                "plus the final one)");
  if ((long)B * (gamma + 1) > kMaxVerifyRows)
    return fail(DFLASH_ERR_UNSUPPORTED, "B * (gamma + 1) must be <= %ld", kMaxVerifyRows);
  if (!(temperature > 0.0) || !(1.0 / temperature < 3.0e38))
    return fail(DFLASH_ERR_INVALID_ARG, "temperature must be > 0 (greedy verification is "
                "dflash_verify_greedy)");
  if (logits_dtype != DFLASH_DTYPE_BF16 && logits_dtype != DFLASH_DTYPE_F32)
    return fail(DFLASH_ERR_INVALID_ARG, "logits_dtype must be DFLASH_DTYPE_BF16 or _F32");
  if (!logits || (gamma > 0 && (!draft || !draft_probs)) || !emitted || !num_emitted ||
      !accepted)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  const SamplingPlan sp = plan_sampling(B, gamma, V, num_sms());
  int r;
  if ((r = check_ws(ws, ws_bytes, sp.ws_bytes))) return r;
  Prof pr(DFLASH_PROF_VERIFY, 4, (cudaStream_t)stream);
  // the kernels work in base 2: y = logit * log2(e) / temperature
  DF_CUDA(launch_verify_sampling(logits, logits_dtype, (float)(1.4426950408889634 / temperature),
                                 draft_probs,
                                 draft, B, gamma, V, seed, eos, emitted, num_emitted, accepted,
                                 ws, sp, status_ptr(), (cudaStream_t)stream));
  return DFLASH_OK;
}

// ---------------------------------------------------------------------------------------
size_t dflash_decayed_ce_workspace_size(int T, int D, int V) {
  if (T < 1 || D < 1 || V < 1) return 0;
  return ce_layout(T, D, V, nullptr).bytes + 256;
}

int dflash_decayed_ce_loss(const float* hidden, const void* lm_head, const int32_t* targets,
                           const uint8_t* loss_mask, int T, int block_size, int D, int V,
                           double decay, float* ce, float* loss, void* ws, size_t ws_bytes,
                           void* stream) {
  if (T < 1 || block_size < 1 || D < 1 || V < 1 || T % block_size != 0)
    return fail(DFLASH_ERR_INVALID_ARG, "need T, block_size, D, V >= 1 and T a multiple of "
                "block_size");
  if (!(decay > 0.0)) return fail(DFLASH_ERR_INVALID_ARG, "decay must be > 0");
  if (D % 8 != 0)
    return fail(DFLASH_ERR_UNSUPPORTED, "D must be a multiple of 8 (16-byte rows for TMA)");
  if (!targets || !loss_mask || !ce || !loss)
    return fail(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  int r;
  if ((r = check_ptr16(hidden, "hidden", DFLASH_DTYPE_F32))) return r;
  if ((r = check_ptr16(lm_head, "lm_head", DFLASH_DTYPE_BF16))) return r;
  const CeLayout l = ce_layout(T, D, V, ws);
  if ((r = check_ws(ws, ws_bytes, l.bytes))) return r;
  Prof pr(DFLASH_PROF_GEMM, 5, (cudaStream_t)stream);
  DF_CUDA(launch_decayed_ce(hidden, lm_head, targets, loss_mask, T, block_size, D, V, decay, ce,
                            loss, l, status_ptr(), (cudaStream_t)stream));
  return DFLASH_OK;
}

// ---- testing hooks -----------------------------------------------------------------------
int dflash_testing_gemm(int engine, int dtype, const void* A, long lda, const void* Bm, long ldb,
                        float* C, long ldc, long M, int N, int K, int splits, void* stream) {
  if (M < 1 || N < 1 || K < 1 || !A || !Bm || !C) return fail(DFLASH_ERR_INVALID_ARG, "bad gemm args");
  cudaStream_t s = (cudaStream_t)stream;
  if (engine == DFLASH_TESTING_ENGINE_TC) {
    if ((dtype != DFLASH_DTYPE_BF16 && dtype != DFLASH_DTYPE_F16) ||
        !gemm_tc_supported(M, N, K, lda, ldb))
      return fail(DFLASH_ERR_UNSUPPORTED, "tensor-core GEMM needs bf16 or fp16 and 16-byte rows");
    DF_CUDA(launch_gemm_tc(dtype, A, lda, Bm, ldb, C, ldc, M, N, K, splits, nullptr,
                           status_ptr(), s));
  } else {
    if (dtype == DFLASH_DTYPE_F16) return fail(DFLASH_ERR_UNSUPPORTED, "CUDA-core GEMM: bf16 or fp32");
    DF_CUDA(launch_gemm_simt(dtype, A, lda, Bm, ldb, C, ldc, M, N, K, splits, s));
  }
  return DFLASH_OK;
}

int dflash_testing_gemm_splits(long M, int N, int K) { return gemm_splits(M, N, K); }

int dflash_testing_rope_table(float* cos_t, float* sin_t, int p0, int P, int head_dim,
                              double theta, void* stream) {
  if (!cos_t || !sin_t || ((uintptr_t)cos_t | (uintptr_t)sin_t) % 16 != 0)
    return fail(DFLASH_ERR_INVALID_ARG, "cos_t / sin_t must be non-null and 16-byte aligned");
  if (head_dim < 2 || head_dim % 2 != 0 || head_dim > 256 || P < 1 || p0 < 0 ||
      (long)p0 + P > (1L << 24) || !(theta > 1.0))
    return fail(DFLASH_ERR_INVALID_ARG,
                "need head_dim even in [2, 256], P >= 1, 0 <= p0, p0 + P <= 2^24, theta > 1");
  DF_CUDA(launch_rope_table(cos_t, sin_t, p0, P, head_dim, theta, (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_testing_gemm_pairs(int mode) {
  if (mode < 0 || mode > 1) return fail(DFLASH_ERR_INVALID_ARG, "mode must be 0 or 1");
  set_gemm_tc_pairs(mode);
  return DFLASH_OK;
}

int dflash_testing_fused_epilogues(int mode) {
  if (mode < 0 || mode > 2) return fail(DFLASH_ERR_INVALID_ARG, "mode must be 0, 1 or 2");
  g_fused_mode.store(mode);
  return DFLASH_OK;
}

int dflash_testing_gemm_withheld(const void* A, long lda, const void* Bm, long ldb, float* C,
                                 long ldc, long M, int N, int K, long wait_ns, void* stream) {
  if (M < 1 || N < 1 || K < 1 || !A || !Bm || !C || wait_ns < 1000 || wait_ns > 100000000L)
    return fail(DFLASH_ERR_INVALID_ARG, "bad withheld-gemm args (wait_ns in [1 us, 100 ms])");
  if (!gemm_tc_supported(M, N, K, lda, ldb))
    return fail(DFLASH_ERR_UNSUPPORTED, "tensor-core GEMM needs 16-byte rows");
  DF_CUDA(launch_gemm_tc_withheld(A, lda, Bm, ldb, C, ldc, M, N, K, (uint64_t)wait_ns,
                                  status_ptr(), (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_testing_gemm_ws(const void* X, long ldx, const void* W, int w_dtype, long ldw,
                           float* C, long ldc, long M, int N, int K, int max_splits,
                           const int32_t* tile_list, int32_t* splits_out, void* stream) {
  if (M < 1 || N < 1 || K < 1 || !X || !W || !C || max_splits < 1 || max_splits > 8)
    return fail(DFLASH_ERR_INVALID_ARG, "bad gemm_ws args");
  if ((w_dtype != DFLASH_DTYPE_BF16 && w_dtype != DFLASH_DTYPE_F16) || ldx % 8 || ldw % 8 ||
      ldx < K || ldw < K)
    return fail(DFLASH_ERR_UNSUPPORTED, "gemm_ws needs bf16/fp16 weights and 16-byte rows");
  WsArgs a;
  a.X = X;
  a.ldx = ldx;
  a.M = M;
  a.W = W;
  a.w_dtype = w_dtype;
  a.ldw = ldw;
  a.Nw = N;
  a.K = K;
  a.tile_list = tile_list;
  a.C = C;
  a.ldc = ldc;
  a.max_splits = max_splits;
  a.splits_out = splits_out;
  a.status = status_ptr();
  DF_CUDA(launch_gemm_ws(a, (cudaStream_t)stream));
  return DFLASH_OK;
}

int dflash_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (auto& r : g_prof) {
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof.clear();
  g_prof_on = on != 0;
  return DFLASH_OK;
}

int dflash_profile_read(int kind, double* total_ms, long* launches) {
  if (!total_ms || !launches || kind < 0 || kind >= DFLASH_PROF_KINDS)
    return fail(DFLASH_ERR_INVALID_ARG, "bad profile query");
  DF_CUDA(cudaDeviceSynchronize());
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double ms = 0.0;
  long n = 0;
  for (const auto& r : g_prof) {
    if (r.kind != kind) continue;
    float t = 0.f;
    DF_CUDA(cudaEventElapsedTime(&t, r.a, r.b));
    ms += t;
    n += r.count;
  }
  *total_ms = ms;
  *launches = n;
  return DFLASH_OK;
}

long dflash_launch_count(void) { return g_launches.load(); }

}  // extern "C"

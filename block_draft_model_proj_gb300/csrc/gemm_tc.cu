// 16-bit GEMM on the 5th-generation tensor cores: C[z] (fp32) = A[:, Kz] * B[:, Kz]^T.
//
// A [M, K] and B [N, K] are row-major (both K-major), both bf16 or both fp16; C is fp32
// row-major.  This is the contraction behind every projection of the draft body: W_proj
// ("DFlash", How it works: target hidden states projected into the K/V space) runs bf16 x
// bf16 on the target's exact bf16 hidden states; the context K/V projections and the
// per-layer QKV / O / gate-up / down projections run fp16 x fp16, on fp16 copies of the
// layer weights and on activations (norm outputs, the attention output, the SwiGLU
// product) rounded to fp16, whose 11 significant bits keep the body within its stated
// error bound where bf16 activations (8 bits) do not.
//
// Design (sm_103a):
//  * persistent CTAs (one per SM), 128 x 256 output tile, K stepped 64 at a time;
//  * warp 0 = TMA producer: cp.async.bulk.tensor loads of a 128x64 A box and two 128x64
//    B boxes, 128-byte swizzle, into a 4-stage shared-memory ring guarded by mbarriers;
//  * warp 1 = MMA issuer: one thread issues tcgen05.mma.cta_group::1.kind::f16 (M=128,
//    N=256, K=16) with fp32 accumulation in tensor memory; tcgen05.commit frees a stage;
//  * warps 2-5 = epilogue: tcgen05.ld of the accumulator (each warp owns its 32-lane
//    quarter of TMEM), transposed through shared memory into coalesced fp32 row stores;
//  * two 256-column accumulators (all 512 TMEM columns) so the epilogue of tile i overlaps
//    the main loop of tile i+1;
//  * optional K-split: split z writes its own C slice (deterministic; the consumer adds the
//    slices in a fixed order).
// Every mbarrier wait is bounded in time: on expiry the CTA raises a shared abort flag,
// reports DFLASH_ERR_TIMEOUT through the device status word, waits (bounded) for its own
// outstanding TMA copies and MMAs, frees its tensor memory and exits.
#include <cuda.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace dflash {

namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTileABytes = kBM * kBK * 2;    // 16 KB
constexpr uint32_t kStageBBytes = kBN * kBK * 2;   // 32 KB
constexpr uint32_t kStagingFloats = 32 * 33;       // per epilogue warp

constexpr uint32_t kStageABytes = kTileABytes;
// One CTA: a 128 x 256 tile, B stage 256 rows, 4 stages.  CTA pair (kPair): a 256 x 256 tile,
// each CTA holds its 128 A rows and half of the B rows (128), 6 stages of 32 KB.
template <int kPair>
struct Ring {
  static constexpr int kStages = kPair ? 6 : 4;
  static constexpr uint32_t kStageB = kPair ? kStageBBytes / 2 : kStageBBytes;
  // bytes one stage's full barrier waits for: the leader's barrier counts both CTAs' copies
  static constexpr uint32_t kTx = (kPair ? 2u : 1u) * (kStageABytes + kStageB);
};
constexpr size_t kSmemBytes = 1024 + 4 * (size_t)(kStageABytes + kStageBBytes) +
                              4 * kStagingFloats * sizeof(float) + 256;
static_assert(Ring<1>::kStages * (kStageABytes + Ring<1>::kStageB) ==
                  Ring<0>::kStages * (kStageABytes + Ring<0>::kStageB),
              "both rings fill the same shared memory");

// Instruction descriptor, kind::f16: D = fp32 (bits 4-5 = 1), A and B format at bits 7-9
// and 10-12 (0 = fp16, 1 = bf16), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t idesc_16bit(bool bf16, int M = kBM) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_16bit(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The CTA pair's MMA (M = 256): A rows 0-127 from this CTA's shared memory and 128-255 from
// the peer's, B columns 0-127 from this CTA's and 128-255 from the peer's (same offsets);
// each CTA's tensor memory receives its own 128 rows.  Issued by the even CTA only.
__device__ __forceinline__ void umma_16bit_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

enum : int {
  kEpiStoreF32 = 0,
  kEpiKvCache = 1,
  kEpiSwiGLU = 2,
  kEpiCrossEntropy = 3,
  kEpiQkv = 4,
  kEpiResidual = 5
};

struct TcParams {
  long M;
  int N, K;
  int m_tiles, n_tiles, splits, kb_per_split, num_kb;
  int* splits_out;  // non-null: splits is an upper bound, the count is chosen on the device
  int sms;
  float* C;
  long ldc;
  const int32_t* tile_list;    // optional: [0] = count, [1..] = active M tiles in order
  int m_fastest;               // tile order: M tiles fastest (shares each B tile) or N fastest
  uint32_t idesc;              // instruction descriptor: bf16 or fp16 operands
  unsigned* status;
  KvCacheEpilogue kv;          // used by the kEpiKvCache epilogue only
  ActOut act;                  // kEpiSwiGLU: SiLU(gate) * up, [M][swiglu_I]
  int swiglu_I;                // kEpiSwiGLU: B rows [0, I) gate, [I, 2I) up
  CrossEntropyEpilogue ce;     // kEpiCrossEntropy: per-tile softmax statistics of each row
  QkvEpilogue qkv;             // kEpiQkv: attention-ready Q / K (RoPE) and V^T
  const uint8_t* row_valid;    // kEpiResidual: rows added into C (= the residual stream)
  uint32_t idesc_pair;         // the CTA pair's instruction descriptor (M = 256)
  uint64_t wait_ns;            // limit of every bounded wait (kWaitLimitNs)
  int test_withhold;           // testing only: the producer issues no copy and no arrival,
                               // so the first wait of the MMA thread runs out
};

// Number of M tiles the work list runs over: all, or the compacted active ones.
__device__ __forceinline__ int active_m_tiles(const TcParams& p) {
  return p.tile_list ? p.tile_list[0] : p.m_tiles;
}

// Work item t -> (M unit, N tile, K split).  Every role walks the same sequence.  A unit is
// one M tile, or for a CTA pair two consecutive entries of the M tile order.
__device__ __forceinline__ void decode_tile(const TcParams& p, int m_units, int t, int& mu,
                                            int& n_t, int& z) {
  if (p.m_fastest) {
    mu = t % m_units;
    const int rest = t / m_units;
    n_t = rest % p.n_tiles;
    z = rest / p.n_tiles;
  } else {
    n_t = t % p.n_tiles;
    const int rest = t / p.n_tiles;
    mu = rest % m_units;
    z = rest / m_units;
  }
}

// This CTA's M tile of unit mu.  The second tile of a pair's last unit may not exist (an odd
// tile count): the CTA then takes tile m_tiles, whose rows lie past M -- its loads read the
// zero fill and its epilogue writes nothing.
__device__ __forceinline__ int unit_m_tile(const TcParams& p, int m_cnt, int mu, int pair,
                                           uint32_t rank) {
  const int mi = pair ? 2 * mu + (int)rank : mu;
  if (mi >= m_cnt) return p.m_tiles;
  return p.tile_list ? p.tile_list[1 + mi] : mi;
}

// Rotate-half RoPE of one 128-channel head held in tensor-memory columns hbase .. +127 of
// the thread's lane (channel i pairs with i + 64; cs / sn = the position's table row of 64
// angles), rounded to fp16 and stored as dst[0 .. 127].  Every lane takes part in the
// tensor-memory loads (.sync.aligned); only lanes with `write` store, zeros when !live.
__device__ __forceinline__ void rope_head_f16(uint32_t hbase, const float* cs, const float* sn,
                                              __half* dst, bool write, bool live, bool& bad) {
#pragma unroll 1
  for (int ch = 0; ch < 2; ++ch) {  // channel chunks (32ch .. 32ch+31) and their pairs +64
    uint32_t lo[32], hi[32];
    tmem_ld_32x32b_x32(hbase + ch * 32, lo);
    tmem_ld_32x32b_x32(hbase + 64 + ch * 32, hi);
    if (!write) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // 8 channels (16 bytes of fp16) per step
      uint32_t wa[4] = {0u, 0u, 0u, 0u}, wb[4] = {0u, 0u, 0u, 0u};
      if (live) {
#pragma unroll
        for (int t2 = 0; t2 < 4; ++t2) {
          const int t = 8 * q + 2 * t2;
          const float2 c2 = *reinterpret_cast<const float2*>(cs + ch * 32 + t);
          const float2 s2 = *reinterpret_cast<const float2*>(sn + ch * 32 + t);
          const float x00 = __uint_as_float(lo[t]), x10 = __uint_as_float(hi[t]);
          const float x01 = __uint_as_float(lo[t + 1]), x11 = __uint_as_float(hi[t + 1]);
          const float a0 = x00 * c2.x - x10 * s2.x, a1 = x01 * c2.y - x11 * s2.y;
          const float b0 = x10 * c2.x + x00 * s2.x, b1 = x11 * c2.y + x01 * s2.y;
          bad = bad || !(fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(b0), fabsf(b1))) +
                         0.f * (a0 + a1 + b0 + b1) < 65520.f);
          const __half2 ha = __floats2half2_rn(a0, a1);
          const __half2 hb = __floats2half2_rn(b0, b1);
          wa[t2] = *reinterpret_cast<const uint32_t*>(&ha);
          wb[t2] = *reinterpret_cast<const uint32_t*>(&hb);
        }
      }
      reinterpret_cast<uint4*>(dst + ch * 32)[q] = make_uint4(wa[0], wa[1], wa[2], wa[3]);
      reinterpret_cast<uint4*>(dst + 64 + ch * 32)[q] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
    }
  }
}

// One 128-channel V head of the thread's lane, rounded to fp16 and stored transposed:
// channel d at dst[d * stride] (consecutive lanes hold consecutive positions, so the stores
// of a warp are coalesced).  Zeros when !live; nothing stored without `write`.
__device__ __forceinline__ void v_head_f16(uint32_t hbase, __half* dst, long stride, bool write,
                                           bool live, bool& bad) {
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(hbase + ch * 32, v);
    if (!write) continue;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const float x = live ? __uint_as_float(v[t]) : 0.f;
      bad = bad || !(fabsf(x) < 65520.f);
      dst[(long)(ch * 32 + t) * stride] = __float2half_rn(x);
    }
  }
}

// Context K/V epilogue of the K/V projection of e.layers consecutive layers (N = layers *
// 2*Hkv*dh, dh = 128: every 256-column tile holds two whole heads; per layer the K heads, then
// the V heads).  Row m of the tile is context
// position c = m mod L of row b = m / L, cache position pos_offset + c.  K heads get RoPE
// (rotate-half: channel i pairs with i + 64; table row c) and are written as cache rows
// [pos][dh]; V heads are written transposed, [dh][pos].  Rows at or past ctx_len[b] are not
// written.  The cache holds fp16 (round to nearest even).
__device__ __forceinline__ void kv_cache_epilogue(const TcParams& p, uint32_t tbase, int m_t,
                                                  int n_t, int quarter, int lane) {
  const KvCacheEpilogue& e = p.kv;
  const long m = (long)m_t * kBM + quarter * 32 + lane;
  const int b = (int)(m / e.L);
  const int c = (int)(m - (long)b * e.L);
  bool row_ok = m < p.M;
  if (row_ok && e.ctx_len) row_ok = c < e.ctx_len[b];
  const long pos = (e.row_pos0 && row_ok ? (long)e.row_pos0[b] : (long)e.pos_offset) + c;
  const long trow = e.row_pos0 ? pos : c;  // RoPE table row of this position
  const long plane = (long)e.L_cache * 128;
  bool bad = false;  // a value outside the fp16 range (or NaN) met the cache
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    const int hg = n_t * 2 + hh;               // head over all layers
    if (hg >= e.layers * 2 * e.Hkv) break;     // warp-uniform
    const int l = hg / (2 * e.Hkv);
    const int head = hg - l * 2 * e.Hkv;       // 0 .. 2*Hkv-1: K heads, then V heads
    __half* kvl = e.kv + (long)l * e.layer_elems;
    const uint32_t hbase = tbase + hh * 128;
    if (head < e.Hkv) {
      __half* dst = kvl + ((long)b * 2 * e.Hkv + head) * plane + pos * 128;
      rope_head_f16(hbase, e.cos_t + trow * 64, e.sin_t + trow * 64, dst, row_ok, true, bad);
    } else {
      __half* dst = kvl + ((long)b * 2 * e.Hkv + e.Hkv + (head - e.Hkv)) * plane + pos;
      v_head_f16(hbase, dst, e.L_cache, row_ok, true, bad);
    }
  }
  if (bad) report(p.status, kStatusRange, kKernEpilogue);
}

// QKV epilogue of a draft layer (N = (Hq + 2 Hkv) * 128: every 256-column tile holds two
// whole heads, Q heads first, then K, then V).  Row m is slot m = (b, k, j) of the blocks
// (b = m / NS, ks = k * S + j = m mod NS).  Q and K heads get RoPE at the slot's position
// ("DFlash Draft Body", How It Works step 3: position ids of the drafted slots) into
// q [B][Hkv][NS][grp][128] and kb [B][Hkv][NS][128]; V heads go transposed into
// vbt [B][Hkv][128][ns_pad].  An invalid slot is written as zeros.
__device__ __forceinline__ void qkv_epilogue(const TcParams& p, uint32_t tbase, int m_t, int n_t,
                                             int quarter, int lane) {
  const QkvEpilogue& e = p.qkv;
  const long m = (long)m_t * kBM + quarter * 32 + lane;
  const bool row_ok = m < p.M;
  const bool live = row_ok && e.valid[m] != 0;
  const long b = m / e.NS;
  const long ks = m - b * e.NS;
  int pp = 0;
  if (live) {
    pp = e.pos[m];
    if (pp < 0 || pp >= e.P) {
      report(p.status, kStatusCheck, kKernEpilogue);
      pp = 0;
    }
  }
  const int grp = e.Hq / e.Hkv;
  const int heads = e.Hq + 2 * e.Hkv;
  bool bad = false;
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    const int hd = n_t * 2 + hh;
    if (hd >= heads) break;  // warp-uniform
    const uint32_t hbase = tbase + hh * 128;
    if (hd < e.Hq + e.Hkv) {
      __half* dst;
      if (hd < e.Hq) {
        const int g = hd / grp, h = hd - g * grp;
        dst = e.q + (((b * e.Hkv + g) * e.NS + ks) * grp + h) * 128;
      } else {
        dst = e.kb + ((b * e.Hkv + (hd - e.Hq)) * e.NS + ks) * 128;
      }
      rope_head_f16(hbase, e.cos_t + (long)pp * 64, e.sin_t + (long)pp * 64, dst, row_ok, live,
                    bad);
    } else {
      __half* dst = e.vbt + (b * e.Hkv + (hd - e.Hq - e.Hkv)) * 128 * (long)e.ns_pad + ks;
      v_head_f16(hbase, dst, e.ns_pad, row_ok, live, bad);
    }
  }
  if (bad) report(p.status, kStatusRange, kKernEpilogue);
}

// Residual epilogue: C[row][col] += tile for the valid rows (C is the fp32 residual stream,
// row stride ldc a multiple of 4).  The thread owns its TMEM lane's row: for each 32-column
// chunk it issues the eight 16-byte loads of its 128-byte piece of the row first, then reads
// the accumulator chunk, adds and stores.
__device__ __forceinline__ void residual_epilogue(const TcParams& p, uint32_t tbase, int m_t,
                                                  int n_t, int quarter, int lane) {
  const long row = (long)m_t * kBM + quarter * 32 + lane;
  const bool live = row < p.M && p.row_valid[row] != 0;
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    const int col0 = n_t * kBN + c * 32;
    const bool ok = live && col0 < p.N;  // N is a multiple of 32
    float4* xp = reinterpret_cast<float4*>(p.C + row * p.ldc + col0);
    float4 xr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xr[i] = ok ? xp[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t v[32];
    tmem_ld_32x32b_x32(tbase + c * 32, v);
    if (!ok) continue;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      xp[i] = make_float4(xr[i].x + __uint_as_float(v[4 * i]), xr[i].y + __uint_as_float(v[4 * i + 1]),
                          xr[i].z + __uint_as_float(v[4 * i + 2]),
                          xr[i].w + __uint_as_float(v[4 * i + 3]));
  }
}

// SwiGLU epilogue: accumulator columns [0, 128) are the gate and [128, 256) the up
// projections of channels n_t*128 .. +127; writes act = SiLU(gate) * up.
__device__ __forceinline__ void swiglu_epilogue(const TcParams& p, uint32_t tbase, int m_t, int n_t,
                                                int quarter, int lane) {
  const long m = (long)m_t * kBM + quarter * 32 + lane;
  const bool row_ok = m < p.M;
  const int I = p.swiglu_I;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t g[32], up[32];
    tmem_ld_32x32b_x32(tbase + c * 32, g);
    tmem_ld_32x32b_x32(tbase + 128 + c * 32, up);
    const int ch0 = n_t * 128 + c * 32;
    if (!row_ok) continue;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float a[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float gt = __uint_as_float(g[4 * q + t]);
        a[t] = gt / (1.f + expf(-gt)) * __uint_as_float(up[4 * q + t]);
      }
      const int ch = ch0 + 4 * q;
      if (ch + 3 < I) {
        p.act.store4(m * I + ch, make_float4(a[0], a[1], a[2], a[3]));
      } else {
        for (int t = 0; t < 4; ++t)
          if (ch + t < I) p.act.store(m * I + ch + t, a[t]);
      }
    }
  }
}

// Cross-entropy epilogue (lm_head logits, never stored): row m of the tile, columns
// n_t*256 .. +255 below V.  Writes the tile's (max, sum of exp(logit - max)) of the row and,
// from the one tile that holds it, the logit of the row's target token.
__device__ __forceinline__ void cross_entropy_epilogue(const TcParams& p, uint32_t tbase, int m_t,
                                                       int n_t, int quarter, int lane) {
  const CrossEntropyEpilogue& e = p.ce;
  const long m = (long)m_t * kBM + quarter * 32 + lane;
  const bool row_ok = m < p.M;
  const int tgt = row_ok ? e.targets[m] : -1;
  float mx = -INFINITY, sum = 0.f, tlogit = 0.f;
  bool has_t = false;
#pragma unroll 1
  for (int c = 0; c < kBN / 32; ++c) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tbase + c * 32, v);
    const int col0 = n_t * kBN + c * 32;
    if (col0 >= e.V) continue;  // warp-uniform; the loads above stay .sync.aligned
    const int nv = min(32, e.V - col0);
    float cm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nv) cm = fmaxf(cm, __uint_as_float(v[i]));
    if (cm > mx) {
      sum = mx == -INFINITY ? 0.f : sum * expf(mx - cm);
      mx = cm;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < nv) sum += expf(__uint_as_float(v[i]) - mx);
      if (col0 + i == tgt) {
        tlogit = __uint_as_float(v[i]);
        has_t = true;
      }
    }
  }
  if (row_ok) {
    float* part = e.part + ((size_t)m * p.n_tiles + n_t) * 2;
    part[0] = mx;
    part[1] = sum;
    if (has_t) e.target_logit[m] = tlogit;
  }
}

template <int kEpi, int kPair>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const TcParams p) {
  using R = Ring<kPair>;
  constexpr int kStages = R::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kStageABytes;
  float* staging = reinterpret_cast<float*>(sB + kStages * R::kStageB);
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + 4 * kStagingFloats);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA pair: rank 0 (the leader) issues the MMAs and owns the full / tempty barriers that
  // count both CTAs; each CTA loads its own A rows and half of B and stores its own rows.
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kPair ? 8 : 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       smem_u32(tmem_slot)),
                   "r"(kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();  // the peer's barriers are initialised before any use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // prologue done (barriers, tensor memory): wait for the predecessor grid's results, then
  // let the successor grid be scheduled
  pdl_wait();
  pdl_trigger();

  const int m_cnt = active_m_tiles(p);
  const int m_units = kPair ? (m_cnt + 1) / 2 : m_cnt;
  const int workers = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;  // CTAs or CTA pairs
  const int worker = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  int n_splits = p.splits, kb_per = p.kb_per_split;
  if (p.splits_out) {
    n_splits = choose_splits((long)m_units * p.n_tiles, p.num_kb, p.splits, p.sms / (kPair + 1));
    kb_per = (p.num_kb + n_splits - 1) / n_splits;
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.splits_out = n_splits;
  }
  const int total = m_units * p.n_tiles * n_splits;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t ph = 0;
      int issued[kStages];
      uint32_t issued_ph[kStages];
      for (int s = 0; s < kStages; ++s) issued[s] = 0, issued_ph[s] = 0;
      bool ok = p.test_withhold == 0;
      for (int t = worker; t < total && ok; t += workers) {
        int mu, n_t, z;
        decode_tile(p, m_units, t, mu, n_t, z);
        const int m_t = unit_m_tile(p, m_cnt, mu, kPair, rank);
        const int kb0 = z * kb_per;
        const int kb1 = min(p.num_kb, kb0 + kb_per);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, p.wait_ns)) { ok = false; break; }
          uint8_t* a_dst = sA + stage * kStageABytes;
          uint8_t* b_dst = sB + stage * R::kStageB;
          if constexpr (kPair) {
            // the leader's full barrier counts both CTAs' bytes of the stage
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], R::kTx);
            const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
            tma_load_2d_pair(&map_a, fb, a_dst, kb * kBK, m_t * kBM);
            // this CTA's half of the B tile: columns 128*rank .. +127 of the output tile, or
            // (SwiGLU) the gate rows of 128 channels (leader) and their up rows (peer)
            const int brow = kEpi == kEpiSwiGLU ? (rank ? p.swiglu_I : 0) + n_t * 128
                                                : n_t * kBN + (int)rank * 128;
            tma_load_2d_pair(&map_b, fb, b_dst, kb * kBK, brow);
          } else {
            mbar_arrive_expect_tx(&full[stage], R::kTx);
            tma_load_2d(&map_a, &full[stage], a_dst, kb * kBK, m_t * kBM);
            // the two 128-row halves of the B tile: consecutive rows, or (SwiGLU) the gate
            // rows of 128 channels and the up rows of the same channels
            const int brow0 = kEpi == kEpiSwiGLU ? n_t * 128 : n_t * kBN;
            const int brow1 = kEpi == kEpiSwiGLU ? p.swiglu_I + n_t * 128 : n_t * kBN + 128;
            tma_load_2d(&map_b, &full[stage], b_dst, kb * kBK, brow0);
            tma_load_2d(&map_b, &full[stage], b_dst + R::kStageB / 2, kb * kBK, brow1);
          }
          issued[stage] = 1;
          issued_ph[stage] = ph;
          if (++stage == kStages) { stage = 0; ph ^= 1u; }
        }
      }
      // wait for the copies still in flight (a pair's leader: both CTAs' copies, which its
      // full barriers count; the peer's copies complete on those barriers only)
      if (!kPair || rank == 0)
        for (int s = 0; s < kStages; ++s)
          if (issued[s]) mbar_drain_wait(&full[s], issued_ph[s], p.wait_ns / 4);
    }
  } else if (warp == 1) {
    if (lane == 0 && (!kPair || rank == 0)) {
      // ---------------- MMA issuer ----------------
      int stage = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t acc_ph = 0;
      bool ok = true;
      for (int t = worker; t < total && ok; t += workers) {
        int mu, n_t, z;
        decode_tile(p, m_units, t, mu, n_t, z);
        const int kb0 = z * kb_per;
        const int kb1 = min(p.num_kb, kb0 + kb_per);
        if (!mbar_wait(&tempty[acc], acc_ph ^ 1u, abort_flag, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], ph, abort_flag, p.wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint64_t a_desc = sw128_desc(smem_u32(sA + stage * kStageABytes));
          const uint64_t b_desc = sw128_desc(smem_u32(sB + stage * R::kStageB));
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // advancing K by 16 elements = 32 bytes inside the 128-byte swizzle atom (the
            // descriptor's address field counts 16-byte units)
            const uint32_t accum = (kb > kb0 || k > 0) ? 1u : 0u;
            if constexpr (kPair)
              umma_16bit_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, p.idesc_pair, accum);
            else
              umma_16bit(d_tmem, a_desc + 2 * k, b_desc + 2 * k, p.idesc, accum);
          }
          if constexpr (kPair) umma_commit_pair_multicast(&empty[stage], 3);  // both CTAs' stage
          else umma_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        if constexpr (kPair) umma_commit_pair_multicast(&tfull[acc], 3);
        else umma_commit(&tfull[acc]);
        if (++acc == 2) { acc = 0; acc_ph ^= 1u; }
      }
      // all MMAs issued by this thread complete before tensor memory is released
      if constexpr (kPair) umma_commit_pair(drain);
      else umma_commit(drain);
      mbar_drain_wait(drain, 0, p.wait_ns / 4);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    float* stg = staging + (warp - 2) * kStagingFloats;
    // a pair's accumulator is released on the leader's barrier (8 arrivals: both CTAs)
    const uint32_t tempty_leader = kPair ? mapa_shared(smem_u32(tempty), 0) : 0u;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int t = worker; t < total; t += workers) {
      int mu, n_t, z;
      decode_tile(p, m_units, t, mu, n_t, z);
      const int m_t = unit_m_tile(p, m_cnt, mu, kPair, rank);
      // warp-uniform result: the tcgen05.ld below is .sync.aligned
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_ph, abort_flag, p.wait_ns) ? 1 : 0))
        break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN);
      if constexpr (kEpi == kEpiStoreF32) {
        float* Cz = p.C + (long)z * p.M * p.ldc;
        const long row0 = (long)m_t * kBM + quarter * 32;
        const int col0 = n_t * kBN;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) stg[lane * 33 + i] = __uint_as_float(v[i]);
          __syncwarp();
          const int col = col0 + c * 32 + lane;
#pragma unroll 4
          for (int r = 0; r < 32; ++r) {
            const long row = row0 + r;
            if (row < p.M && col < p.N) Cz[row * p.ldc + col] = stg[r * 33 + lane];
          }
          __syncwarp();
        }
      } else if constexpr (kEpi == kEpiKvCache) {
        kv_cache_epilogue(p, tbase, m_t, n_t, quarter, lane);
      } else if constexpr (kEpi == kEpiCrossEntropy) {
        cross_entropy_epilogue(p, tbase, m_t, n_t, quarter, lane);
      } else if constexpr (kEpi == kEpiQkv) {
        qkv_epilogue(p, tbase, m_t, n_t, quarter, lane);
      } else if constexpr (kEpi == kEpiResidual) {
        residual_epilogue(p, tbase, m_t, n_t, quarter, lane);
      } else {
        swiglu_epilogue(p, tbase, m_t, n_t, quarter, lane);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair) mbar_arrive_cluster(tempty_leader + (uint32_t)(acc * 8));
        else mbar_arrive(&tempty[acc]);
      }
      if (++acc == 2) { acc = 0; acc_ph ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();  // the leader's MMAs into the peer's memory are done
  tc_fence_after();
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_dealloc_pair(tmem_base, kTmemCols);
    } else {
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                   "r"(kTmemCols)
                   : "memory");
    }
  }
  if (threadIdx.x == 0 && *abort_flag) report(p.status, kStatusTimeout, kKernGemmTc);
}

// ---- host side ------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D map of 16-bit elements (bf16 or fp16) over a [rows, cols] row-major matrix with row
// stride ld (elements), box = box_rows x 64 columns, 128-byte swizzle, zero fill out of
// bounds.
bool encode_kmajor(CUtensorMap* map, const void* base, long rows, int cols, long ld,
                   int box_rows, bool bf16) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

bool gemm_tc_supported(long M, int N, int K, long lda, long ldb) {
  return M >= 1 && N >= 1 && K >= 1 && lda % 8 == 0 && ldb % 8 == 0 && lda >= K && ldb >= K &&
         get_encode_fn() != nullptr;
}

namespace {

std::atomic<int> g_pair_mode{0};  // 0: CTA pairs from two M tiles up; 1: one CTA per tile

// CTA pairs the device can hold at once with this kernel's shared memory (once per kernel
// and device).
template <int kEpi>
int max_active_pairs() {
  static int cached[64] = {};  // per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 256);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<kEpi, 1>, &cfg) != cudaSuccess || n < 1)
    n = sm_count() / 2;
  cached[dev] = n;
  return n;
}

template <int kEpi>
cudaError_t launch_variant(const CUtensorMap& ma, const CUtensorMap& mb, const TcParams& p,
                           long units, bool pair, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<kEpi, 0>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_tc_kernel<kEpi, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (pair) {
    const long pairs = max_active_pairs<kEpi>();
    const int grid = 2 * (int)(units < pairs ? units : pairs);
    return launch_pdl_cluster(gemm_tc_kernel<kEpi, 1>, dim3(grid), dim3(kThreads), kSmemBytes,
                              stream, 2, ma, mb, p);
  }
  const int sms = sm_count();
  const int grid = (int)(units < sms ? units : sms);
  return launch_pdl(gemm_tc_kernel<kEpi, 0>, dim3(grid), dim3(kThreads), kSmemBytes, stream, ma,
                    mb, p);
}

cudaError_t launch_common(int elem, const void* A, long lda, const void* Bm, long ldb, float* C,
                          long ldc, long M, int N, int K, int splits, const int32_t* tile_list,
                          unsigned* status, int* splits_out, int epi, const KvCacheEpilogue* kv, const ActOut* act,
                          cudaStream_t stream, uint64_t wait_ns = kWaitLimitNs,
                          int test_withhold = 0, const CrossEntropyEpilogue* ce = nullptr,
                          const QkvEpilogue* qkv = nullptr, const uint8_t* row_valid = nullptr) {
  if (elem != DFLASH_DTYPE_BF16 && elem != DFLASH_DTYPE_F16) return cudaErrorInvalidValue;
  if (((uintptr_t)A | (uintptr_t)Bm) % 16 != 0) return cudaErrorInvalidValue;
  const bool bf16 = elem == DFLASH_DTYPE_BF16;
  CUtensorMap ma, mb;
  if (!encode_kmajor(&ma, A, M, K, lda, kBM, bf16)) return cudaErrorInvalidValue;
  if (!encode_kmajor(&mb, Bm, N, K, ldb, 128, bf16)) return cudaErrorInvalidValue;
  TcParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.m_tiles = (int)((M + kBM - 1) / kBM);
  p.n_tiles = (N + kBN - 1) / kBN;
  p.swiglu_I = 0;
  if (epi == kEpiSwiGLU) {  // N = 2I: one tile per 128 channels
    p.swiglu_I = N / 2;
    p.n_tiles = (p.swiglu_I + 127) / 128;
    p.act = *act;
  }
  p.num_kb = (K + kBK - 1) / kBK;
  if (splits < 1) splits = 1;
  if (splits > p.num_kb) splits = p.num_kb;
  p.kb_per_split = (p.num_kb + splits - 1) / splits;
  p.splits = (p.num_kb + p.kb_per_split - 1) / p.kb_per_split;  // no empty split
  p.splits_out = splits_out;
  p.sms = sm_count();
  p.C = C;
  p.ldc = ldc;
  p.tile_list = tile_list;
  // M tiles fastest when A is the smaller operand: the CTAs that share a B tile then run
  // in the same wave and read it once
  p.m_fastest = (double)M <= (double)N ? 1 : 0;
  p.idesc = idesc_16bit(bf16);
  p.idesc_pair = idesc_16bit(bf16, 2 * kBM);
  p.status = status;
  p.wait_ns = wait_ns;
  p.test_withhold = test_withhold;
  if (kv) p.kv = *kv;
  if (ce) p.ce = *ce;
  if (qkv) p.qkv = *qkv;
  p.row_valid = row_valid;
  // Two or more M tiles: CTA pairs (M = 256 MMAs, each CTA reading half of every B tile),
  // whose MMAs run at the tensor cores' full rate; the one-CTA kernel's A-and-B-from-shared-
  // memory MMA is bound by shared-memory operand reads.
  const bool pair = g_pair_mode.load() == 0 && p.m_tiles >= 2;
  const long m_units = pair ? (p.m_tiles + 1) / 2 : p.m_tiles;
  const long units = m_units * p.n_tiles * p.splits;
  if (epi == kEpiKvCache) return launch_variant<kEpiKvCache>(ma, mb, p, units, pair, stream);
  if (epi == kEpiCrossEntropy)
    return launch_variant<kEpiCrossEntropy>(ma, mb, p, units, pair, stream);
  if (epi == kEpiSwiGLU) return launch_variant<kEpiSwiGLU>(ma, mb, p, units, pair, stream);
  if (epi == kEpiQkv) return launch_variant<kEpiQkv>(ma, mb, p, units, pair, stream);
  if (epi == kEpiResidual) return launch_variant<kEpiResidual>(ma, mb, p, units, pair, stream);
  return launch_variant<kEpiStoreF32>(ma, mb, p, units, pair, stream);
}

}  // namespace

cudaError_t launch_gemm_tc(int elem, const void* A, long lda, const void* Bm, long ldb, float* C,
                           long ldc, long M, int N, int K, int splits, const int32_t* tile_list,
                           unsigned* status, cudaStream_t stream, int* splits_out) {
  return launch_common(elem, A, lda, Bm, ldb, C, ldc, M, N, K, splits, tile_list, status,
                       splits_out, kEpiStoreF32, nullptr, nullptr, stream);
}

cudaError_t launch_gemm_tc_swiglu(int elem, const void* A, long lda, const void* Bm, long ldb,
                                  long M, int I, int K, const int32_t* tile_list,
                                  const ActOut& act, unsigned* status, cudaStream_t stream) {
  if (I < 1) return cudaErrorInvalidValue;
  return launch_common(elem, A, lda, Bm, ldb, nullptr, 0, M, 2 * I, K, 1, tile_list, status,
                       nullptr,
                       kEpiSwiGLU, nullptr, &act, stream);
}

cudaError_t launch_gemm_tc_kv_cache(int elem, const void* A, long lda, const void* Bm, long ldb,
                                    long M, int N, int K, const int32_t* tile_list,
                                    const KvCacheEpilogue& kv, unsigned* status,
                                    cudaStream_t stream) {
  if (kv.layers < 1 || N != kv.layers * 2 * kv.Hkv * 128 || kv.L < 1 ||
      (kv.layers > 1 && kv.layer_elems < (long)2 * kv.Hkv * kv.L_cache * 128))
    return cudaErrorInvalidValue;
  if (((uintptr_t)kv.kv | (uintptr_t)kv.cos_t | (uintptr_t)kv.sin_t) % 16 != 0)
    return cudaErrorInvalidValue;
  return launch_common(elem, A, lda, Bm, ldb, nullptr, 0, M, N, K, 1, tile_list, status, nullptr,
                       kEpiKvCache, &kv, nullptr, stream);
}

cudaError_t launch_gemm_tc_cross_entropy(const void* A, long lda, const void* Bm, long ldb,
                                         long M, int V, int K, const int32_t* tile_list,
                                         const CrossEntropyEpilogue& ce, unsigned* status,
                                         cudaStream_t stream) {
  if (V < 1 || !ce.targets || !ce.part || !ce.target_logit) return cudaErrorInvalidValue;
  CrossEntropyEpilogue e = ce;
  e.V = V;
  return launch_common(DFLASH_DTYPE_BF16, A, lda, Bm, ldb, nullptr, 0, M, V, K, 1, tile_list,
                       status, nullptr, kEpiCrossEntropy, nullptr, nullptr, stream, kWaitLimitNs,
                       0, &e);
}

cudaError_t launch_gemm_tc_qkv(const void* A, long lda, const void* Bm, long ldb, long M, int N,
                               int K, const int32_t* tile_list, const QkvEpilogue& e,
                               unsigned* status, cudaStream_t stream) {
  if (e.Hq < 1 || e.Hkv < 1 || e.Hq % e.Hkv != 0 || N != (e.Hq + 2 * e.Hkv) * 128 || e.NS < 1 ||
      e.ns_pad < e.NS || M % e.NS != 0 || e.P < 1 || !e.pos || !e.valid || !e.q || !e.kb ||
      !e.vbt)
    return cudaErrorInvalidValue;
  if (((uintptr_t)e.q | (uintptr_t)e.kb | (uintptr_t)e.cos_t | (uintptr_t)e.sin_t) % 16 != 0)
    return cudaErrorInvalidValue;
  return launch_common(DFLASH_DTYPE_F16, A, lda, Bm, ldb, nullptr, 0, M, N, K, 1, tile_list,
                       status, nullptr, kEpiQkv, nullptr, nullptr, stream, kWaitLimitNs, 0,
                       nullptr, &e);
}

cudaError_t launch_gemm_tc_residual(const void* A, long lda, const void* Bm, long ldb, float* x,
                                    long ldx, long M, int N, int K, const int32_t* tile_list,
                                    const uint8_t* valid, unsigned* status, cudaStream_t stream) {
  if (!x || !valid || ldx < N || N % 32 != 0 || ldx % 4 != 0 || (uintptr_t)x % 16 != 0)
    return cudaErrorInvalidValue;
  return launch_common(DFLASH_DTYPE_F16, A, lda, Bm, ldb, x, ldx, M, N, K, 1, tile_list, status,
                       nullptr, kEpiResidual, nullptr, nullptr, stream, kWaitLimitNs, 0, nullptr,
                       nullptr, valid);
}

void set_gemm_tc_pairs(int mode) { g_pair_mode.store(mode); }

cudaError_t launch_gemm_tc_withheld(const void* A, long lda, const void* Bm, long ldb, float* C,
                                    long ldc, long M, int N, int K, uint64_t wait_ns,
                                    unsigned* status, cudaStream_t stream) {
  return launch_common(DFLASH_DTYPE_BF16, A, lda, Bm, ldb, C, ldc, M, N, K, 1, nullptr, status,
                       nullptr, kEpiStoreF32, nullptr, nullptr, stream, wait_ns, 1);
}

}  // namespace dflash

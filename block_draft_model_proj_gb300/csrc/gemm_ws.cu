// Weight-streaming projection GEMM of the draft layers on the 5th-generation tensor cores.
//
// C[z][t][n] (fp32) = sum over the K slice z of X[t][k] * W[n][k] for the token rows t of the
// active 128-row tiles, computed transposed: D[n][t] = W[n, :] X[t, :]^T with the weight rows
// as the MMA's M = 128 operand and up to 128 tokens (one 128-row token tile) as N.  This is
// the form of the draft layers' projections ("DFlash Draft Body", How It Works step 3: QKV,
// O, gate/up, down) in calls of up to 512 draft slots, against 4096 x 4096 .. 24576 x 4096
// weights.
//
//  * The weights arrive as bf16 (the model's own) or fp16 and are read from global memory
//    exactly as given: TMA brings a 128 x 128 tile (two 64-column boxes) into shared
//    memory, four converter warps
//    turn it into fp16 (round to nearest even; exact for bf16 values of magnitude in
//    [2^-14, 65504]) and store it into tensor memory, where the MMA reads its A operand
//    (tcgen05.mma ... kind::f16 with A in tensor memory).  No converted copy of the
//    weights ever exists in global memory.
//  * The activations X are fp16 (their 11 significant bits keep the body within its error
//    bound); TMA loads 128 x 128 tiles of the active token tiles only, one per unit, and the
//    MMA's N covers only the rows present (16 for a 16-token decode step).
//  * K is cut into `splits` slices when the (weight tile, token tile) units alone would
//    leave SMs idle.  The count is chosen on the device from the number of active token
//    tiles, written to *splits_out, and read by the kernel that sums the slices.
//  * Epilogues: fp32 slices; SiLU(gate) * up (weight rows of a tile interleaved gate / up,
//    so each pair of TMEM lanes holds one channel).
//
// Warp roles (448 threads, one CTA per SM, persistent): warp 0 TMA producers (lane 0 the
// weight ring, lane 1 the token ring); warp 1 MMA issuer; warps 2-9 converters in two
// groups of four that take alternate K-steps; warps 10-13 epilogue.  Shared memory holds
// two rings: weight tiles, freed as soon as the converters have read them, and token tiles,
// freed by the MMA.  A K-step is 128 wide (eight MMAs per barrier wait and per commit).
// Tensor memory holds two 128-column accumulators (the epilogue of one unit overlaps the next
// unit's MMAs) and a 4-slot ring of converted A tiles (64 columns each), so the conversion
// runs ahead of the MMA and the
// weight tiles' load-and-convert latency stays off the token ring.  The converters and the
// producers run ahead into the next unit while the epilogue drains.
// Every mbarrier wait is bounded
// in time; on expiry the CTA reports DFLASH_ERR_TIMEOUT, drains its own copies and MMAs,
// frees its tensor memory and exits.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace dflash {
namespace {

using namespace tc;

constexpr int kWM = 128;   // weight rows per unit (MMA M)
constexpr int kTT = 128;   // rows of a token tile, one per unit (MMA N <= 128)
constexpr int kBK = 128;   // K per stage: two boxes of 64 (a 128-byte swizzled row each)
constexpr int kBox = 64;   // K of one TMA box
constexpr int kMaxWStages = 6;  // weight ring
constexpr int kMaxXStages = 4;  // token ring
constexpr int kASlots = 4;  // converted A tiles in tensor memory (64 columns each)
constexpr int kThreads = 448;
constexpr uint32_t kWSub = 128 * kBox * 2;              // 16 KB: 128 weight rows x 64 K
constexpr uint32_t kWBytes = 2 * kWSub;                 // 32 KB weight stage
constexpr uint32_t kRingBytes = 196 * 1024;             // shared-memory ring budget
constexpr uint32_t kTmemCols = 512;                     // two accumulators 2 x 128, A ring 4 x 64
constexpr uint32_t kTmemAcc = 0, kTmemA = 256;
constexpr uint32_t kEpiBufFloats = 32 * 36;             // per epilogue warp: [32][32 + 4]
constexpr size_t kSmemBytes = 1024 + kRingBytes + 512 + 4 * kEpiBufFloats * sizeof(float);
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kMaxWStages % 2 == 0, "the converter groups need an even weight-stage count");
static_assert(kMaxXStages <= kASlots, "a token stage is released through the K-step barriers");
static_assert(kTmemA + kASlots * 64 <= kTmemCols, "tensor memory");

struct WsParams {
  long M;            // token rows of X (and C)
  int Nw;            // weight rows (output features)
  int K;
  int w_tiles;       // units along the weight rows
  int m_tiles;       // 128-row token tiles (all)
  int num_kb;
  int max_splits;
  int sms;
  const int32_t* tile_list;  // optional: [0] = count, [1..] = active token tiles
  int xrows;                 // rows of a token-tile load (128, or M rounded up to 16)
  int w_stages;              // weight ring stages (32 KB each)
  int x_stages;              // token ring stages
  uint32_t x_stage_bytes;    // token tile(s) of one K-step
  int* splits_out;           // optional: the split count chosen on the device
  int w_bf16;                // weights bf16 (converted here) or fp16
  int interleave;            // TMEM lane 2i <- weight row i, lane 2i+1 <- row 64 + i
  int epi;
  float* C;
  long ldc;
  int c_vec;         // C rows 16-byte aligned (ldc % 4 == 0, C 16-byte aligned)
  int act_vec;       // SwiGLU output rows 4-element aligned (I % 4 == 0, 8-byte base)
  ActOut act;        // kEpiSwiGLU
  int swiglu_I;
  unsigned* status;
};

enum : int { kEpiF32 = 0, kEpiSwiGLU = 1 };

struct Sched {
  int tiles;   // active token tiles (the units along the tokens)
  int splits;
  int per;     // K-steps per slice
  long units;
};

__device__ __forceinline__ Sched schedule(const WsParams& p) {
  Sched s;
  s.tiles = p.tile_list ? p.tile_list[0] : p.m_tiles;
  const long units1 = (long)p.w_tiles * s.tiles;
  s.splits = choose_splits(units1, p.num_kb, p.max_splits, p.sms);
  s.per = (p.num_kb + s.splits - 1) / s.splits;
  s.units = units1 * s.splits;
  return s;
}

// A unit: weight tile wt, token tile t0, K slice z.  The token tiles of one weight tile are
// consecutive so the CTAs that share a weight tile run together.  rows0: token rows present.
struct Unit {
  int wt, t0, z, rows0;
};

__device__ __forceinline__ Unit decode(const WsParams& p, const Sched& s, long u) {
  Unit x;
  const int pi = (int)(u % s.tiles);
  const long rest = u / s.tiles;
  x.wt = (int)(rest % p.w_tiles);
  x.z = (int)(rest / p.w_tiles);
  x.t0 = p.tile_list ? p.tile_list[1 + pi] : pi;
  x.rows0 = (int)min((long)kTT, p.M - (long)x.t0 * kTT);
  return x;
}

// MMA N of a unit: the rows present, rounded up to 16
__device__ __forceinline__ uint32_t unit_idesc(const Unit& x) {
  return idesc_f16(kWM, (x.rows0 + 15) & ~15);
}

// bf16 pair -> fp16 pair (round to nearest even); `mag` collects the largest bf16 magnitude
// bits of each half (a magnitude of 0x4780 or more, 65536 and up, leaves the fp16 range)
__device__ __forceinline__ uint32_t cvt_pair(uint32_t w, bool bf16, uint32_t& mag) {
  if (!bf16) return w;
  mag = __vmaxu2(mag, w & 0x7FFF7FFFu);
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---- epilogues ---------------------------------------------------------------------------
// The thread owns TMEM lane r (weight row of the unit) and reads the 128 token columns in
// chunks of 32.

__device__ __forceinline__ void epi_f32(const WsParams& p, uint32_t tacc, int wt, int tt, int rows,
                                        int z, int r, int lane, float* buf) {
  float* Cz = p.C + (long)z * p.M * p.ldc;
  const int n0 = wt * kWM + (r - lane);  // this warp's 32 weight rows start here
  const int n = n0 + lane;
  const bool n_ok = n < p.Nw;
  // 32 x 32 blocks turned through shared memory so each lane writes 16-byte pieces of token
  // rows (a warp store covers four rows of 128 bytes) instead of one float per token
  const bool vec = p.c_vec && n0 + 32 <= p.Nw;
#pragma unroll 1
  for (int c = 0; c * 32 < rows; ++c) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tacc + c * 32, v);
    const long t0 = (long)tt * kTT + c * 32;
    if (vec) {
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 32; ++j) buf[j * 36 + lane] = __uint_as_float(v[j]);
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int j = 4 * q + (lane >> 3);
        if (c * 32 + j < rows)
          *reinterpret_cast<float4*>(Cz + (t0 + j) * p.ldc + n0 + 4 * (lane & 7)) =
              *reinterpret_cast<const float4*>(buf + j * 36 + 4 * (lane & 7));
      }
      continue;
    }
    if (!n_ok) continue;
#pragma unroll 8
    for (int j = 0; j < 32; ++j)
      if (c * 32 + j < rows) Cz[(t0 + j) * p.ldc + n] = __uint_as_float(v[j]);
  }
}

// Lanes 2i / 2i+1 hold gate / up of channel wt*64 + i.  The pair trades halves so that the
// even lane forms tokens 0..15 and the odd lane tokens 16..31 of each chunk.
__device__ __forceinline__ void epi_swiglu(const WsParams& p, uint32_t tacc, int wt, int tt,
                                           int rows, int r, int lane, float* buf) {
  const int I = p.swiglu_I;
  const int ch = wt * 64 + (r >> 1);
  const int ch_w = wt * 64 + ((r - lane) >> 1);  // this warp's 16 channels start here
  const bool odd = lane & 1;
#pragma unroll 1
  for (int c = 0; c * 32 < rows; ++c) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(tacc + c * 32, v);
    const int j0 = c * 32 + (odd ? 16 : 0);
    const long t0 = (long)tt * kTT + j0;
    if (p.act_vec) {
      // [32 tokens][16 channels] through shared memory: each lane then writes runs of four
      // channels of one token
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float mine = __uint_as_float(odd ? v[j] : v[16 + j]);
        const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
        const float g = odd ? other : __uint_as_float(v[j]);
        const float u = odd ? __uint_as_float(v[16 + j]) : other;
        buf[((odd ? 16 : 0) + j) * 20 + (lane >> 1)] = g / (1.f + expf(-g)) * u;
      }
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int idx = q * 32 + lane;
        const int tok = idx >> 2, c4 = idx & 3;
        const int ch0 = ch_w + 4 * c4;
        if (c * 32 + tok < rows && ch0 < I)
          p.act.store4(((long)tt * kTT + c * 32 + tok) * I + ch0,
                       *reinterpret_cast<const float4*>(buf + tok * 20 + 4 * c4));
      }
      continue;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float mine = __uint_as_float(odd ? v[j] : v[16 + j]);
      const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
      const float g = odd ? other : __uint_as_float(v[j]);
      const float u = odd ? __uint_as_float(v[16 + j]) : other;
      if (ch < I && j0 + j < rows) p.act.store((t0 + j) * I + ch, g / (1.f + expf(-g)) * u);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_ws_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
               const WsParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int SW = p.w_stages, SX = p.x_stages;
  uint8_t* wring = smem;                                  // SW x 16 KB
  uint8_t* xring = smem + (size_t)SW * kWBytes;           // SX x x_stage_bytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRingBytes);
  uint64_t* wfull = bars;                   // weight tile landed
  uint64_t* wempty = wfull + kMaxWStages;   // converters done reading it
  uint64_t* xfull = wempty + kMaxWStages;   // token tiles landed
  uint64_t* afull = xfull + kMaxXStages;    // [4] converted A in tensor memory
  // [4] the MMAs of K-step i (counted over the CTA's whole schedule) are done: A slot i % 4
  // and token stage i % SX are free again (one commit per K-step serves both)
  uint64_t* aempty = afull + kASlots;
  uint64_t* tfull = aempty + kASlots;       // [2] accumulator ready
  uint64_t* tempty = tfull + 2;             // [2] accumulator drained
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* epi_buf = reinterpret_cast<float*>(smem + kRingBytes + 512);  // [4][kEpiBufFloats]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 4);
    }
    for (int s = 0; s < SX; ++s) {
      mbar_init(&xfull[s], 1);
    }
    for (int a = 0; a < kASlots; ++a) {
      mbar_init(&afull[a], 4);
      mbar_init(&aempty[a], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_w)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_x)) : "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // prologue done (barriers, tensor memory): wait for the predecessor grid's results, then
  // let the successor grid be scheduled
  pdl_wait();
  pdl_trigger();

  const Sched sc = schedule(p);
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.splits_out) *p.splits_out = sc.splits;
  // a token stage: the unit's token tile, one K-major operand of up to 128 rows per K box
  const uint32_t xsub_bytes = p.x_stage_bytes / 2;

  if (warp == 0) {
    if (lane < 2) {
      // ---------------- TMA producers: lane 0 weight tiles, lane 1 token tiles ----------------
      const bool is_w = lane == 0;
      const int S = is_w ? SW : SX;
      uint64_t* full = is_w ? wfull : xfull;
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      long n_issued = 0;
      for (long u = blockIdx.x; u < sc.units && ok; u += gridDim.x) {
        const Unit x = decode(p, sc, u);
        const int kb0 = x.z * sc.per, kb1 = min(p.num_kb, kb0 + sc.per);
        for (int kb = kb0; kb < kb1; ++kb) {
          // weight stage: the converters of its previous use are done; token stage: the MMAs
          // of K-step n_issued - SX are done (phase (n_issued - SX) / 8 of aempty)
          const bool freed =
              is_w ? mbar_wait(&wempty[stage], ph ^ 1u, abort_flag, kWaitLimitNs)
                   : (n_issued < S ||
                      mbar_wait(&aempty[(n_issued - S) % kASlots],
                                (uint32_t)(((n_issued - S) / kASlots) & 1), abort_flag, kWaitLimitNs));
          if (!freed) { ok = false; break; }
          if (is_w) {
            mbar_arrive_expect_tx(&full[stage], kWBytes);
            for (int h = 0; h < 2; ++h) {
              uint8_t* dst = wring + (size_t)stage * kWBytes + h * kWSub;
              const int k0 = kb * kBK + h * kBox;
              if (p.epi == kEpiSwiGLU) {  // 64 gate rows, then the 64 up rows of the same channels
                tma_load_2d(&map_w, &full[stage], dst, k0, x.wt * 64);
                tma_load_2d(&map_w, &full[stage], dst + kWSub / 2, k0, p.swiglu_I + x.wt * 64);
              } else {
                tma_load_2d(&map_w, &full[stage], dst, k0, x.wt * kWM);
              }
            }
          } else {
            mbar_arrive_expect_tx(&full[stage], p.x_stage_bytes);
            for (int h = 0; h < 2; ++h) {
              uint8_t* dst = xring + (size_t)stage * p.x_stage_bytes + h * xsub_bytes;
              const int k0 = kb * kBK + h * kBox;
              tma_load_2d(&map_x, &full[stage], dst, k0, x.t0 * kTT);
            }
          }
          ++n_issued;
          if (++stage == S) { stage = 0; ph ^= 1u; }
        }
      }
      // wait for this thread's own copies still in flight (the last S issued)
      for (long j = n_issued - S > 0 ? n_issued - S : 0; j < n_issued; ++j)
        mbar_drain_wait(&full[j % S], (uint32_t)((j / S) & 1), kWaitLimitNs / 4);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int stage = 0;  // token ring
      uint32_t ph = 0;
      long i = 0;  // K-step counter: A slot i % 8
      int acc = 0;  // two accumulators: the epilogue of one unit overlaps the next unit
      uint32_t acc_ph = 0;
      bool ok = true;
      for (long u = blockIdx.x; u < sc.units && ok; u += gridDim.x) {
        const Unit x = decode(p, sc, u);
        const int kb0 = x.z * sc.per, kb1 = min(p.num_kb, kb0 + sc.per);
        const uint32_t idesc = unit_idesc(x);
        if (!mbar_wait(&tempty[acc], acc_ph ^ 1u, abort_flag, kWaitLimitNs)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + kTmemAcc + (uint32_t)(acc * kTT);
        for (int kb = kb0; kb < kb1; ++kb, ++i) {
          const int slot = (int)(i % kASlots);
          if (!mbar_wait(&afull[slot], (uint32_t)((i / kASlots) & 1), abort_flag, kWaitLimitNs) ||
              !mbar_wait(&xfull[stage], ph, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem + kTmemA + (uint32_t)(slot * 64);
          // K = 16 per MMA: A columns 8k .. 8k+7 (packed pairs); token box k / 4, +32 bytes
          // inside it (the descriptor's address field counts 16-byte units)
          const uint64_t x_desc = sw128_desc(smem_u32(xring + (size_t)stage * p.x_stage_bytes));
          const uint64_t x_sub = xsub_bytes >> 4;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_f16_ts(d_tmem, a_tmem + k * 8, x_desc + (k >> 2) * x_sub + (uint64_t)((k & 3) * 2),
                        idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          umma_commit(&aempty[slot]);
          if (++stage == SX) { stage = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == 2) { acc = 0; acc_ph ^= 1u; }
      }
      umma_commit(drain);
      mbar_drain_wait(drain, 0, kWaitLimitNs / 4);
    }
  } else if (warp < 10) {
    // ---------------- converters (warps 2..9): W tile -> fp16 A in tensor memory ----------------
    // group g = 0 / 1 takes the K-steps with i % 2 == g; within a group, warp w covers TMEM
    // lane quarter w % 4
    const int group = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // TMEM lane = A row
    const int srow_inter = (r & 1) ? 64 + (r >> 1) : (r >> 1);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool wbf16 = p.w_bf16 != 0;
    uint32_t mag = 0;
    long i = 0;
    bool ok = true;
    for (long u = blockIdx.x; u < sc.units && ok; u += gridDim.x) {
      const Unit x = decode(p, sc, u);
      const bool inter = p.interleave != 0;
      const int srow = inter ? srow_inter : r;
      const int kb0 = x.z * sc.per, kb1 = min(p.num_kb, kb0 + sc.per);
      for (int kb = kb0; kb < kb1; ++kb, ++i) {
        if ((int)(i & 1) != group) continue;
        const int stage = (int)(i % SW);
        const int slot = (int)(i % kASlots);
        const bool got = mbar_wait(&wfull[stage], (uint32_t)((i / SW) & 1), abort_flag, kWaitLimitNs) &&
                         mbar_wait(&aempty[slot], (uint32_t)(((i / kASlots) & 1) ^ 1), abort_flag,
                                   kWaitLimitNs);
        if (!__all_sync(0xffffffffu, got ? 1 : 0)) { ok = false; break; }
        tc_fence_after();
        // row srow of each 128-byte-swizzled 64-K box: 16-byte chunk c at chunk position
        // c ^ (row % 8); box h lands in A columns [32h, 32h + 32) of the slot
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const uint8_t* row = wring + (size_t)stage * kWBytes + h * kWSub + (srow >> 3) * 1024 +
                               (srow & 7) * 128;
          uint32_t a[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 w = *reinterpret_cast<const uint4*>(row + ((c ^ (srow & 7)) * 16));
            a[4 * c] = cvt_pair(w.x, wbf16, mag);
            a[4 * c + 1] = cvt_pair(w.y, wbf16, mag);
            a[4 * c + 2] = cvt_pair(w.z, wbf16, mag);
            a[4 * c + 3] = cvt_pair(w.w, wbf16, mag);
          }
          if (h == 1) {
            // the weight stage is in registers: hand it back before the last tensor-memory store
            __syncwarp();
            if (lane == 0) mbar_arrive(&wempty[stage]);
          }
          tmem_st_32x32b_x32(tmem + kTmemA + (uint32_t)(slot * 64 + h * 32) + lane_off, a);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[slot]);
      }
    }
    if ((mag & 0xFFFFu) >= 0x4780u || (mag >> 16) >= 0x4780u)
      report(p.status, kStatusRange, kKernConvert);
  } else {
    // ---------------- epilogue (warps 10..13) ----------------
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int acc = 0;
    uint32_t acc_ph = 0;
    for (long u = blockIdx.x; u < sc.units; u += gridDim.x) {
      const Unit x = decode(p, sc, u);
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&tfull[acc], acc_ph, abort_flag, kWaitLimitNs) ? 1 : 0))
        break;
      tc_fence_after();
      const uint32_t tacc = tmem + kTmemAcc + (uint32_t)(acc * kTT) + lane_off;
      float* buf = epi_buf + (warp - 10) * kEpiBufFloats;
      if (p.epi == kEpiF32) epi_f32(p, tacc, x.wt, x.t0, x.rows0, x.z, r, lane, buf);
      else epi_swiglu(p, tacc, x.wt, x.t0, x.rows0, r, lane, buf);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) { acc = 0; acc_ph ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && *abort_flag) report(p.status, kStatusTimeout, kKernGemmTc);
}

// ---- host side ------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// [rows, cols] row-major 16-bit matrix, row stride ld elements; box = box_rows x 64 columns,
// 128-byte swizzle, zero fill out of bounds
bool encode_rows(CUtensorMap* map, const void* base, long rows, int cols, long ld, int box_rows,
                 bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBox, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

cudaError_t launch(const WsArgs& a, int epi, int w_tiles, int interleave, const ActOut* act,
                   cudaStream_t stream) {
  if (a.w_dtype != DFLASH_DTYPE_BF16 && a.w_dtype != DFLASH_DTYPE_F16) return cudaErrorInvalidValue;
  if (((uintptr_t)a.X | (uintptr_t)a.W) % 16 != 0 || a.ldx % 8 != 0 || a.ldw % 8 != 0 ||
      a.K < 1 || a.M < 1 || a.Nw < 1)
    return cudaErrorInvalidValue;
  CUtensorMap mw, mx;
  const int wbox = epi == kEpiSwiGLU ? 64 : kWM;
  if (!encode_rows(&mw, a.W, a.Nw, a.K, a.ldw, wbox, a.w_dtype == DFLASH_DTYPE_BF16))
    return cudaErrorInvalidValue;
  // token-tile loads: 128 rows, or all M rows (rounded up to 16) when M <= 128
  const int xrows = a.M > kTT ? kTT : (int)((a.M + 15) / 16 * 16);
  if (!encode_rows(&mx, a.X, a.M, a.K, a.ldx, xrows, false)) return cudaErrorInvalidValue;
  WsParams p;
  p.M = a.M;
  p.Nw = a.Nw;
  p.K = a.K;
  p.w_tiles = w_tiles;
  p.m_tiles = (int)((a.M + kTT - 1) / kTT);
  p.num_kb = (a.K + kBK - 1) / kBK;
  p.max_splits = epi == kEpiF32 ? (a.max_splits < 1 ? 1 : a.max_splits) : 1;
  p.sms = sm_count();
  p.tile_list = a.tile_list;
  p.xrows = xrows;
  p.x_stage_bytes = (uint32_t)xrows * kBK * 2;
  // tokens: 4 stages when they are small (decode), else 2; the weights take the rest
  p.x_stages = p.x_stage_bytes <= 16384 ? kMaxXStages : 2;
  p.w_stages = (int)((kRingBytes - (uint32_t)p.x_stages * p.x_stage_bytes) / kWBytes);
  if (p.w_stages > kMaxWStages) p.w_stages = kMaxWStages;
  // the two converter groups take alternate K-steps: with an even stage count every stage
  // stays with one group (step i and step i + w_stages have the same parity), so a group can
  // never mistake the other group's phase of a stage for its own
  p.w_stages &= ~1;
  if (p.w_stages < 2) return cudaErrorInvalidValue;
  p.splits_out = a.splits_out;
  p.w_bf16 = a.w_dtype == DFLASH_DTYPE_BF16;
  p.interleave = interleave;
  p.epi = epi;
  p.C = a.C;
  p.ldc = a.ldc;
  p.c_vec = (a.ldc % 4 == 0) && ((uintptr_t)a.C % 16 == 0);
  if (act) p.act = *act;
  p.swiglu_I = epi == kEpiSwiGLU ? a.Nw / 2 : 0;
  p.act_vec = act && p.swiglu_I % 4 == 0 && ((uintptr_t)act->p % 16 == 0);
  p.status = a.status;
  // enough CTAs for the largest schedule the device can pick (all token tiles active)
  long max_units = 0;
  for (int s = 1; s <= p.max_splits; ++s) {
    const long u = (long)w_tiles * p.m_tiles * s;
    if (u > max_units) max_units = u;
  }
  const int grid = (int)(max_units < p.sms ? max_units : p.sms);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(gemm_ws_kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, mw, mx, p);
}

}  // namespace

int gemm_ws_splits(long units1, int K, int max_splits) {
  return choose_splits(units1, (K + kBK - 1) / kBK, max_splits, sm_count());
}

cudaError_t launch_gemm_ws(const WsArgs& a, cudaStream_t stream) {
  return launch(a, kEpiF32, (a.Nw + kWM - 1) / kWM, 0, nullptr, stream);
}

cudaError_t launch_gemm_ws_swiglu(const WsArgs& a, const ActOut& act, cudaStream_t stream) {
  if (a.Nw % 2 != 0) return cudaErrorInvalidValue;
  // a unit covers 64 channels: its 64 gate rows and the 64 up rows of the same channels
  // (rows past 2I read as zeros; channels past I are not stored)
  return launch(a, kEpiSwiGLU, (a.Nw / 2 + 63) / 64, 1, &act, stream);
}

}  // namespace dflash

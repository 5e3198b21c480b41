// Anchored block-sparse dual-source attention on the 5th-generation tensor cores.
//
// "DFlash Draft Body", How It Works step 3: within a layer each block reads the target
// prefix before its anchor and all positions of the same block, never another block, and
// the target sequence is not updated.  "DFlash" (How it works): the target's projected K/V
// are attended alongside the draft tokens' own K/V.  "DFlash: drafting, verification, and
// speed" (One DFlash generation cycle): a block must not read target features containing
// its future answers, hence the strict prefix c < anchor.
//
// Key set of a valid slot of block (b, k), anchor a: context positions c < min(a, L) with
// mask[b, c] != 0, plus every valid slot of block (b, k).  GQA: query head h reads KV head
// h / (Hq / Hkv).  Excluded keys are removed by selection (never by an additive -inf), and
// value columns past the last readable key are zeroed in shared memory, so nothing beyond
// a block's prefix -- not even a non-finite value -- can reach its output.
//
// Work unit = (row b, KV head g, query tile t, key chunk c).  A query tile packs the
// S x (Hq/Hkv) query rows of 128 / (S * Hq/Hkv) consecutive blocks of (b, g) into the 128
// lanes of an M = 128 MMA; consecutive blocks have nearby anchors (the plan sorts them), so
// one key range serves the whole tile and per-row anchors only mask the tail.  The prefix is
// cut into chunks of `chunk` keys so long prefixes spread over many SMs; chunk 0 also takes
// the tile's own-block keys.  Each unit writes an unnormalised partial (m, l, O) per row;
// attn_combine_kernel merges the chunks of a tile in chunk order (deterministic) and writes
// the attention output (fp16) for the O projection.
//
// Arithmetic: kind::f16 MMAs with fp32 accumulation.  Q, the block K/V and the context K/V
// cache are fp16 (11 significant bits, as many as tf32), P is rounded to fp16; the softmax
// runs in fp32 in registers (one TMEM lane = one query row per thread), base-2 exponent,
// with a lazily updated running maximum (the accumulator is rescaled only when the maximum
// grows by more than 2^8, so P stays <= 256).
//
// Key tiles are 128 keys.  Tensor memory holds the O accumulator [0,128) and three S/P
// buffers [128,256), [256,384), [384,512) (S = Q K^T lands there; each softmax warp
// overwrites the first half of its own 64 S columns with its packed fp16 P, and O += P V
// reads P from there).  Shared memory holds Q (TMA, once per unit), a 3-stage K ring and a
// 2-stage V^T ring of 32 KB stages.
// Warp roles: warp 0 TMA producers (lane 0 Q and the K ring, lane 1 the V^T ring); warp 1
// MMA issuer, one thread, in a fixed order (S of the tile three ahead right behind each PV);
// warps 2-9 softmax / correction / partial output: two warps per TMEM lane quarter, one per
// half of the key columns (and of the O columns), so each SM sub-partition runs two softmax
// warps; the halves agree on the running row maximum through shared memory behind an
// mbarrier per lane quarter.  A half tile whose 64 mask bytes are all set takes a short path
// (one warp vote over its 16 mask words), and P = 2^(x * scale - m) is one FMA into the
// special-function unit's exponential (an excluded key gives exactly 0).  Every mbarrier
// wait is bounded in time; on expiry the CTA reports DFLASH_ERR_TIMEOUT, drains its own
// copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace dflash {

namespace {

using namespace tc;

constexpr int kDH = 128;   // head dim handled by this kernel
constexpr int kM = 128;    // query rows per tile (TMEM lanes)
constexpr int kKT = 128;   // keys per tile (the N of the S MMA)
constexpr int kRingK = 3;  // stages of the K ring
constexpr int kRingV = 2;  // stages of the V^T ring
constexpr int kSP = 3;     // S/P buffers in tensor memory
static_assert(kSP == kRingK, "S(i) completing frees K stage i % kRingK and S buffer i % kSP");
constexpr int kThreads = 320;          // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr int kSoftmaxWarps = 8;       // two per TMEM lane quarter, each owns half the keys
constexpr int kHalfKT = 64;            // key columns per softmax thread
constexpr uint32_t kTmemCols = 512;    // O [0,128), S/P 3 x 128 [128,512)
constexpr uint32_t kTmemO = 0, kTmemS = 128;
constexpr uint32_t kKSub = kKT * 64 * 2;   // K [128 keys][64 dh] fp16, 16 KB
constexpr uint32_t kKBytes = 2 * kKSub;    // 32 KB
constexpr uint32_t kVSub = kDH * 64 * 2;   // V^T [128 dh][64 keys] fp16, 16 KB
constexpr uint32_t kVBytes = 2 * kVSub;    // 32 KB
constexpr uint32_t kQBytes = 2 * kKSub;   // Q [128 rows][64 dh] x 2 fp16, 32 KB
constexpr uint32_t kBarBytes = 512;
// K ring + V ring + Q + barriers + row-max exchange [2][2][128] + row-sum exchange [2][128]
constexpr size_t kSmemBytes = 1024 + kRingK * (size_t)kKBytes + kRingV * (size_t)kVBytes +
                              kQBytes + kBarBytes + (4 * 128 + 2 * 128) * sizeof(float);
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
constexpr uint32_t kIdescS = idesc_f16(kM, kKT);
constexpr uint32_t kIdescPV = idesc_f16(kM, kDH);
constexpr float kRescaleLog2 = 8.0f;

struct AttnTcParams {
  int B, N, S, L, Hkv, grp, R, bpt, tiles, chunk, max_chunks;
  const __half* q;  // [B][Hkv][N][S][grp][dh]
  long q_rows;
  const int32_t* anchors;
  const uint8_t* valid;
  const uint8_t* mask;
  float* part_o;  // [units][128][128]
  float* part_m;  // [units][128]
  float* part_l;  // [units][128]
  unsigned* status;
  float scale_log2;
  int direct;   // one key chunk: the unit normalises and writes the output rows itself
  int Hq;
  ActOut out;   // [T][Hq*dh], written directly when `direct`
};

struct UnitInfo {
  int b, g, t, c, k0, k1, a_max, cs, ce, nblk, n;
};

__device__ __forceinline__ UnitInfo decode_unit(const AttnTcParams& p, int unit) {
  UnitInfo u;
  u.c = unit % p.max_chunks;
  int rest = unit / p.max_chunks;
  u.t = rest % p.tiles;
  rest /= p.tiles;
  u.g = rest % p.Hkv;
  u.b = rest / p.Hkv;
  u.k0 = u.t * p.bpt;
  u.k1 = min(p.N, u.k0 + p.bpt);
  int amax = 0;
  for (int k = u.k0; k < u.k1; ++k) {
    const int a = p.anchors[u.b * p.N + k];
    if (a > amax) amax = a;
  }
  u.a_max = min(amax, p.L);
  u.cs = u.c * p.chunk;
  u.ce = min(u.cs + p.chunk, u.a_max);
  // chunk 0 also takes the tile's own-block keys: bpt * S of them, in tiles of kKT
  u.nblk = u.c == 0 ? (p.bpt * p.S + kKT - 1) / kKT : 0;
  const int nctx = u.ce > u.cs ? (u.ce - u.cs + kKT - 1) / kKT : 0;
  u.n = u.nblk + nctx;
  return u;
}

__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap map_kc, const __grid_constant__ CUtensorMap map_vc,
               const __grid_constant__ CUtensorMap map_kb, const __grid_constant__ CUtensorMap map_vb,
               const __grid_constant__ CUtensorMap map_q, const AttnTcParams p) {
  pdl_wait();
  const UnitInfo u = decode_unit(p, blockIdx.x);
  if (u.n == 0) return;  // a chunk past this tile's longest prefix: no work

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sK = smem;                        // K ring: stage s at s * kKBytes
  uint8_t* sV = sK + kRingK * kKBytes;       // V^T ring: stage s at s * kVBytes
  uint8_t* sQ = sV + kRingV * kVBytes;       // Q of the tile: two [128 rows][64 dh] boxes
  uint64_t* bars = reinterpret_cast<uint64_t*>(sQ + kQBytes);
  uint64_t* k_full = bars;
  uint64_t* v_full = k_full + kRingK;
  uint64_t* v_empty = v_full + kRingV;
  uint64_t* s_full = v_empty + kRingV;
  uint64_t* p_full = s_full + kSP;
  uint64_t* q_full = p_full + kSP;
  uint64_t* drain = q_full + 1;
  // row-max exchange between the two warps of a TMEM lane quarter: [quarter][tile parity]
  uint64_t* max_bar = drain + 1;
  uint64_t* sum_bar = max_bar + 8;  // [quarter]: row-sum exchange at the end
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sum_bar + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red_max = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + kBarBytes);  // [2][2][128]
  float* red_sum = red_max + 4 * 128;                                                       // [2][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s2 = 0; s2 < kRingK; ++s2) {
      mbar_init(&k_full[s2], 1);
    }
    for (int s2 = 0; s2 < kRingV; ++s2) {
      mbar_init(&v_full[s2], 1);
      mbar_init(&v_empty[s2], 1);
    }
    for (int i = 0; i < kSP; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftmaxWarps);
    }
    mbar_init(q_full, 1);
    mbar_init(drain, 1);
    for (int i = 0; i < 8; ++i) mbar_init(&max_bar[i], 2);
    for (int i = 0; i < 4; ++i) mbar_init(&sum_bar[i], 2);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the successor grid may be scheduled once this CTA holds its tensor memory
  pdl_trigger();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + kTmemO, tmem_s0 = tmem + kTmemS;

  const int planes_per_b = 2 * p.Hkv;
  const int plane_k = u.b * planes_per_b + u.g;
  const int plane_v = u.b * planes_per_b + p.Hkv + u.g;

  if (warp == 0) {
    // ---------------- TMA producers: lane 0 = Q, then the K ring; lane 1 = the V^T ring ----------------
    // Q is two [128 rows][64 dh] boxes, a K tile two [128 keys][64 dh] boxes (the two halves
    // of dh), a V^T tile two [128 dh][64 keys] boxes (the two halves of the keys), each
    // 128-byte swizzled.
    if (lane < 2) {
      const bool is_k = lane == 0;
      const int ring = is_k ? kRingK : kRingV;
      uint64_t* full = is_k ? k_full : v_full;
      // a K stage is free once the S MMAs that read it have completed: the K ring and the S
      // buffers have the same depth, so that is the previous phase of s_full of the same index
      uint64_t* empty = is_k ? s_full : v_empty;
      if (is_k) {
        const int qrow0 = ((u.b * p.Hkv + u.g) * p.N + u.k0) * p.R;
        mbar_arrive_expect_tx(q_full, kQBytes);
        for (int h = 0; h < 2; ++h) tma_load_2d(&map_q, q_full, sQ + h * kKSub, h * 64, qrow0);
      }
      int issued[kRingK] = {0, 0, 0};
      uint32_t issued_ph[kRingK] = {0, 0, 0};
      for (int i = 0; i < u.n; ++i) {
        const int st = i % ring;
        const uint32_t ph = (uint32_t)(i / ring) & 1u;
        if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, kWaitLimitNs)) break;
        if (is_k) {
          mbar_arrive_expect_tx(&full[st], kKBytes);
          uint8_t* dst = sK + st * kKBytes;
          if (i < u.nblk) {
            const int kbrow0 = ((u.b * p.Hkv + u.g) * p.N + u.k0) * p.S + i * kKT;
            for (int q = 0; q < 2; ++q) tma_load_2d(&map_kb, &full[st], dst + q * kKSub, q * 64, kbrow0);
          } else {
            const int c0 = u.cs + (i - u.nblk) * kKT;
            for (int q = 0; q < 2; ++q) tma_load_3d(&map_kc, &full[st], dst + q * kKSub, q * 64, c0, plane_k);
          }
        } else {
          mbar_arrive_expect_tx(&full[st], kVBytes);
          uint8_t* dst = sV + st * kVBytes;
          if (i < u.nblk) {
            for (int h = 0; h < 2; ++h)
              tma_load_2d(&map_vb, &full[st], dst + h * kVSub, u.k0 * p.S + i * kKT + 64 * h,
                          (u.b * p.Hkv + u.g) * kDH);
          } else {
            for (int h = 0; h < 2; ++h)
              tma_load_3d(&map_vc, &full[st], dst + h * kVSub, u.cs + (i - u.nblk) * kKT + 64 * h, 0,
                          plane_v);
          }
        }
        issued[st] = 1;
        issued_ph[st] = ph;
      }
      for (int s2 = 0; s2 < ring; ++s2)
        if (issued[s2]) mbar_drain_wait(&full[s2], issued_ph[s2], kWaitLimitNs / 4);
      if (is_k) mbar_drain_wait(q_full, 0, kWaitLimitNs / 4);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      // A fixed order with blocking waits: S(0), S(1), S(2); then per tile i: O += P_i V_i
      // once the softmax has written P_i and V_i has landed, followed at once by S(i + 3) into
      // the buffer P_i occupied.  The tensor core performs one thread's MMAs in issue order, so
      // S(i + 3) overwrites that buffer only after PV(i) has read it; with three buffers the
      // chain softmax(i) -> PV(i) -> S(i + 3) -> softmax(i + 3) spans the softmax of two other
      // tiles.  The MMAs of a group are issued back to back (unrolled, descriptors formed
      // from one base: the address field counts 16-byte units), one commit per group:
      // PV(i)'s completion (v_empty) frees V stage i and tells the softmax the accumulator is
      // up to date; S's (s_full) hands the scores to the softmax, whose first reader frees the
      // K stage.
      bool ok = mbar_wait(q_full, 0, abort_flag, kWaitLimitNs);
      tc_fence_after();
      const uint64_t q_desc = sw128_desc(smem_u32(sQ));
      auto issue_s = [&](int s) -> bool {
        if (!mbar_wait(&k_full[s % kRingK], (uint32_t)(s / kRingK) & 1u, abort_flag, kWaitLimitNs))
          return false;
        tc_fence_after();
        const uint64_t k_desc = sw128_desc(smem_u32(sK + (s % kRingK) * kKBytes));
        const uint32_t s_tmem = tmem_s0 + (uint32_t)((s % kSP) * kKT);
        // K = 16 dh per MMA: Q and K sub-tile k / 4, +32 bytes inside it
#pragma unroll
        for (int k = 0; k < kDH / 16; ++k) {
          const uint64_t off = (uint64_t)(((k >> 2) * kKSub + (k & 3) * 32) >> 4);
          umma_f16_ss(s_tmem, q_desc + off, k_desc + off, kIdescS, k ? 1u : 0u);
        }
        umma_commit(&s_full[s % kSP]);
        return true;
      };
      for (int s = 0; s < kSP && s < u.n && ok; ++s) ok = issue_s(s);
      for (int i = 0; i < u.n && ok; ++i) {
        ok = mbar_wait(&p_full[i % kSP], (uint32_t)(i / kSP) & 1u, abort_flag, kWaitLimitNs) &&
             mbar_wait(&v_full[i % kRingV], (uint32_t)(i / kRingV) & 1u, abort_flag, kWaitLimitNs);
        if (!ok) break;
        tc_fence_after();
        const uint64_t v_desc = sw128_desc(smem_u32(sV + (i % kRingV) * kVBytes));
        const uint32_t a_base = tmem_s0 + (uint32_t)((i % kSP) * kKT);
        // K = 16 keys per MMA: P of keys 16k .. 16k+15 sits at columns 64 * (k / 4) +
        // 8 * (k % 4) of the buffer (each softmax half packs its 64 keys into the first 32 of
        // its own 64 S columns); V^T sub-tile k / 4, +32 bytes per 16 keys inside it
        const uint32_t first = i == 0 ? 0u : 1u;
#pragma unroll
        for (int k = 0; k < kKT / 16; ++k)
          umma_f16_ts(tmem_o, a_base + (k >> 2) * 64 + (k & 3) * 8,
                      v_desc + (uint64_t)(((k >> 2) * kVSub + (k & 3) * 32) >> 4), kIdescPV,
                      k == 0 ? first : 1u);
        umma_commit(&v_empty[i % kRingV]);
        if (i + kSP < u.n) ok = issue_s(i + kSP);
      }
      umma_commit(drain);
      mbar_drain_wait(drain, 0, kWaitLimitNs / 4);
    }
  } else {
    // ---------------- softmax / correction / partial output (warps 2..9) ----------------
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;   // key columns [64*half, 64*half + 64) of each tile
    const int r = quarter * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int kbo = r / p.R;
    const int within = r - kbo * p.R;
    const int j = within / p.grp;
    const int kb = u.k0 + kbo;
    bool row_valid = false;
    int a_row = 0;
    if (kb < u.k1) {
      const int a = p.anchors[u.b * p.N + kb];
      row_valid = a >= 0 && p.valid[(u.b * p.N + kb) * p.S + j] != 0;
      a_row = min(max(a, 0), p.L);
    }
    const uint8_t* mrow = p.mask + (size_t)u.b * p.L;
    float m_run = -INFINITY, l_run = 0.f;  // l_run: this half's share of the row sum
    bool ok = true;
    // every wait result is made warp-uniform: the tcgen05.ld / st below are .sync.aligned
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, kWaitLimitNs) ? 1 : 0) != 0;
    };
    // context mask words of this half of a tile (the same for every row of the unit): lane
    // w < 16 loads word w one tile ahead, so the global-memory latency is off the softmax's
    // critical path; the words are broadcast by shuffles where they are used.  Words past
    // the chunk read as 0; the row's own prefix limit is applied at use.
    auto load_mask = [&](int i) -> uint32_t {
      const int c = u.cs + (i - u.nblk) * kKT + half * kHalfKT + 4 * lane;
      return (lane < kHalfKT / 4 && i >= u.nblk && i < u.n && c < u.ce)
                 ? __ldg(reinterpret_cast<const uint32_t*>(mrow + c)) : 0u;
    };
    uint32_t mword_next = load_mask(0);
    for (int i = 0; i < u.n && ok; ++i) {
      const uint32_t mword = mword_next;
      mword_next = load_mask(i + 1);
      if (!wait_all(&s_full[i % kSP], (uint32_t)(i / kSP) & 1u)) { ok = false; break; }
      tc_fence_after();
      const uint32_t s_tmem = tmem_s0 + (uint32_t)((i % kSP) * kKT + half * kHalfKT) + lane_off;
      uint32_t sv[kHalfKT];
      tmem_ld_32x32b_x32_nowait(s_tmem, sv);
      tmem_ld_32x32b_x32_nowait(s_tmem + 32, sv + 32);
      tmem_wait_ld();
      const bool blk_tile = i < u.nblk;
      const int c0 = blk_tile ? 0 : u.cs + (i - u.nblk) * kKT + half * kHalfKT;
      // Readable keys keep their raw score, the others become -inf (selection); the scale
      // 1/sqrt(dh) * log2(e) is applied later inside the exponent's FMA.
      float mh = -INFINITY;
      if (!row_valid) {
#pragma unroll
        for (int kk = 0; kk < kHalfKT; ++kk) sv[kk] = __float_as_uint(-INFINITY);
      } else if (blk_tile) {
        // own-block keys: column kk of this half is slot kk - off of this row's block,
        // readable when that slot is valid
        const int off = kbo * p.S - i * kKT - half * kHalfKT;
        const int j0 = max(0, -off), j1 = min(p.S, kHalfKT - off);
        uint64_t bm = 0;
        const uint8_t* vrow = p.valid + (size_t)(u.b * p.N + kb) * p.S;
        for (int jj = j0; jj < j1; ++jj)
          if (vrow[jj]) bm |= 1ull << (jj + off);
#pragma unroll
        for (int kk = 0; kk < kHalfKT; ++kk) {
          const float v = ((bm >> kk) & 1ull) ? __uint_as_float(sv[kk]) : -INFINITY;
          sv[kk] = __float_as_uint(v);
          mh = fmaxf(mh, v);
        }
      }
      if (!blk_tile) {
        // context keys c0 .. c0 + 63.  Warp-uniform test: no zero byte in the 16 mask words of
        // this half tile (words past the chunk read as 0).  Then a row only cuts at its own
        // prefix limit; otherwise every key is tested against its mask byte.
        const bool word_ok = lane >= kHalfKT / 4 ||
                             ((mword - 0x01010101u) & ~mword & 0x80808080u) == 0u;
        const bool mask_full = __all_sync(0xffffffffu, word_ok);
        if (mask_full) {
          if (!row_valid) {
          } else if (c0 + kHalfKT <= a_row) {
#pragma unroll
            for (int kk = 0; kk < kHalfKT; kk += 8) {  // eight independent chains
              float m8 = __uint_as_float(sv[kk]);
#pragma unroll
              for (int e = 1; e < 8; ++e) m8 = fmaxf(m8, __uint_as_float(sv[kk + e]));
              mh = fmaxf(mh, m8);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < kHalfKT; ++kk) {
              const float v = c0 + kk < a_row ? __uint_as_float(sv[kk]) : -INFINITY;
              sv[kk] = __float_as_uint(v);
              mh = fmaxf(mh, v);
            }
          }
        } else {
          // mask word w4 from lane w4 to every lane (all lanes take part in the shuffle)
#pragma unroll
          for (int w4 = 0; w4 < kHalfKT / 4; ++w4) {
            const uint32_t mw = __shfl_sync(0xffffffffu, mword, w4);
            if (!row_valid) continue;
            const int c = c0 + 4 * w4;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int kk = 4 * w4 + e;
              const bool okk = ((mw >> (8 * e)) & 0xFFu) != 0 && c + e < a_row && c + e < u.ce;
              const float v = okk ? __uint_as_float(sv[kk]) : -INFINITY;
              sv[kk] = __float_as_uint(v);
              mh = fmaxf(mh, v);
            }
          }
        }
      }
      // the two halves of a row agree on the tile maximum
      float* xm = red_max + (i & 1) * 256;
      xm[half * 128 + r] = mh;
      __syncwarp();
      if (lane == 0) mbar_arrive(&max_bar[quarter * 2 + (i & 1)]);
      if (!wait_all(&max_bar[quarter * 2 + (i & 1)], (uint32_t)(i >> 1) & 1u)) { ok = false; break; }
      const float mt = fmaxf(mh, xm[(1 - half) * 128 + r]) * p.scale_log2;  // -inf stays
      // running maximum: taken as is the first time a row sees a key, otherwise kept
      // unless the tile's maximum exceeds it by more than 2^8 (then the accumulator and
      // the row sum are rescaled)
      float factor = 1.f;
      if (mt > m_run) {
        if (m_run == -INFINITY) {
          m_run = mt;
        } else if (mt > m_run + kRescaleLog2) {
          factor = exp2f(m_run - mt);
          m_run = mt;
        }
      }
      l_run *= factor;
      // P = 2^(x - m): an excluded key (x = -inf) gives exactly +0; a row that has not seen
      // a readable key yet (m_run = -inf) has only excluded keys here.  Packed as fp16 pairs
      // into the first 32 of this half's 64 S columns.
      // four partial row sums (independent addition chains)
      float lsum4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pw[kHalfKT / 2];
      if (m_run == -INFINITY) {
#pragma unroll
        for (int kk = 0; kk < kHalfKT / 2; ++kk) pw[kk] = 0u;
      } else {
#pragma unroll
        for (int kk = 0; kk < kHalfKT / 2; ++kk) {
          const float x0 = fmaf(__uint_as_float(sv[2 * kk]), p.scale_log2, -m_run);
          const float x1 = fmaf(__uint_as_float(sv[2 * kk + 1]), p.scale_log2, -m_run);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          lsum4[kk & 3] += p0 + p1;
          const __half2 h2 = __floats2half2_rn(p0, p1);
          pw[kk] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      l_run += (lsum4[0] + lsum4[1]) + (lsum4[2] + lsum4[3]);
      tmem_st_32x32b_x32(s_tmem, pw);
      // the accumulator is rescaled before PV(i) (released below) adds to it; PV(i - 1)
      // must have landed first (a finite m_run means there was an earlier tile; its
      // completion is the phase of v_empty that frees its V stage).  This half rescales O
      // columns [64*half, 64*half + 64).
      if (__any_sync(0xffffffffu, factor != 1.f)) {
        if (!wait_all(&v_empty[(i - 1) % kRingV], (uint32_t)((i - 1) / kRingV) & 1u)) { ok = false; break; }
        tc_fence_after();
        for (int part = 0; part < 2; ++part) {
          uint32_t ov[32];
          const uint32_t oa = tmem_o + lane_off + half * 64 + part * 32;
          tmem_ld_32x32b_x32(oa, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * factor);
          tmem_st_32x32b_x32(oa, ov);
        }
      }
      tmem_wait_st();
      // value columns past the last readable key of this tile: zero them (this thread owns
      // V^T row r of key sub-tile `half`) so that whatever the cache holds there cannot
      // meet a zero P as NaN
      if (!blk_tile && u.cs + (i - u.nblk) * kKT + kKT > u.a_max) {
        const int st = i % kRingV;
        if (!wait_all(&v_full[st], (uint32_t)(i / kRingV) & 1u)) { ok = false; break; }
        const int nvalid = u.a_max - (u.cs + (i - u.nblk) * kKT) - half * kHalfKT;
        // row r of a swizzled [128][64] fp16 sub-tile: 16-byte chunk c (keys 8c .. 8c+7)
        // sits at chunk position c ^ (r % 8)
        uint8_t* rowp = sV + st * kVBytes + half * kVSub + (r >> 3) * 1024 + (r & 7) * 128;
        for (int c = 0; c < 8; ++c) {
          const int key0 = c * 8;
          if (key0 + 8 <= nvalid) continue;
          uint4* dst = reinterpret_cast<uint4*>(rowp + ((c ^ (r & 7)) * 16));
          uint4 val = *dst;
          uint32_t wv[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k0 = key0 + 2 * e;  // keys k0 (low half) and k0 + 1 (high half)
            if (k0 >= nvalid) wv[e] = 0u;
            else if (k0 + 1 >= nvalid) wv[e] &= 0xFFFFu;
          }
          *dst = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[i % kSP]);
    }
    // final accumulator: with one key chunk, O / l straight to the output rows; otherwise a
    // partial (m, l, O) of this unit.  Each half handles its 64 columns.  Every MMA of the
    // unit has completed once the issuer's final commit (drain) has landed.
    const bool fin = ok && wait_all(drain, 0);
    if (fin && p.direct) {
      tc_fence_after();
      red_sum[half * 128 + r] = l_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sum_bar[quarter]);
      const bool sum_ok = wait_all(&sum_bar[quarter], 0);
      const float l = l_run + red_sum[(1 - half) * 128 + r];
      // invalid slots of an existing block get exact zeros (the O projection reads them)
      const float inv = sum_ok && row_valid && l > 0.f ? 1.f / l : 0.f;
      const bool row_exists = kbo < p.bpt && kb < u.k1;
      const int h = within - j * p.grp;
      const long orow = (((long)u.b * p.N + kb) * p.S + j) * (long)p.Hq * kDH +
                        (long)(u.g * p.grp + h) * kDH + half * 64;
      for (int part = 0; part < 2; ++part) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tmem_o + lane_off + half * 64 + part * 32, ov);
        if (!row_exists) continue;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          p.out.store4(orow + part * 32 + 4 * e,
                       make_float4(__uint_as_float(ov[4 * e]) * inv, __uint_as_float(ov[4 * e + 1]) * inv,
                                   __uint_as_float(ov[4 * e + 2]) * inv, __uint_as_float(ov[4 * e + 3]) * inv));
      }
    } else if (fin) {
      tc_fence_after();
      const size_t rowi = (size_t)blockIdx.x * kM + r;
      float4* po = reinterpret_cast<float4*>(p.part_o + rowi * kDH + half * 64);
      for (int part = 0; part < 2; ++part) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tmem_o + lane_off + half * 64 + part * 32, ov);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          po[part * 8 + e] = make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                         __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]));
      }
      red_sum[half * 128 + r] = l_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sum_bar[quarter]);
      if (wait_all(&sum_bar[quarter], 0) && half == 0) {
        p.part_m[rowi] = m_run;
        p.part_l[rowi] = l_run + red_sum[128 + r];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && *abort_flag) report(p.status, kStatusTimeout, kKernAttnTc);
}

// One warp per query row of a tile: merge the chunk partials in chunk order, normalise,
// write the attention output row [t][(g*grp + h)*dh ...].
__global__ void attn_combine_kernel(const AttnTcParams p, ActOut out, int Hq) {
  pdl_wait();
  pdl_trigger();
  const int warps = blockDim.x >> 5;
  const long gw = (long)blockIdx.x * warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long total = (long)p.B * p.Hkv * p.tiles * kM;
  if (gw >= total) return;
  const int r = (int)(gw % kM);
  long rest = gw / kM;
  const int t = (int)(rest % p.tiles);
  rest /= p.tiles;
  const int g = (int)(rest % p.Hkv);
  const int b = (int)(rest / p.Hkv);
  const int k0 = t * p.bpt, k1 = min(p.N, k0 + p.bpt);
  const int kbo = r / p.R;
  if (kbo >= p.bpt) return;
  const int kb = k0 + kbo;
  if (kb >= k1) return;
  const int within = r - kbo * p.R;
  const int j = within / p.grp, h = within - j * p.grp;
  const long trow = ((long)b * p.N + kb) * p.S + j;
  const long col0 = (long)(g * p.grp + h) * kDH;
  const long orow = trow * (long)Hq * kDH + col0;
  const int a = p.anchors[b * p.N + kb];
  const bool row_valid = a >= 0 && p.valid[((long)b * p.N + kb) * p.S + j] != 0;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float lsum = 0.f;
  if (row_valid) {
    int amax = 0;
    for (int k = k0; k < k1; ++k) amax = max(amax, p.anchors[b * p.N + k]);
    amax = min(amax, p.L);
    const int nch = amax > p.chunk ? (amax + p.chunk - 1) / p.chunk : 1;
    const long unit0 = (((long)b * p.Hkv + g) * p.tiles + t) * p.max_chunks;
    float M = -INFINITY;
    for (int c = 0; c < nch; ++c) {
      const long ri = (unit0 + c) * kM + r;
      if (p.part_l[ri] > 0.f) M = fmaxf(M, p.part_m[ri]);
    }
    for (int c = 0; c < nch; ++c) {
      const long ri = (unit0 + c) * kM + r;
      const float l = p.part_l[ri];
      if (!(l > 0.f)) continue;
      const float f = exp2f(p.part_m[ri] - M);
      lsum += l * f;
      const float4 o = reinterpret_cast<const float4*>(p.part_o + ri * kDH)[lane];
      acc[0] += o.x * f;
      acc[1] += o.y * f;
      acc[2] += o.z * f;
      acc[3] += o.w * f;
    }
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  for (int e = 0; e < 4; ++e) out.store(orow + lane * 4 + e, acc[e] * inv);
}

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

// fp16 map with a 128-byte swizzle; dims/box innermost first; strides in bytes for dims 1..
bool encode_f16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, rank, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

AttnTcLayout attention_tc_layout(int B, int N, int S, int L, int Hq, int Hkv, int num_sms) {
  AttnTcLayout lay;
  lay.grp = Hq / Hkv;
  lay.R = S * lay.grp;
  lay.bpt = kM / lay.R;
  lay.tiles = (N + lay.bpt - 1) / lay.bpt;
  // key chunk: enough units for about four waves over the SMs when every tile reads the
  // whole context, between 256 and 4096 keys (a power of two)
  const double per_unit = (double)L * B * Hkv * lay.tiles / (4.0 * (num_sms > 0 ? num_sms : 1));
  lay.chunk = 256;
  while (lay.chunk < 4096 && lay.chunk < per_unit) lay.chunk *= 2;
  // one chunk when the (row, KV head, tile) units alone nearly fill the SMs (three
  // quarters or more) and no unit is long: each unit then normalises its own output (no
  // partials, no combine pass), and its fixed cost -- tensor memory, Q, the first K/V tiles
  // in flight, about two key tiles' worth -- is paid once per tile instead of once per chunk
  const long base_units = (long)B * Hkv * lay.tiles;
  if (L <= 4096 && 4 * base_units >= 3L * (num_sms > 0 ? num_sms : 1))
    lay.chunk = (L + kKT - 1) / kKT * kKT;
  lay.max_chunks = (L + lay.chunk - 1) / lay.chunk;
  if (lay.max_chunks < 1) lay.max_chunks = 1;
  lay.units = (long)B * Hkv * lay.tiles * lay.max_chunks;
  lay.part_floats = lay.units * kM * (kDH + 2);
  return lay;
}

bool attention_tc_supported(int S, int Hq, int Hkv, int dh) {
  if (dh != kDH || Hq % Hkv != 0) return false;
  const int grp = Hq / Hkv;
  const int R = S * grp;
  // a query tile covers 128 / grp block slots: the block V^T tiles then start at a key index
  // that is a multiple of 8 (16 bytes of fp16), as a tiled TMA load requires
  return R >= 1 && R <= kM && (kM % R) == 0 && (kM / grp) % 8 == 0;
}

cudaError_t launch_attention_tc(const AttnTcArgs& a, cudaStream_t stream) {
  const AttnTcLayout lay = attention_tc_layout(a.B, a.N, a.S, a.L, a.Hq, a.Hkv, a.num_sms);
  AttnTcParams p;
  p.B = a.B;
  p.N = a.N;
  p.S = a.S;
  p.L = a.L;
  p.Hkv = a.Hkv;
  p.grp = lay.grp;
  p.R = lay.R;
  p.bpt = lay.bpt;
  p.tiles = lay.tiles;
  p.chunk = lay.chunk;
  p.max_chunks = lay.max_chunks;
  p.q = a.q;
  p.q_rows = (long)a.B * a.Hkv * a.N * lay.R;
  p.anchors = a.anchors;
  p.valid = a.valid;
  p.mask = a.mask;
  p.part_o = a.partials;
  p.part_m = a.partials + lay.units * kM * kDH;
  p.part_l = p.part_m + lay.units * kM;
  p.status = a.status;
  p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)kDH));
  p.direct = lay.max_chunks == 1 ? 1 : 0;
  p.Hq = a.Hq;
  p.out = a.out;

  CUtensorMap mkc, mvc, mkb, mvb, mq;
  const long planes = (long)a.B * 2 * a.Hkv;
  {
    cuuint64_t dims[3] = {(cuuint64_t)kDH, (cuuint64_t)a.L, (cuuint64_t)planes};
    cuuint64_t str[2] = {(cuuint64_t)kDH * 2, (cuuint64_t)a.L * kDH * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kKT, 1};  // [kKT keys][64 dh]
    if (!encode_f16(&mkc, a.kv_layer, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)a.L, (cuuint64_t)kDH, (cuuint64_t)planes};
    cuuint64_t str[2] = {(cuuint64_t)a.L * 2, (cuuint64_t)a.L * kDH * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kDH, 1};  // [128 dh][64 keys]
    if (!encode_f16(&mvc, a.kv_layer, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const long kb_rows = (long)a.B * a.Hkv * a.N * a.S;
    cuuint64_t dims[2] = {(cuuint64_t)kDH, (cuuint64_t)kb_rows};
    cuuint64_t str[1] = {(cuuint64_t)kDH * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kKT};
    if (!encode_f16(&mkb, a.kb, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.N * a.S, (cuuint64_t)a.B * a.Hkv * kDH};
    cuuint64_t str[1] = {(cuuint64_t)a.ns_pad * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kDH};  // [128 dh][64 keys]
    if (!encode_f16(&mvb, a.vbt, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    // Q rows [B][Hkv][N][R] x dh; rows past the end read the zero fill
    cuuint64_t dims[2] = {(cuuint64_t)kDH, (cuuint64_t)p.q_rows};
    cuuint64_t str[1] = {(cuuint64_t)kDH * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kM};
    if (!encode_f16(&mq, a.q, 2, dims, str, box)) return cudaErrorInvalidValue;
  }
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  {
    const cudaError_t le = launch_pdl(attn_tc_kernel, dim3((unsigned)lay.units), dim3(kThreads),
        kSmemBytes, stream, mkc, mvc, mkb, mvb, mq, p);
    if (le != cudaSuccess) return le;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.direct) return e;
  const long rows = (long)a.B * a.Hkv * lay.tiles * kM;
  const int threads = 256;
  const long blocks = (rows * 32 + threads - 1) / threads;
  {
    const cudaError_t le = launch_pdl(attn_combine_kernel, dim3((unsigned)blocks), dim3(threads), 0,
        stream, p, a.out, a.Hq);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace dflash

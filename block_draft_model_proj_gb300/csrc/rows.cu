// Row-wise kernels of the draft body: RMSNorm steps of the fp32 residual stream, the RoPE
// table, and the element-wise epilogues that follow the projection GEMMs.
//
// Layer structure ("DFlash" page, How it works; the draft decoder layers of the "DFlash
// Draft Body" page, How It Works step 3): pre-norm RMSNorm -> attention -> residual,
// RMSNorm -> SwiGLU MLP -> residual; rotary position embedding with base rope_theta
// ("DFlash", Configuration).  RoPE here is the rotate-half form: channel i pairs with
// channel i + dh/2.
//
// Computed activations that feed a projection GEMM are written through ActOut: fp32 for
// the fp32 configuration, else fp16 for the tensor-core GEMM.  Attention operands (q, block
// k / v) are kept in fp32.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dflash {

namespace {

constexpr double kTwoPi = 6.283185307179586476925286766559;

__device__ __forceinline__ float ld(const void* p, int dt, long i) {
  return dt == DFLASH_DTYPE_BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
                                 : static_cast<const float*>(p)[i];
}

// Ordered compaction of the active tiles by one CTA (up to 1024 threads).
template <typename Pred>
__device__ __forceinline__ void compact_tiles(long tiles, int32_t* list, Pred active) {
  __shared__ int warp_counts[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int base = 0;
  for (long t0 = 0; t0 < tiles; t0 += blockDim.x) {
    const long t = t0 + threadIdx.x;
    const bool on = t < tiles && active(t);
    const unsigned bal = __ballot_sync(0xffffffffu, on);
    __syncthreads();
    if (lane == 0) warp_counts[warp] = __popc(bal);
    __syncthreads();
    int before = 0, sum = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      if (w < warp) before += warp_counts[w];
      sum += warp_counts[w];
    }
    if (on) list[1 + base + before + __popc(bal & ((1u << lane) - 1u))] = (int32_t)t;
    base += sum;
  }
  if (threadIdx.x == 0) list[0] = base;
}


// A 128-row tile of the context rows m = b*L + c holding a row with c < ctx_len[b].
__device__ __forceinline__ bool ctx_tile_active(long t, const int32_t* ctx_len, int B, int L) {
  const long m0 = t * kGemmTileM, m1 = min(m0 + kGemmTileM, (long)B * L);
  for (long m = m0; m < m1;) {
    const int b = (int)(m / L);
    int cl = ctx_len[b];
    cl = cl < 0 ? 0 : (cl > L ? L : cl);
    if ((int)(m - (long)b * L) < cl) return true;
    m = (long)(b + 1) * L;
  }
  return false;
}

// A 128-row tile of the T slots holding a valid slot.
__device__ __forceinline__ bool slot_tile_active(long t, const uint8_t* valid, long T) {
  for (long r = t * kGemmTileM; r < min((t + 1) * kGemmTileM, T); ++r)
    if (valid[r]) return true;
  return false;
}

// Inverse frequencies theta^(-2i/dh) as float pairs (hi + lo carries about 48 bits) and 2*pi
// as a float pair, for the angle reduction below.
struct RopeConsts {
  float inv_hi[128], inv_lo[128];
  float two_pi_hi, two_pi_lo, inv_two_pi;
};

// cos / sin of the angle (p0 + p) * inv_i for p < P, i < half.  The angle is reduced to
// [-pi, pi] in fp32 by Cody and Waite's method (the multiple of 2*pi taken off in two float
// pieces), the product carried as a float pair (the rounding error of the leading product
// from an FMA): the reduced angle is within about 4e-7 of the exact one for positions below
// 2^24 (2.4e-7 measured against fp64 over positions up to 2^20, theta 1e6, dh 128), then
// sincosf evaluates it.
// With a tile job, block 0 builds the active-tile list instead (one launch fewer).
__global__ void rope_table_kernel(float* __restrict__ cos_t, float* __restrict__ sin_t, int p0,
                                  int P, int half, const RopeConsts rc, const TileJob job) {
  pdl_wait();
  pdl_trigger();
  long blk = blockIdx.x, nblk = gridDim.x;
  if (job.kind != TileJob::kNone) {
    if (blockIdx.x == 0) {
      if (job.kind == TileJob::kContext)
        compact_tiles(job.tiles, job.list,
                      [&](long t) { return ctx_tile_active(t, job.ctx_len, job.B, job.L); });
      else
        compact_tiles(job.tiles, job.list,
                      [&](long t) { return slot_tile_active(t, job.valid, job.T); });
      return;
    }
    blk -= 1;
    nblk -= 1;
  }
  const long n = (long)P * half;
  for (long e = blk * blockDim.x + threadIdx.x; e < n; e += nblk * blockDim.x) {
    const int p = (int)(e / half), i = (int)(e - (long)p * half);
    const float pf = (float)(p0 + p);  // exact below 2^24
    const float a_hi = pf * rc.inv_hi[i];
    const float a_lo = fmaf(pf, rc.inv_lo[i], fmaf(pf, rc.inv_hi[i], -a_hi));
    const float k = rintf(a_hi * rc.inv_two_pi);
    float r = fmaf(-k, rc.two_pi_hi, a_hi);
    r = fmaf(-k, rc.two_pi_lo, r);
    r += a_lo;
    float s, c;
    sincosf(r, &s, &c);
    cos_t[e] = c;
    sin_t[e] = s;
  }
}

__global__ void residual_norm_kernel(int mode, int dt, float* __restrict__ x,
                                     const void* __restrict__ emb, const float* __restrict__ y,
                                     int nsplit, const int* __restrict__ nsplit_dev,
                                     long split_stride, const void* __restrict__ g,
                                     float eps, ActOut h, float* __restrict__ out,
                                     const uint8_t* __restrict__ valid, bool final_norm, int D) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[33];
  const long r = blockIdx.x;
  if (nsplit_dev) nsplit = *nsplit_dev;
  if (valid && valid[r] == 0) {  // an invalid slot: zero output / zero GEMM input, y unread
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
      if (mode == kNormFinal) out[r * D + c] = 0.f;
      else h.store(r * D + c, 0.f);
    }
    return;
  }
  float* xr = x + r * D;
  float ss = 0.f;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float v;
    if (mode == kNormInit) {
      v = ld(emb, dt, r * D + c);
    } else {
      v = xr[c];
      for (int s = 0; s < nsplit; ++s) v += y[s * split_stride + r * D + c];
    }
    if (mode == kNormInit || nsplit > 0) xr[c] = v;
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float rstd = rsqrtf(ss / (float)D + eps);
  if (mode == kNormFinal) {
    const bool ok = valid[r] != 0;
    for (int c = threadIdx.x; c < D; c += blockDim.x) {
      float v = 0.f;
      if (ok) v = final_norm ? xr[c] * rstd * ld(g, dt, c) : xr[c];
      out[r * D + c] = v;
    }
  } else {
    for (int c = threadIdx.x; c < D; c += blockDim.x) h.store(r * D + c, xr[c] * rstd * ld(g, dt, c));
  }
}

__global__ void rows_norm_kernel(int dt, const float* __restrict__ y, int nsplit, long split_stride,
                                 const void* __restrict__ g, float eps, bool with_norm, ActOut out,
                                 int D) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[33];
  const long r = blockIdx.x;
  float ss = 0.f;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float v = 0.f;
    for (int s = 0; s < nsplit; ++s) v += y[s * split_stride + r * D + c];
    ss += v * v;
  }
  ss = with_norm ? block_sum(ss, red) : 0.f;
  const float rstd = with_norm ? rsqrtf(ss / (float)D + eps) : 1.f;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float v = 0.f;
    for (int s = 0; s < nsplit; ++s) v += y[s * split_stride + r * D + c];
    out.store(r * D + c, with_norm ? v * rstd * ld(g, dt, c) : v);
  }
}

__device__ __forceinline__ float sum_splits(const float* y, int nsplit, long stride, long idx) {
  float v = 0.f;
  for (int s = 0; s < nsplit; ++s) v += y[s * stride + idx];
  return v;
}

__device__ __forceinline__ float4 sum_splits4(const float* y, int nsplit, long stride, long idx) {
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < nsplit; ++s) {
    const float4 t = *reinterpret_cast<const float4*>(y + s * stride + idx);
    v.x += t.x;
    v.y += t.y;
    v.z += t.z;
    v.w += t.w;
  }
  return v;
}

// Vectorised residual step: one CTA per row, each thread owns kV float4 groups of the row
// (D % 4 == 0, D <= 4 * kV * blockDim.x), a single pass over global memory.
template <int kV>
__global__ void residual_norm_vec_kernel(int mode, int dt, float* __restrict__ x,
                                         const void* __restrict__ emb, const float* __restrict__ y,
                                         int nsplit, const int* __restrict__ nsplit_dev,
                                         long split_stride, const void* __restrict__ g,
                                         float eps, ActOut h, float* __restrict__ out,
                                         const uint8_t* __restrict__ valid, bool final_norm, int D) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[33];
  const long r = blockIdx.x;
  const int D4 = D / 4;
  if (nsplit_dev) nsplit = *nsplit_dev;
  if (valid && valid[r] == 0) {  // an invalid slot: zero output / zero GEMM input, y unread
    for (int q = threadIdx.x; q < D4; q += blockDim.x) {
      if (mode == kNormFinal)
        *reinterpret_cast<float4*>(out + r * D + 4L * q) = make_float4(0.f, 0.f, 0.f, 0.f);
      else
        h.store4(r * D + 4L * q, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    return;
  }
  float4 v[kV];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kV; ++k) {
    const int q = threadIdx.x + k * blockDim.x;
    if (q >= D4) { v[k] = make_float4(0.f, 0.f, 0.f, 0.f); continue; }
    const long idx = r * D + 4L * q;
    float4 t;
    if (mode == kNormInit) {
      t = load4(emb, dt, idx);
    } else {
      t = *reinterpret_cast<const float4*>(x + idx);
      const float4 a = sum_splits4(y, nsplit, split_stride, idx);
      t.x += a.x;
      t.y += a.y;
      t.z += a.z;
      t.w += a.w;
    }
    // nsplit 0: x already holds the sum (added by the GEMM epilogue), nothing to write back
    if (mode == kNormInit || nsplit > 0) *reinterpret_cast<float4*>(x + idx) = t;
    v[k] = t;
    ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
  }
  ss = block_sum(ss, red);
  const float rstd = rsqrtf(ss / (float)D + eps);
  const bool ok = mode != kNormFinal || valid[r] != 0;
#pragma unroll
  for (int k = 0; k < kV; ++k) {
    const int q = threadIdx.x + k * blockDim.x;
    if (q >= D4) continue;
    const long idx = r * D + 4L * q;
    const float4 gg = load4(g, dt, 4L * q);
    if (mode == kNormFinal) {
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok)
        o = final_norm ? make_float4(v[k].x * rstd * gg.x, v[k].y * rstd * gg.y,
                                     v[k].z * rstd * gg.z, v[k].w * rstd * gg.w)
                       : v[k];
      *reinterpret_cast<float4*>(out + idx) = o;
    } else {
      h.store4(idx, make_float4(v[k].x * rstd * gg.x, v[k].y * rstd * gg.y, v[k].z * rstd * gg.z,
                                v[k].w * rstd * gg.w));
    }
  }
}

template <int kV>
__global__ void rows_norm_vec_kernel(int dt, const float* __restrict__ y, int nsplit,
                                     long split_stride, const void* __restrict__ g, float eps,
                                     bool with_norm, ActOut out, int D,
                                     const int32_t* __restrict__ ctx_len, int L) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[33];
  const long r = blockIdx.x;
  // context rows no block reads (c >= ctx_len[b]) are left unwritten
  if (ctx_len && (int)(r % L) >= ctx_len[r / L]) return;
  const int D4 = D / 4;
  float4 v[kV];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kV; ++k) {
    const int q = threadIdx.x + k * blockDim.x;
    v[k] = q < D4 ? sum_splits4(y, nsplit, split_stride, r * D + 4L * q)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
  }
  ss = with_norm ? block_sum(ss, red) : 0.f;
  const float rstd = with_norm ? rsqrtf(ss / (float)D + eps) : 1.f;
#pragma unroll
  for (int k = 0; k < kV; ++k) {
    const int q = threadIdx.x + k * blockDim.x;
    if (q >= D4) continue;
    float4 o = v[k];
    if (with_norm) {
      const float4 gg = load4(g, dt, 4L * q);
      o = make_float4(o.x * rstd * gg.x, o.y * rstd * gg.y, o.z * rstd * gg.z, o.w * rstd * gg.w);
    }
    out.store4(r * D + 4L * q, o);
  }
}

__device__ __forceinline__ float silu_mul(float gt, float up) { return gt / (1.f + expf(-gt)) * up; }

// SwiGLU, four consecutive channels per thread (I % 4 == 0)
// valid (optional): rows of invalid slots (whose GEMM rows may be unwritten) get zeros
__global__ void swiglu_vec_kernel(const float* __restrict__ y, int nsplit,
                                  const int* __restrict__ nsplit_dev, long split_stride,
                                  ActOut act, long T, int I, const uint8_t* __restrict__ valid) {
  pdl_wait();
  pdl_trigger();
  if (nsplit_dev) nsplit = *nsplit_dev;
  const int I4 = I / 4;
  const long n = T * I4;
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const long t = e / I4;
    const int i = (int)(e - t * I4) * 4;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!valid || valid[t]) {
      const float4 gt = sum_splits4(y, nsplit, split_stride, t * 2 * I + i);
      const float4 up = sum_splits4(y, nsplit, split_stride, t * 2 * I + I + i);
      o = make_float4(silu_mul(gt.x, up.x), silu_mul(gt.y, up.y), silu_mul(gt.z, up.z),
                      silu_mul(gt.w, up.w));
    }
    act.store4(t * I + i, o);
  }
}


// Attention operands in their attention-ready layouts (OutT: fp32 for the CUDA-core
// attention, fp16 for the tensor-core attention):
//   q   [B][Hkv][N][S][grp][dh]   (the query rows of one KV head are contiguous per block)
//   kb  [B][Hkv][N*S][dh]         (block keys)
//   vbt [B][Hkv][dh][ns_pad]      (block values, transposed)
// Invalid slots get zero operands: they are never keys, and their GEMM rows may have been
// skipped (unwritten) when a whole 128-row tile held no valid slot.

__device__ __forceinline__ void store4(float* dst, float4 v) { *reinterpret_cast<float4*>(dst) = v; }
__device__ __forceinline__ void store4(__half* dst, float4 v) {
  const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(dst) = w;
}

// two consecutive elements (dst 2-element aligned)
__device__ __forceinline__ void store_pair(float* dst, float a, float b) {
  *reinterpret_cast<float2*>(dst) = make_float2(a, b);
}
__device__ __forceinline__ void store_pair(__half* dst, float a, float b) {
  *reinterpret_cast<__half2*>(dst) = __floats2half2_rn(a, b);
}

// Q and K heads with RoPE: one thread per (row t, head, 4 consecutive pairs i .. i+3), the
// pairs (i, i + dh/2) rotated by the angle of position pos[t].  dh % 8 == 0.  Run by blocks
// blk = 0 .. nblk-1 of the launch (grid-stride over the elements).
template <typename OutT>
__device__ __forceinline__ void qk_rope_blocks(
    int blk, int nblk, const float* __restrict__ y, int nsplit, long split_stride,
    const int32_t* __restrict__ pos, const uint8_t* __restrict__ valid,
    const float* __restrict__ cos_t, const float* __restrict__ sin_t, int P,
    OutT* __restrict__ q, OutT* __restrict__ kb, long T, int N, int S, int Hq, int Hkv, int dh,
    unsigned* status) {
  const int half = dh / 2, q4 = half / 4;
  const int heads = Hq + Hkv;  // Q then K heads (the V heads are transposed by other blocks)
  const int grp = Hq / Hkv;
  const long width = (long)(Hq + 2 * Hkv) * dh;
  const long n = T * heads * q4;
  for (long e = blk * (long)blockDim.x + threadIdx.x; e < n; e += (long)nblk * blockDim.x) {
    const long t = e / ((long)heads * q4);
    const int rem = (int)(e - t * heads * q4);
    const int hd = rem / q4, i = (rem - hd * q4) * 4;
    const long base = t * width + (long)hd * dh;
    const bool vt = valid[t] != 0;
    // loaded whatever the slot's validity (the rows exist; an invalid slot's may be
    // unwritten) and discarded by the select: the loads do not wait for the flag
    float4 a = sum_splits4(y, nsplit, split_stride, base + i);
    float4 bb = sum_splits4(y, nsplit, split_stride, base + i + half);
    if (!vt) a = bb = make_float4(0.f, 0.f, 0.f, 0.f);
    const int b = (int)(t / ((long)N * S));
    const int ks = (int)(t - (long)b * N * S);  // k * S + j
    const int k = ks / S, j = ks - k * S;
    int pp = pos[t];
    if (pp < 0 || pp >= P) {
      if (vt && i == 0) report(status, kStatusCheck, kKernEpilogue);
      pp = 0;
    }
    const float4 c = *reinterpret_cast<const float4*>(cos_t + (long)pp * half + i);
    const float4 sn = *reinterpret_cast<const float4*>(sin_t + (long)pp * half + i);
    const float4 lo = make_float4(a.x * c.x - bb.x * sn.x, a.y * c.y - bb.y * sn.y,
                                  a.z * c.z - bb.z * sn.z, a.w * c.w - bb.w * sn.w);
    const float4 hi = make_float4(bb.x * c.x + a.x * sn.x, bb.y * c.y + a.y * sn.y,
                                  bb.z * c.z + a.z * sn.z, bb.w * c.w + a.w * sn.w);
    OutT* dst;
    if (hd < Hq) {
      const int g = hd / grp, h = hd - g * grp;
      dst = q + (((((long)b * Hkv + g) * N + k) * S + j) * grp + h) * dh;
    } else {
      const int g = hd - Hq;
      dst = kb + ((((long)b * Hkv + g) * N + k) * S + j) * dh;
    }
    store4(dst + i, lo);
    store4(dst + i + half, hi);
  }
}

// V heads, transposed through shared memory: one block per (row b, KV head g, 32 slots).
// Each thread loads float4 pieces of the slots' V rows (a warp reads one 128-float row,
// coalesced along the channels), all of them before the first is used, then the block
// writes dh rows of 32 slots of vbt, two slots per store (coalesced along the slots).
// dh % 4 == 0, dh <= 256.
constexpr int kVtSlots = 32;
template <typename OutT>
__device__ __forceinline__ void v_transpose_block(
    int bi, float (*tile)[257], const float* __restrict__ y, int nsplit, long split_stride,
    const uint8_t* __restrict__ valid, OutT* __restrict__ vbt, int ns_pad, int N, int S, int Hq,
    int Hkv, int dh) {
  const int NS = N * S;
  const int tiles = (NS + kVtSlots - 1) / kVtSlots;
  const int bt = bi % tiles;
  const int bg = bi / tiles;  // b * Hkv + g
  const int b = bg / Hkv, g = bg - b * Hkv;
  const int ks0 = bt * kVtSlots;
  const long width = (long)(Hq + 2 * Hkv) * dh;
  const int vcol = (Hq + Hkv + g) * dh;
  const int d4n = dh / 4;                 // float4 pieces per row
  const int pieces = kVtSlots * d4n;      // <= 2048
  // up to 8 pieces per thread; rows of invalid slots (whose GEMM rows may be unwritten) are
  // read and then discarded by the select, so the loads do not wait for the flags
  float4 acc[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sp = 0; sp < nsplit; ++sp) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int pc = threadIdx.x + u * 256;
      if (pc < pieces) {
        const int jj = pc / d4n, d4 = pc - jj * d4n;
        const int ks = min(ks0 + jj, NS - 1);
        const float4 f = *reinterpret_cast<const float4*>(
            y + sp * split_stride + ((long)b * NS + ks) * width + vcol + 4 * d4);
        acc[u].x += f.x;
        acc[u].y += f.y;
        acc[u].z += f.z;
        acc[u].w += f.w;
      }
    }
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int pc = threadIdx.x + u * 256;
    if (pc < pieces) {
      const int jj = pc / d4n, d4 = pc - jj * d4n;
      const int ks = ks0 + jj;
      const bool ok = ks < NS && valid[(long)b * NS + ks] != 0;
      tile[jj][4 * d4] = ok ? acc[u].x : 0.f;
      tile[jj][4 * d4 + 1] = ok ? acc[u].y : 0.f;
      tile[jj][4 * d4 + 2] = ok ? acc[u].z : 0.f;
      tile[jj][4 * d4 + 3] = ok ? acc[u].w : 0.f;
    }
  }
  __syncthreads();
  // row d of vbt: slots ks0 .. ks0 + 31 as 16 pairs
  for (int idx = threadIdx.x; idx < dh * (kVtSlots / 2); idx += blockDim.x) {
    const int d = idx / (kVtSlots / 2), pr = idx - d * (kVtSlots / 2);
    const int ks = ks0 + 2 * pr;
    OutT* dst = vbt + ((long)bg * dh + d) * ns_pad + ks;
    const float v0 = tile[2 * pr][d], v1 = tile[2 * pr + 1][d];
    if (ks + 1 < ns_pad) {
      store_pair(dst, v0, v1);
    } else if (ks < ns_pad) {
      dst[0] = from_f<OutT>(v0);
    }
  }
}

// The attention operands from the QKV projection's fp32 slices, one launch: blocks
// 0 .. vblocks-1 transpose the V heads (one per row b, KV head g and 32 slots), the others
// apply RoPE to the Q and K heads.
template <typename OutT>
__global__ void __launch_bounds__(256) qkv_rope_kernel(
    const float* __restrict__ y, int nsplit, const int* __restrict__ nsplit_dev, long split_stride,
    const int32_t* __restrict__ pos, const uint8_t* __restrict__ valid,
    const float* __restrict__ cos_t, const float* __restrict__ sin_t, int P, OutT* __restrict__ q,
    OutT* __restrict__ kb, OutT* __restrict__ vbt, int ns_pad, long T, int N, int S, int Hq,
    int Hkv, int dh, int vblocks, unsigned* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tile[kVtSlots][257];
  if (nsplit_dev) nsplit = *nsplit_dev;
  if ((int)blockIdx.x < vblocks)
    v_transpose_block<OutT>((int)blockIdx.x, tile, y, nsplit, split_stride, valid, vbt, ns_pad, N,
                            S, Hq, Hkv, dh);
  else
    qk_rope_blocks<OutT>((int)blockIdx.x - vblocks, (int)gridDim.x - vblocks, y, nsplit,
                         split_stride, pos, valid, cos_t, sin_t, P, q, kb, T, N, S, Hq, Hkv, dh,
                         status);
}

// Context K: one thread per (b, c, head, pair i); plane (b, 0, g) holds K as [L_cache][dh].
__global__ void ctx_k_scatter_kernel(const float* __restrict__ y, int nsplit, long split_stride,
                                     const float* __restrict__ cos_t,
                                     const float* __restrict__ sin_t, float* __restrict__ kv,
                                     int B, int L, int pos_offset, int L_cache, int Hkv, int dh,
                                     const int32_t* __restrict__ ctx_len,
                                     const int32_t* __restrict__ row_pos0) {
  const int half = dh / 2;
  const long per_row = (long)Hkv * half;
  const long n = (long)B * L * per_row;
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const long bc = e / per_row;
    const int rem = (int)(e - bc * per_row);
    const int g = rem / half, i = rem - g * half;
    const int b = (int)(bc / L), c = (int)(bc - (long)b * L);
    if (ctx_len && c >= ctx_len[b]) continue;
    const long src = bc * 2L * Hkv * dh + (long)g * dh;
    const float a = sum_splits(y, nsplit, split_stride, src + i);
    const float bb = sum_splits(y, nsplit, split_stride, src + i + half);
    // table row c holds position pos_offset + c; with row_pos0 the table starts at 0
    const long pos = (row_pos0 ? (long)row_pos0[b] : (long)pos_offset) + c;
    const long trow = row_pos0 ? pos : c;
    const float cs = cos_t[trow * half + i], sn = sin_t[trow * half + i];
    float* dst = kv + ((((long)b * 2) * Hkv + g) * L_cache + pos) * dh;
    dst[i] = a * cs - bb * sn;
    dst[i + half] = bb * cs + a * sn;
  }
}

// Context V: one thread per (b, head, channel d, c), c fastest so the transposed writes
// are coalesced; plane (b, 1, g) holds V^T as [dh][L_cache].
__global__ void ctx_vt_scatter_kernel(const float* __restrict__ y, int nsplit, long split_stride,
                                      float* __restrict__ kv, int B, int L, int pos_offset,
                                      int L_cache, int Hkv, int dh,
                                      const int32_t* __restrict__ ctx_len,
                                      const int32_t* __restrict__ row_pos0) {
  const long n = (long)B * Hkv * dh * L;
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const int c = (int)(e % L);
    long rest = e / L;
    const int d = (int)(rest % dh);
    rest /= dh;
    const int g = (int)(rest % Hkv);
    const int b = (int)(rest / Hkv);
    if (ctx_len && c >= ctx_len[b]) continue;
    const long src = ((long)b * L + c) * 2L * Hkv * dh + (long)(Hkv + g) * dh + d;
    const float v = sum_splits(y, nsplit, split_stride, src);
    const long pos = (row_pos0 ? (long)row_pos0[b] : (long)pos_offset) + c;
    kv[((((long)b * 2 + 1) * Hkv + g) * dh + d) * L_cache + pos] = v;
  }
}

__global__ void swiglu_kernel(const float* __restrict__ y, int nsplit,
                              const int* __restrict__ nsplit_dev, long split_stride, ActOut act,
                              long T, int I, const uint8_t* __restrict__ valid) {
  pdl_wait();
  pdl_trigger();
  if (nsplit_dev) nsplit = *nsplit_dev;
  const long n = T * I;
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const long t = e / I;
    const int i = (int)(e - t * I);
    if (valid && !valid[t]) {
      act.store(e, 0.f);
      continue;
    }
    const float gt = sum_splits(y, nsplit, split_stride, t * 2 * I + i);
    const float up = sum_splits(y, nsplit, split_stride, t * 2 * I + I + i);
    act.store(e, gt / (1.f + expf(-gt)) * up);
  }
}

inline int grid_for(long n, int threads) {
  long g = (n + threads - 1) / threads;
  if (g > 152L * 32) g = 152L * 32;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

cudaError_t launch_rope_table(float* cos_t, float* sin_t, int p0, int P, int head_dim,
                              double theta, cudaStream_t stream, const TileJob& job) {
  const int half = head_dim / 2;
  if (half > 128) return cudaErrorInvalidValue;
  if (p0 < 0 || (long)p0 + P > (1L << 24)) return cudaErrorInvalidValue;
  RopeConsts rc;
  for (int i = 0; i < half; ++i) {
    const double v = pow(theta, -2.0 * (double)i / (double)head_dim);
    rc.inv_hi[i] = (float)v;
    rc.inv_lo[i] = (float)(v - (double)rc.inv_hi[i]);
  }
  rc.two_pi_hi = (float)kTwoPi;
  rc.two_pi_lo = (float)(kTwoPi - (double)rc.two_pi_hi);
  rc.inv_two_pi = (float)(1.0 / kTwoPi);
  const long n = (long)P * half;
  {
    TileJob j = job;
    if (j.kind == TileJob::kContext) j.tiles = ((long)j.B * j.L + kGemmTileM - 1) / kGemmTileM;
    if (j.kind == TileJob::kSlots) j.tiles = (j.T + kGemmTileM - 1) / kGemmTileM;
    const int grid = grid_for(n, 256) + (j.kind != TileJob::kNone ? 1 : 0);
    const cudaError_t le = launch_pdl(rope_table_kernel, dim3(grid), dim3(256), 0, stream, cos_t,
                                      sin_t, p0, P, half, rc, j);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_residual_norm(int mode, int dtype, float* x, const void* emb, const float* y,
                                 int nsplit, const int* nsplit_dev, const void* g, double eps,
                                 ActOut h, float* out, const uint8_t* valid, bool final_norm,
                                 long rows, int D, cudaStream_t stream) {
  if (D % 4 == 0 && D <= 4 * 4 * 1024) {
    // a quarter of the row's float4 groups per thread: 4 independent 16-byte loads in
    // flight per thread and several rows per SM
    const int D4 = D / 4;
    const int threads = std::min(1024, std::max(32, ((D4 + 3) / 4 + 31) / 32 * 32));
    const int per = (D4 + threads - 1) / threads;
    if (per <= 1)
      {
    const cudaError_t le = launch_pdl(residual_norm_vec_kernel<1>, dim3(rows), dim3(threads), 0,
        stream, mode, dtype, x, emb, y, nsplit, nsplit_dev, rows * D, g, (float)eps, h, out, valid,
        final_norm, D);
    if (le != cudaSuccess) return le;
  }
    else
      {
    const cudaError_t le = launch_pdl(residual_norm_vec_kernel<4>, dim3(rows), dim3(threads), 0,
        stream, mode, dtype, x, emb, y, nsplit, nsplit_dev, rows * D, g, (float)eps, h, out, valid,
        final_norm, D);
    if (le != cudaSuccess) return le;
  }
    return cudaGetLastError();
  }
  const int threads = D >= 2048 ? 512 : 256;
  {
    const cudaError_t le = launch_pdl(residual_norm_kernel, dim3(rows), dim3(threads), 0, stream,
        mode, dtype, x, emb, y, nsplit, nsplit_dev, rows * D, g, (float)eps, h, out, valid,
        final_norm, D);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_rows_norm(int dtype, const float* y, int nsplit, const void* g, double eps,
                             bool with_norm, ActOut out, long rows, int D,
                             const int32_t* ctx_len, int L, cudaStream_t stream) {
  if (D % 4 == 0 && D <= 4 * 4 * 1024) {
    // a quarter of the row's float4 groups per thread: 4 independent 16-byte loads in
    // flight per thread and several rows per SM
    const int D4 = D / 4;
    const int threads = std::min(1024, std::max(32, ((D4 + 3) / 4 + 31) / 32 * 32));
    const int per = (D4 + threads - 1) / threads;
    if (per <= 1)
      {
    const cudaError_t le = launch_pdl(rows_norm_vec_kernel<1>, dim3(rows), dim3(threads), 0, stream,
        dtype, y, nsplit, rows * D, g, (float)eps, with_norm, out, D, ctx_len, L);
    if (le != cudaSuccess) return le;
  }
    else
      {
    const cudaError_t le = launch_pdl(rows_norm_vec_kernel<4>, dim3(rows), dim3(threads), 0, stream,
        dtype, y, nsplit, rows * D, g, (float)eps, with_norm, out, D, ctx_len, L);
    if (le != cudaSuccess) return le;
  }
    return cudaGetLastError();
  }
  const int threads = D >= 2048 ? 512 : 256;
  {
    const cudaError_t le = launch_pdl(rows_norm_kernel, dim3(rows), dim3(threads), 0, stream, dtype,
        y, nsplit, rows * D, g, (float)eps, with_norm, out, D);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

// One CTA of 128 threads per 128-slot tile: when no slot of the tile is valid, thread i
// zeroes q, kb and the vbt column of slot tile*128 + i.  The extra CTA(s) past the last
// tile zero the pad columns N*S .. ns_pad-1 of every vbt row.
__global__ void __launch_bounds__(128) qkv_clear_kernel(const uint8_t* __restrict__ valid,
                                                         __half* __restrict__ q,
                                                         __half* __restrict__ kb,
                                                         __half* __restrict__ vbt, int ns_pad,
                                                         long T, int NS, int Hq, int Hkv, int dh,
                                                         long tiles) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x < tiles) {
    const long t = (long)blockIdx.x * 128 + threadIdx.x;
    const int any = __syncthreads_or(t < T && valid[t] != 0);
    if (any || t >= T) return;
    const long b = t / NS, ks = t - b * NS;
    const int grp = Hq / Hkv;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int g = 0; g < Hkv; ++g) {
      uint4* qd = reinterpret_cast<uint4*>(q + ((b * Hkv + g) * NS + ks) * grp * dh);
      for (int i = 0; i < grp * dh / 8; ++i) qd[i] = z;
      uint4* kd = reinterpret_cast<uint4*>(kb + ((b * Hkv + g) * NS + ks) * dh);
      for (int i = 0; i < dh / 8; ++i) kd[i] = z;
      __half* vd = vbt + (b * Hkv + g) * (long)dh * ns_pad + ks;
      for (int d = 0; d < dh; ++d) vd[(long)d * ns_pad] = __float2half_rn(0.f);
    }
    return;
  }
  const int pad = ns_pad - NS;
  if (pad <= 0) return;
  const long rows = T / NS * Hkv * dh;  // vbt rows (b, g, d)
  for (long e = (long)(blockIdx.x - tiles) * 128 + threadIdx.x; e < rows * pad;
       e += (long)(gridDim.x - tiles) * 128) {
    const long r = e / pad;
    vbt[r * ns_pad + NS + (e - r * pad)] = __float2half_rn(0.f);
  }
}

cudaError_t launch_qkv_clear(const uint8_t* valid, __half* q, __half* kb, __half* vbt, int ns_pad,
                             long T, int N, int S, int Hq, int Hkv, int dh, cudaStream_t stream) {
  const int NS = N * S;
  if (T < 1 || NS < 1 || T % NS != 0 || dh % 8 != 0 || Hq % Hkv != 0 || ns_pad < NS)
    return cudaErrorInvalidValue;
  const long tiles = (T + 127) / 128;
  const long grid = tiles + 16;  // 16 CTAs for the pad columns
  cudaError_t e = launch_pdl(qkv_clear_kernel, dim3((unsigned)grid), dim3(128), 0, stream, valid,
                             q, kb, vbt, ns_pad, T, NS, Hq, Hkv, dh, tiles);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_qkv_rope(const float* y, int nsplit, const int* nsplit_dev, const int32_t* pos,
                            const uint8_t* valid, const float* cos_t, const float* sin_t, int P,
                            void* q, void* kb, void* vbt, int ns_pad, long T, int N, int S, int Hq,
                            int Hkv, int dh, bool f16, unsigned* status, cudaStream_t stream) {
  if (dh % 8 != 0 || dh > 256) return cudaErrorInvalidValue;
  const long n = T * (Hq + Hkv) * (dh / 8);
  const long stride = T * (long)(Hq + 2 * Hkv) * dh;
  const long B = T / ((long)N * S);
  const int vblocks = (int)(B * Hkv * ((N * S + kVtSlots - 1) / kVtSlots));
  const int grid = vblocks + grid_for(n, 256);
  cudaError_t e;
  if (f16)
    e = launch_pdl(qkv_rope_kernel<__half>, dim3(grid), dim3(256), 0, stream, y, nsplit,
                   nsplit_dev, stride, pos, valid, cos_t, sin_t, P, static_cast<__half*>(q),
                   static_cast<__half*>(kb), static_cast<__half*>(vbt), ns_pad, T, N, S, Hq, Hkv,
                   dh, vblocks, status);
  else
    e = launch_pdl(qkv_rope_kernel<float>, dim3(grid), dim3(256), 0, stream, y, nsplit,
                   nsplit_dev, stride, pos, valid, cos_t, sin_t, P, static_cast<float*>(q),
                   static_cast<float*>(kb), static_cast<float*>(vbt), ns_pad, T, N, S, Hq, Hkv,
                   dh, vblocks, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_ctx_kv_scatter(const float* y, int nsplit, const float* cos_t,
                                  const float* sin_t, float* kv_layer, int B, int L,
                                  int pos_offset, int L_cache, int Hkv, int dh,
                                  const int32_t* ctx_len, const int32_t* row_pos0,
                                  cudaStream_t stream) {
  const long stride = (long)B * L * 2 * Hkv * dh;
  const long nk = (long)B * L * Hkv * (dh / 2);
  ctx_k_scatter_kernel<<<grid_for(nk, 256), 256, 0, stream>>>(
      y, nsplit, stride, cos_t, sin_t, kv_layer, B, L, pos_offset, L_cache, Hkv, dh, ctx_len,
      row_pos0);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long nv = (long)B * Hkv * dh * L;
  ctx_vt_scatter_kernel<<<grid_for(nv, 256), 256, 0, stream>>>(
      y, nsplit, stride, kv_layer, B, L, pos_offset, L_cache, Hkv, dh, ctx_len, row_pos0);
  return cudaGetLastError();
}

namespace {

// bf16 -> fp16, eight elements (16 bytes) per thread and iteration.  A bf16 value is the
// upper half of an fp32 value; cvt.rn.f16x2.f32 rounds two of them to nearest even.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, bool& bad) {
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
  const float m = fmaxf(fabsf(lo), fabsf(hi)) + 0.f * (lo + hi);  // NaN if either is
  bad = bad || !(m < 65520.f);
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(256) convert_bf16_f16_kernel(
    const uint4* __restrict__ src, uint4* __restrict__ dst, long n8,
    const uint16_t* __restrict__ src_tail, uint16_t* __restrict__ dst_tail, int tail,
    unsigned* status) {
  pdl_wait();
  pdl_trigger();
  bool bad = false;
  const long stride = (long)gridDim.x * blockDim.x;
  long i = blockIdx.x * (long)blockDim.x + threadIdx.x;
  // four independent 16-byte loads in flight per thread
  for (; i + 3 * stride < n8; i += 4 * stride) {
    uint4 w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) w[u] = __ldcs(src + i + u * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint4 o;
      o.x = bf16x2_to_f16x2(w[u].x, bad);
      o.y = bf16x2_to_f16x2(w[u].y, bad);
      o.z = bf16x2_to_f16x2(w[u].z, bad);
      o.w = bf16x2_to_f16x2(w[u].w, bad);
      dst[i + u * stride] = o;
    }
  }
  for (; i < n8; i += stride) {
    const uint4 w = __ldcs(src + i);
    uint4 o;
    o.x = bf16x2_to_f16x2(w.x, bad);
    o.y = bf16x2_to_f16x2(w.y, bad);
    o.z = bf16x2_to_f16x2(w.z, bad);
    o.w = bf16x2_to_f16x2(w.w, bad);
    dst[i] = o;
  }
  if (blockIdx.x == 0 && threadIdx.x < tail) {
    const float v = __uint_as_float((uint32_t)src_tail[threadIdx.x] << 16);
    bad = bad || !(fabsf(v) < 65520.f);
    const __half h = __float2half_rn(v);
    dst_tail[threadIdx.x] = *reinterpret_cast<const uint16_t*>(&h);
  }
  if (bad) report(status, kStatusRange, kKernConvert);
}

__global__ void __launch_bounds__(1024) slot_tile_list_kernel(const uint8_t* __restrict__ valid,
                                                              long T, int32_t* list, long tiles) {
  pdl_wait();
  pdl_trigger();
  compact_tiles(tiles, list, [&](long t) { return slot_tile_active(t, valid, T); });
}

}  // namespace

cudaError_t launch_slot_tile_list(const uint8_t* valid, long T, int32_t* list,
                                  cudaStream_t stream) {
  const long tiles = (T + kGemmTileM - 1) / kGemmTileM;
  {
    const cudaError_t le = launch_pdl(slot_tile_list_kernel, dim3(1), dim3(1024), 0, stream, valid,
        T, list, tiles);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_convert_bf16_f16(const void* src, void* dst, size_t n, unsigned* status,
                                    cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  if (((uintptr_t)src | (uintptr_t)dst) % 16 != 0) return cudaErrorInvalidValue;
  const long n8 = (long)(n / 8);
  const int tail = (int)(n % 8);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // at most two CTAs per SM: enough bytes in flight for HBM, and room left beside them for
  // a GEMM running concurrently on another stream
  long blocks = (n8 + 1023) / 1024;
  const long cap = (long)(sms > 0 ? sms : 1) * 2;
  // the SM's shared-memory carveout set to the maximum, as the tensor-core kernels use it:
  // an SM holding these CTAs can then take a GEMM CTA at the same time
  static bool carveout = false;
  if (!carveout) {
    cudaError_t e = cudaFuncSetAttribute(convert_bf16_f16_kernel,
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    carveout = true;
  }
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  {
    const cudaError_t le = launch_pdl(convert_bf16_f16_kernel, dim3((unsigned)blocks), dim3(256), 0,
        stream, static_cast<const uint4*>(src), static_cast<uint4*>(dst), n8,
        static_cast<const uint16_t*>(src) + n8 * 8, static_cast<uint16_t*>(dst) + n8 * 8, tail,
        status);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

namespace {

// One thread per row: how many of the P verified positions commit, where they start, and
// the new cache length ("DFlash: drafting, verification, and speed", One DFlash generation
// cycle: only the anchor and the accepted proposals stay).
__global__ void append_plan_kernel(const int32_t* __restrict__ accepted,
                                   int32_t* __restrict__ cache_len, int B, int P, int L_cache,
                                   int32_t* __restrict__ n_out, int32_t* __restrict__ start_out,
                                   unsigned* status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int n = P;
  if (accepted) n = min(max(accepted[b] + 1, 0), P);
  const int start = cache_len[b];
  if (start < 0 || (long)start + n > (long)L_cache) {
    report(status, kStatusCheck, kKernEpilogue);
    n = 0;
  }
  n_out[b] = n;
  start_out[b] = start < 0 ? 0 : start;
  cache_len[b] = start + n;
}

}  // namespace

cudaError_t launch_append_plan(const int32_t* accepted, int32_t* cache_len, int B, int P,
                               int L_cache, int32_t* n, int32_t* start, unsigned* status,
                               cudaStream_t stream) {
  const cudaError_t le = launch_pdl(append_plan_kernel, dim3((B + 255) / 256), dim3(256), 0,
                                    stream, accepted, cache_len, B, P, L_cache, n, start, status);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

cudaError_t launch_swiglu(const float* y, int nsplit, const int* nsplit_dev, ActOut act, long T,
                          int I, const uint8_t* valid, cudaStream_t stream) {
  if (I % 4 == 0) {
    const long n4 = T * (I / 4);
    return launch_pdl(swiglu_vec_kernel, dim3(grid_for(n4, 256)), dim3(256), 0, stream, y, nsplit,
                      nsplit_dev, T * 2L * I, act, T, I, valid);
  }
  const long n = T * I;
  return launch_pdl(swiglu_kernel, dim3(grid_for(n, 256)), dim3(256), 0, stream, y, nsplit,
                    nsplit_dev, T * 2L * I, act, T, I, valid);
}

}  // namespace dflash

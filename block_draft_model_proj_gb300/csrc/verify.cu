// Greedy block verification: vocab-wide argmax per position, then the accepted prefix.
//
// "DFlash: drafting, verification, and speed", One DFlash generation cycle: the target
// chooses its highest-probability token at every position of the drafted block; the
// longest prefix of proposals that agrees with those choices is accepted; the target's
// choice at the first disagreement is emitted, or the last choice (the bonus) when every
// proposal agrees; a matched EOS proposal ends the block.
//
// Kernel 1 (HBM-bound, the whole cost): the [B*(gamma+1), V] logits are cut into
// `chunks` equal column ranges per row; one CTA reduces one range with 16-byte vector loads
// to (max value, lowest index of that value) and writes it to the workspace.  Values are
// compared exactly in fp32 (bf16 and fp32 inputs convert to fp32 without rounding), ties
// keep the lower index, so the result does not depend on the split.
// Kernel 2: one warp per request combines its rows' partials in chunk order and runs the
// accepted-prefix scan.
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace dflash {

namespace {

constexpr int kVerifyThreads = 256;
constexpr int kMaxVerifyDevices = 64;

struct ArgMax {
  float v;
  int i;
};

// (v, i) beats (w, j): larger value, or equal value and lower index.  NaN never wins.
__device__ __forceinline__ bool better(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);
}

__device__ __forceinline__ void consider(ArgMax& a, float v, int i) {
  if (better(v, i, a.v, a.i)) { a.v = v; a.i = i; }
}

// 16-byte streaming load, issued where it stands (volatile asm): a batch of these is in
// flight together before any of its values is used
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 u;
  asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
               : "l"(p));
  return u;
}

// The 8 bf16 values of u against the running best of this thread, whose elements come in
// increasing index order: only a strictly larger value replaces it (ties keep the earlier,
// lower index); before anything is found (index sentinel) an equal value -- -inf -- is taken
// too.  The vector's maximum comes from packed bf16 max instructions (which skip NaN); the
// index search runs only when that maximum beats the running best.
__device__ __forceinline__ void consider8(ArgMax& a, const uint4& u, int base) {
  const __nv_bfloat162 w0 = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 w1 = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  const __nv_bfloat162 w2 = *reinterpret_cast<const __nv_bfloat162*>(&u.z);
  const __nv_bfloat162 w3 = *reinterpret_cast<const __nv_bfloat162*>(&u.w);
  const __nv_bfloat162 m2 = __hmax2(__hmax2(w0, w1), __hmax2(w2, w3));
  const float mv = fmaxf(__low2float(m2), __high2float(m2));
  if (mv > a.v || (a.i == 0x7fffffff && mv == a.v)) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float f = __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
      if (f == mv) {
        a.v = mv;
        a.i = base + e;
        break;
      }
    }
  }
}


template <typename T>
__global__ void __launch_bounds__(kVerifyThreads)
argmax_partial_kernel(const T* __restrict__ logits, int V, int chunks, int chunk_len,
                      bool vec_ok, float* __restrict__ part_v, int* __restrict__ part_i) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y, chunk = blockIdx.x;
  const int c0 = chunk * chunk_len;
  const int c1 = min(V, c0 + chunk_len);
  const T* p = logits + (size_t)row * V;
  ArgMax best{-INFINITY, 0x7fffffff};
  constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
  int c = c0;
  if (vec_ok) {
    const int nvec = (c1 - c0) / kVec;
    const uint4* pv = reinterpret_cast<const uint4*>(p + c0);
    int t = threadIdx.x;
    // batches of 4 independent 16-byte loads per thread (8 resident CTAs per SM keep ~128 KB
    // in flight per SM), the last batch masked
    constexpr int kUnroll = 4;
    for (; t < nvec; t += kUnroll * kVerifyThreads) {
      uint4 u[kUnroll];
#pragma unroll
      for (int q = 0; q < kUnroll; ++q)
        u[q] = t + q * kVerifyThreads < nvec ? ld_stream(pv + t + q * kVerifyThreads)
                                             : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u,
                                                          0xFF80FF80u);
#pragma unroll
      for (int q = 0; q < kUnroll; ++q) {
        if (t + q * kVerifyThreads >= nvec) break;
        const int base = c0 + (t + q * kVerifyThreads) * kVec;
        if constexpr (sizeof(T) == 2) {
          consider8(best, u[q], base);
        } else {  // strictly larger only: this thread's elements come in index order
          const float f[4] = {__uint_as_float(u[q].x), __uint_as_float(u[q].y),
                              __uint_as_float(u[q].z), __uint_as_float(u[q].w)};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (f[e] > best.v || (best.i == 0x7fffffff && f[e] == best.v)) {
              best.v = f[e];
              best.i = base + e;
            }
        }
      }
    }
    c = c0 + nvec * kVec;
  }
  for (int e = c + threadIdx.x; e < c1; e += kVerifyThreads) consider(best, to_f(p[e]), e);

  // block reduction of (v, i)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best.v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, best.i, o);
    consider(best, ov, oi);
  }
  __shared__ float sv[kVerifyThreads / 32];
  __shared__ int si[kVerifyThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { sv[warp] = best.v; si[warp] = best.i; }
  __syncthreads();
  if (threadIdx.x == 0) {
    ArgMax r = {sv[0], si[0]};
    for (int w = 1; w < kVerifyThreads / 32; ++w) consider(r, sv[w], si[w]);
    part_v[(size_t)row * chunks + chunk] = r.v;
    part_i[(size_t)row * chunks + chunk] = r.i;
  }
}

// One warp per request b: lanes compute the target choices of its S = gamma + 1 rows,
// lane 0 scans the proposals.
__global__ void verify_scan_kernel(const float* __restrict__ part_v, const int* __restrict__ part_i,
                                   int chunks, const int32_t* __restrict__ draft, int B, int gamma,
                                   int32_t eos, int32_t* __restrict__ emitted,
                                   int32_t* __restrict__ num_emitted, int32_t* __restrict__ accepted,
                                   int32_t* __restrict__ choices_out) {
  pdl_wait();
  pdl_trigger();
  const int warps_per_block = blockDim.x >> 5;
  const int b = blockIdx.x * warps_per_block + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const int S = gamma + 1;
  extern __shared__ int sh_choice[];
  int* choice = sh_choice + (threadIdx.x >> 5) * S;
  for (int i = lane; i < S; i += 32) {
    const size_t row = (size_t)b * S + i;
    ArgMax r = {part_v[row * chunks], part_i[row * chunks]};
    for (int c = 1; c < chunks; ++c) consider(r, part_v[row * chunks + c], part_i[row * chunks + c]);
    // an all-NaN row keeps index 0x7fffffff: report index 0 like a first-element argmax
    const int ch = r.i == 0x7fffffff ? 0 : r.i;
    choice[i] = ch;
    if (choices_out) choices_out[row] = ch;
  }
  __syncwarp();
  if (lane == 0) {
    const int32_t* d = draft + (size_t)b * gamma;
    int32_t* em = emitted + (size_t)b * S;
    int n = 0;
    bool stopped = false;
    while (n < gamma && d[n] == choice[n]) {
      em[n] = d[n];
      ++n;
      if (eos >= 0 && d[n - 1] == eos) { stopped = true; break; }
    }
    int count = n;
    if (!stopped) em[count++] = choice[n];  // correction at the mismatch, or the bonus
    for (int e = count; e < S; ++e) em[e] = -1;
    num_emitted[b] = count;
    accepted[b] = n;
  }
}

}  // namespace

VerifyPlan plan_verify_for(long rows, int V, long resident_ctas) {
  VerifyPlan vp;
  // about three waves of resident CTAs, chunks of at least 4096 elements
  long best = (3 * resident_ctas + rows - 1) / rows;
  const long max_chunks = (V + 4095) / 4096;
  if (best > max_chunks) best = max_chunks;
  if (best < 1) best = 1;
  long len = (V + best - 1) / best;
  len = (len + 7) / 8 * 8;
  vp.chunk_len = (int)len;
  vp.chunks = (int)((V + len - 1) / len);
  vp.ws_bytes = (size_t)rows * vp.chunks * (sizeof(float) + sizeof(int));
  return vp;
}

VerifyPlan cap_verify_chunks(VerifyPlan vp, long rows, int V, long max_entries) {
  if ((long)vp.chunks * rows <= max_entries) return vp;
  // fewer, longer chunks: at most max_entries / rows of them, each a multiple of 8
  // elements (16-byte aligned vector loads); ceil(V / len) <= that count since
  // len >= V / count
  const long chunks = max_entries / rows;
  long len = ((long)V + chunks - 1) / chunks;
  len = (len + 7) / 8 * 8;
  vp.chunk_len = (int)len;
  vp.chunks = (int)(((long)V + len - 1) / len);
  vp.ws_bytes = (size_t)rows * vp.chunks * (sizeof(float) + sizeof(int));
  return vp;
}

VerifyPlan plan_verify(int B, int gamma, int V, int num_sms) {
  const long rows = (long)B * (gamma + 1);
  // resident argmax CTAs per SM, looked up once per device
  static std::atomic<int> per_sm_cache[kMaxVerifyDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxVerifyDevices) dev = -1;
  int per_sm = dev >= 0 ? per_sm_cache[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, argmax_partial_kernel<__nv_bfloat16>,
                                                      kVerifyThreads, 0) != cudaSuccess || n < 1) {
      cudaGetLastError();  // no device here: plan with a typical occupancy
      n = 4;
    } else if (dev >= 0) {
      per_sm_cache[dev].store(n, std::memory_order_relaxed);
    }
    per_sm = n;
  }
  return plan_verify_for(rows, V, (long)per_sm * (num_sms > 0 ? num_sms : 1));
}

cudaError_t launch_verify(const void* logits, int dtype, const int32_t* draft, int B, int gamma,
                          int V, int32_t eos, int32_t* emitted, int32_t* num_emitted,
                          int32_t* accepted, int32_t* choices, float* part_v, int* part_i,
                          const VerifyPlan& vp, cudaStream_t stream) {
  const int rows = B * (gamma + 1);
  dim3 grid(vp.chunks, rows);
  const size_t elem = dtype == DFLASH_DTYPE_BF16 ? 2 : 4;
  const bool vec_ok = ((uintptr_t)logits % 16 == 0) && ((size_t)V * elem % 16 == 0) &&
                      ((size_t)vp.chunk_len * elem % 16 == 0);
  const cudaError_t le =
      dtype == DFLASH_DTYPE_BF16
          ? launch_pdl(argmax_partial_kernel<__nv_bfloat16>, dim3(grid), dim3(kVerifyThreads), 0,
                       stream, (const __nv_bfloat16*)logits, V, vp.chunks, vp.chunk_len, vec_ok,
                       part_v, part_i)
          : launch_pdl(argmax_partial_kernel<float>, dim3(grid), dim3(kVerifyThreads), 0, stream,
                       (const float*)logits, V, vp.chunks, vp.chunk_len, vec_ok, part_v, part_i);
  if (le != cudaSuccess) return le;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int warps = B < 4 ? B : 4;
  const size_t smem = (size_t)warps * (gamma + 1) * sizeof(int);
  if (smem > kScanSmemDefault) {
    if (smem > kScanSmemMax) return cudaErrorInvalidValue;  // rejected on the host first
    const cudaError_t ae = cudaFuncSetAttribute(
        verify_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (ae != cudaSuccess) return ae;
  }
  e = launch_pdl(verify_scan_kernel, dim3((B + warps - 1) / warps), dim3(warps * 32), smem, stream,
                 part_v, part_i, vp.chunks, draft, B, gamma, eos, emitted, num_emitted, accepted,
                 choices);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dflash

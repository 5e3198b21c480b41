// Shared device/host helpers of libdflash (no method arithmetic here).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"

namespace dflash {

// ---- device status word ------------------------------------------------------------
// One sticky word per device (defined in api.cu).  Kernels receive its address as a
// parameter.  Bit layout: bit 0 = a bounded wait ran out, bit 1 = an index check failed;
// bits 8..15 = id of the first kernel that reported (kernel ids below).
enum : unsigned {
  kStatusTimeout = 1u,
  kStatusCheck = 2u,
  kStatusRange = 4u,  // a value outside the fp16 range met an fp16 store
};
enum : unsigned {
  kKernPlan = 1, kKernVerify = 2, kKernGemmTc = 3, kKernAttn = 4, kKernEpilogue = 5,
  kKernNorm = 6, kKernAttnTc = 7, kKernActivation = 8, kKernConvert = 9,
};

__device__ __forceinline__ void report(unsigned* status, unsigned bit, unsigned kernel_id) {
  if (status) {
    unsigned prev = atomicOr(status, bit);
    if ((prev & 0xFF00u) == 0) atomicOr(status, kernel_id << 8);
  }
}

// ---- element types -------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f(float v) { return v; }
  static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

template <> struct Elem<__half> {
  static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
  static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
};

template <typename T> __device__ __forceinline__ float to_f(T v) { return Elem<T>::to_f(v); }
template <typename T> __device__ __forceinline__ T from_f(float v) { return Elem<T>::from_f(v); }

// Destination of a computed activation that feeds a projection GEMM: one fp32 array in the
// fp32 configuration; one IEEE fp16 array in the bf16 configuration, where the draft layers'
// projections run fp16 x fp16 on the tensor cores.  fp16 keeps 11 significant bits (8 times
// finer than bf16); a value outside its finite range is stored as +-inf / NaN and reported
// through the status word (kStatusRange).
struct ActOut {
  void* p = nullptr;
  int dtype = DFLASH_DTYPE_F32;
  unsigned* status = nullptr;
  __device__ __forceinline__ void range_check(float v) const {
    if (!(fabsf(v) < 65520.f)) report(status, kStatusRange, kKernActivation);
  }
  __device__ __forceinline__ void store(long i, float v) const {
    if (dtype == DFLASH_DTYPE_BF16) {
      range_check(v);
      static_cast<__half*>(p)[i] = __float2half_rn(v);
    } else {
      static_cast<float*>(p)[i] = v;
    }
  }
  // four consecutive elements starting at i (i a multiple of 4)
  __device__ __forceinline__ void store4(long i, float4 v) const {
    if (dtype == DFLASH_DTYPE_BF16) {
      // fmaxf drops NaN operands; the product term is NaN when an element is NaN or inf
      range_check(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))) +
                  0.f * (v.x + v.y + v.z + v.w));
      const __half2 h01 = __floats2half2_rn(v.x, v.y);
      const __half2 h23 = __floats2half2_rn(v.z, v.w);
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t*>(&h01);
      w.y = *reinterpret_cast<const uint32_t*>(&h23);
      *reinterpret_cast<uint2*>(static_cast<__half*>(p) + i) = w;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(p) + i) = v;
    }
  }
};

// Four consecutive elements of a bf16 or fp32 array as fp32 (i a multiple of 4).
__device__ __forceinline__ float4 load4(const void* p, int dtype, long i) {
  if (dtype == DFLASH_DTYPE_BF16) {
    const uint2 w = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p) + i);
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
}

// ---- reductions --------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the block; every thread gets the result.  `red` holds >= 33 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float t = lane < nwarps ? red[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) red[32] = t;
  }
  __syncthreads();
  return red[32];
}

// ---- programmatic dependent launch ----------------------------------------------------------
// Kernels of the hot path are launched with programmatic stream serialization: a kernel may
// start (its prologue, its launch latency) while its predecessor on the stream finishes.
// pdl_wait() blocks until every predecessor grid has completed and its memory is visible;
// each such kernel calls it before its first global-memory access.  pdl_trigger() lets the
// successor grid be scheduled once every CTA of this grid has called it (or exited).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- time-bounded waits ----------------------------------------------------------------
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Any device-side wait gives up after this long and reports kStatusTimeout.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

}  // namespace dflash

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
// the fp32 configuration, else the two-term bf16 pair (hi, lo) the tensor-core GEMM
// consumes.  Attention operands (q, block k / v) are kept in fp32.
#include "common.cuh"
#include "internal.h"

namespace dflash {

namespace {

constexpr double kTwoPi = 6.283185307179586476925286766559;

__device__ __forceinline__ float ld(const void* p, int dt, long i) {
  return dt == DFLASH_DTYPE_BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i])
                                 : static_cast<const float*>(p)[i];
}

__device__ __forceinline__ void st(void* p, int dt, long i, float v) {
  if (dt == DFLASH_DTYPE_BF16) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  else static_cast<float*>(p)[i] = v;
}

__global__ void rope_table_kernel(float* __restrict__ cos_t, float* __restrict__ sin_t, int p0,
                                  int P, int half, int head_dim, double theta) {
  const long n = (long)P * half;
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const int p = (int)(e / half), i = (int)(e - (long)p * half);
    const double inv_freq = pow(theta, -2.0 * (double)i / (double)head_dim);
    const double ang = (double)(p0 + p) * inv_freq;
    // reduce to [-pi, pi] in fp64, then evaluate in fp32
    const double r = fma(-rint(ang / kTwoPi), kTwoPi, ang);
    float s, c;
    sincosf((float)r, &s, &c);
    cos_t[e] = c;
    sin_t[e] = s;
  }
}

__global__ void residual_norm_kernel(int mode, int dt, float* __restrict__ x,
                                     const void* __restrict__ emb, const float* __restrict__ y,
                                     int nsplit, long split_stride, const void* __restrict__ g,
                                     float eps, ActOut h, float* __restrict__ out,
                                     const uint8_t* __restrict__ valid, bool final_norm, int D) {
  __shared__ float red[33];
  const long r = blockIdx.x;
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
    xr[c] = v;
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

// one thread per (row t, head, channel pair i); q / k / v are written in fp32
__global__ void qkv_rope_kernel(const float* __restrict__ y, int nsplit, long split_stride,
                                const int32_t* __restrict__ pos, const uint8_t* __restrict__ valid,
                                const float* __restrict__ cos_t, const float* __restrict__ sin_t,
                                int P, float* __restrict__ q, float* __restrict__ k,
                                float* __restrict__ v, long T, int Hq, int Hkv, int dh,
                                unsigned* status) {
  const int half = dh / 2;
  const int heads = Hq + 2 * Hkv;
  const long width = (long)heads * dh;
  const long n = T * heads * half;
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const long t = e / ((long)heads * half);
    const int rem = (int)(e - t * heads * half);
    const int hd = rem / half, i = rem - hd * half;
    const long base = t * width + (long)hd * dh;
    const float a = sum_splits(y, nsplit, split_stride, base + i);
    const float bb = sum_splits(y, nsplit, split_stride, base + i + half);
    if (hd >= Hq + Hkv) {  // V: no rotation
      const long o = t * Hkv * dh + (long)(hd - Hq - Hkv) * dh;
      v[o + i] = a;
      v[o + i + half] = bb;
      continue;
    }
    int p = pos[t];
    if (p < 0 || p >= P) {
      if (valid[t] && i == 0) report(status, kStatusCheck, kKernEpilogue);
      p = 0;
    }
    const float c = cos_t[(long)p * half + i], s = sin_t[(long)p * half + i];
    const float lo = a * c - bb * s, hi = bb * c + a * s;
    if (hd < Hq) {
      const long o = t * Hq * dh + (long)hd * dh;
      q[o + i] = lo;
      q[o + i + half] = hi;
    } else {
      const long o = t * Hkv * dh + (long)(hd - Hq) * dh;
      k[o + i] = lo;
      k[o + i + half] = hi;
    }
  }
}

// one thread per (b, c, kv, head, pair i); the cache is stored in the configuration dtype
__global__ void ctx_kv_scatter_kernel(int dt, const float* __restrict__ y, int nsplit,
                                      long split_stride, const float* __restrict__ cos_t,
                                      const float* __restrict__ sin_t, void* __restrict__ kv,
                                      int B, int L, int pos_offset, int L_cache, int Hkv, int dh) {
  const int half = dh / 2;
  const long per_row = 2L * Hkv * half;
  const long n = (long)B * L * per_row;
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const long bc = e / per_row;
    const int rem = (int)(e - bc * per_row);
    const int hd = rem / half, i = rem - hd * half;  // hd in [0, 2*Hkv): K heads then V heads
    const int b = (int)(bc / L), c = (int)(bc - (long)b * L);
    const long src = bc * 2L * Hkv * dh + (long)hd * dh;
    float a = sum_splits(y, nsplit, split_stride, src + i);
    float bb = sum_splits(y, nsplit, split_stride, src + i + half);
    const int kvsel = hd / Hkv, g = hd - kvsel * Hkv;
    const int p = pos_offset + c;
    if (kvsel == 0) {  // table row c holds position pos_offset + c
      const float cs = cos_t[(long)c * half + i], sn = sin_t[(long)c * half + i];
      const float lo = a * cs - bb * sn, hi = bb * cs + a * sn;
      a = lo;
      bb = hi;
    }
    const long dst = ((((long)b * 2 + kvsel) * Hkv + g) * L_cache + p) * dh;
    st(kv, dt, dst + i, a);
    st(kv, dt, dst + i + half, bb);
  }
}

__global__ void swiglu_kernel(const float* __restrict__ y, int nsplit, long split_stride,
                              ActOut act, long T, int I) {
  const long n = T * I;
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const long t = e / I;
    const int i = (int)(e - t * I);
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
                              double theta, cudaStream_t stream) {
  const long n = (long)P * (head_dim / 2);
  rope_table_kernel<<<grid_for(n, 256), 256, 0, stream>>>(cos_t, sin_t, p0, P, head_dim / 2,
                                                          head_dim, theta);
  return cudaGetLastError();
}

cudaError_t launch_residual_norm(int mode, int dtype, float* x, const void* emb, const float* y,
                                 int nsplit, const void* g, double eps, ActOut h, float* out,
                                 const uint8_t* valid, bool final_norm, long rows, int D,
                                 cudaStream_t stream) {
  const int threads = D >= 2048 ? 512 : 256;
  residual_norm_kernel<<<rows, threads, 0, stream>>>(mode, dtype, x, emb, y, nsplit, rows * D, g,
                                                     (float)eps, h, out, valid, final_norm, D);
  return cudaGetLastError();
}

cudaError_t launch_rows_norm(int dtype, const float* y, int nsplit, const void* g, double eps,
                             bool with_norm, ActOut out, long rows, int D, cudaStream_t stream) {
  const int threads = D >= 2048 ? 512 : 256;
  rows_norm_kernel<<<rows, threads, 0, stream>>>(dtype, y, nsplit, rows * D, g, (float)eps,
                                                 with_norm, out, D);
  return cudaGetLastError();
}

cudaError_t launch_qkv_rope(const float* y, int nsplit, const int32_t* pos, const uint8_t* valid,
                            const float* cos_t, const float* sin_t, int P, float* q, float* k,
                            float* v, long T, int Hq, int Hkv, int dh, unsigned* status,
                            cudaStream_t stream) {
  const long n = T * (Hq + 2 * Hkv) * (dh / 2);
  const long stride = T * (long)(Hq + 2 * Hkv) * dh;
  qkv_rope_kernel<<<grid_for(n, 256), 256, 0, stream>>>(y, nsplit, stride, pos, valid, cos_t,
                                                        sin_t, P, q, k, v, T, Hq, Hkv, dh, status);
  return cudaGetLastError();
}

cudaError_t launch_ctx_kv_scatter(int dtype, const float* y, int nsplit, const float* cos_t,
                                  const float* sin_t, void* kv_layer, int B, int L,
                                  int pos_offset, int L_cache, int Hkv, int dh,
                                  cudaStream_t stream) {
  const long n = (long)B * L * 2 * Hkv * (dh / 2);
  const long stride = (long)B * L * 2 * Hkv * dh;
  ctx_kv_scatter_kernel<<<grid_for(n, 256), 256, 0, stream>>>(
      dtype, y, nsplit, stride, cos_t, sin_t, kv_layer, B, L, pos_offset, L_cache, Hkv, dh);
  return cudaGetLastError();
}

cudaError_t launch_swiglu(const float* y, int nsplit, ActOut act, long T, int I,
                          cudaStream_t stream) {
  const long n = T * I;
  swiglu_kernel<<<grid_for(n, 256), 256, 0, stream>>>(y, nsplit, T * 2L * I, act, T, I);
  return cudaGetLastError();
}

}  // namespace dflash

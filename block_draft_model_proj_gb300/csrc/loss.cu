// Draft training loss over the drafted blocks: the frozen lm_head's cross-entropy against the
// ground-truth tokens with an exponential positional decay, over loss_mask.
//
// "DFlash" (How it works, Loss): cross-entropy with an exponential positional decay that
// weights earlier in-block positions more heavily.  "DFlash Draft Body" (How It Works step 4):
// the loss mask excludes the anchor and invalid positions.  The pages give no decay constant:
// slot j >= 1 weighs exp(-(j - 1) / decay), decay a caller argument; loss = sum(m w CE) /
// sum(m w).
//
// The logits (T x V, 151936 columns) are never stored.  The body's fp32 hidden states are
// rounded to bf16 (rows outside the loss mask to zero); the tensor-core GEMM against the bf16
// lm_head computes each 128 x 256 logits tile in tensor memory and its epilogue reduces the
// tile to (max, sum of exp(logit - max)) per row plus the target's logit.  One warp per row
// then merges the tiles in a fixed order (log-sum-exp) and one CTA sums the weighted
// per-slot losses in a fixed order (fp64 accumulators): deterministic.
#include "common.cuh"
#include "internal.h"

namespace dflash {

namespace {

// hidden fp32 [T][D] -> bf16 (round to nearest even); rows outside the mask to zero.
__global__ void hidden_to_bf16_kernel(const float* __restrict__ h, const uint8_t* __restrict__ mask,
                                      __nv_bfloat16* __restrict__ out, long T, int D) {
  pdl_wait();
  pdl_trigger();
  const int D4 = D / 4;
  const long n = T * D4;
  for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < n;
       e += (long)gridDim.x * blockDim.x) {
    const long t = e / D4;
    const int q = (int)(e - t * D4);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mask[t]) v = *reinterpret_cast<const float4*>(h + t * D + 4L * q);
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&a);
    w.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(out + t * D + 4L * q) = w;
  }
}

__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * expf(m2 - m);
  }
}

// One warp per row: CE = log-sum-exp over the vocab tiles - the target's logit.  Lanes merge
// tiles lane, lane + 32, ... in order, then a fixed butterfly: the same order every call.
__global__ void ce_rows_kernel(const float* __restrict__ part, const float* __restrict__ tlogit,
                               const int32_t* __restrict__ targets,
                               const uint8_t* __restrict__ mask, long T, int n_tiles, int V,
                               float* __restrict__ ce, unsigned* status) {
  pdl_wait();
  pdl_trigger();
  const long t = blockIdx.x * (long)(blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  if (!mask[t]) {
    if (lane == 0) ce[t] = 0.f;
    return;
  }
  const int y = targets[t];
  if (y < 0 || y >= V) {
    if (lane == 0) {
      report(status, kStatusCheck, kKernEpilogue);
      ce[t] = 0.f;
    }
    return;
  }
  float m = -INFINITY, s = 0.f;
  for (int i = lane; i < n_tiles; i += 32)
    merge_ms(m, s, part[((size_t)t * n_tiles + i) * 2], part[((size_t)t * n_tiles + i) * 2 + 1]);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    // both partners merge in the same (lower lane first) order
    if (lane & o) {
      float mm = m2, ss = s2;
      merge_ms(mm, ss, m, s);
      m = mm;
      s = ss;
    } else {
      merge_ms(m, s, m2, s2);
    }
  }
  if (lane == 0) ce[t] = m + logf(s) - tlogit[t];
}

// One CTA: loss = sum(mask * w_j * ce) / sum(mask * w_j), j = t mod S; fp64 accumulation in
// a fixed order.
__global__ void __launch_bounds__(1024) ce_loss_kernel(const float* __restrict__ ce,
                                                       const uint8_t* __restrict__ mask, long T,
                                                       int S, double inv_decay,
                                                       float* __restrict__ loss) {
  pdl_wait();
  pdl_trigger();
  __shared__ double sn[1024], sd[1024];
  double num = 0.0, den = 0.0;
  for (long t = threadIdx.x; t < T; t += blockDim.x) {
    const int j = (int)(t % S);
    if (!mask[t] || j == 0) continue;
    const double w = exp(-(double)(j - 1) * inv_decay);
    num += w * (double)ce[t];
    den += w;
  }
  sn[threadIdx.x] = num;
  sd[threadIdx.x] = den;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) {
      sn[threadIdx.x] += sn[threadIdx.x + o];
      sd[threadIdx.x] += sd[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = sd[0] > 0.0 ? (float)(sn[0] / sd[0]) : 0.f;
}

}  // namespace

CeLayout ce_layout(long T, int D, int V, void* ws) {
  CeLayout l;
  uint8_t* base = static_cast<uint8_t*>(ws);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    off = (off + 255) & ~(size_t)255;
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  };
  l.n_tiles = (V + 255) / 256;
  l.hidden16 = static_cast<__nv_bfloat16*>(take((size_t)T * D * 2));
  l.part = static_cast<float*>(take((size_t)T * l.n_tiles * 2 * sizeof(float)));
  l.tlogit = static_cast<float*>(take((size_t)T * sizeof(float)));
  l.tile_list = static_cast<int32_t*>(take((1 + (size_t)(T + kGemmTileM - 1) / kGemmTileM) *
                                           sizeof(int32_t)));
  l.bytes = off;
  return l;
}

cudaError_t launch_decayed_ce(const float* hidden, const void* lm_head, const int32_t* targets,
                              const uint8_t* mask, long T, int S, int D, int V, double decay,
                              float* ce, float* loss, const CeLayout& l, unsigned* status,
                              cudaStream_t stream) {
  cudaError_t e;
  {
    long n = T * (D / 4);
    long g = (n + 255) / 256;
    if (g > 152L * 16) g = 152L * 16;
    if (g < 1) g = 1;
    e = launch_pdl(hidden_to_bf16_kernel, dim3((unsigned)g), dim3(256), 0, stream, hidden, mask,
                   l.hidden16, T, D);
    if (e != cudaSuccess) return e;
  }
  e = launch_slot_tile_list(mask, T, l.tile_list, stream);
  if (e != cudaSuccess) return e;
  CrossEntropyEpilogue ep;
  ep.targets = targets;
  ep.part = l.part;
  ep.target_logit = l.tlogit;
  e = launch_gemm_tc_cross_entropy(l.hidden16, D, lm_head, D, T, V, D, l.tile_list, ep, status,
                                   stream);
  if (e != cudaSuccess) return e;
  const int warps = 8;
  e = launch_pdl(ce_rows_kernel, dim3((unsigned)((T + warps - 1) / warps)), dim3(warps * 32), 0,
                 stream, (const float*)l.part, (const float*)l.tlogit, targets, mask, T,
                 l.n_tiles, V, ce, status);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ce_loss_kernel, dim3(1), dim3(1024), 0, stream, (const float*)ce, mask, T, S,
                 1.0 / decay, loss);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dflash

// Speculative-sampling verification of drafted blocks.
//
// "DFlash: drafting, verification, and speed", Sampling with temperature is not argmax
// matching: for the target distribution p, the ACTUAL proposal distribution q and a proposal
// y ~ q, accept with probability min(1, p(y) / q(y)); on rejection, sample from the
// normalised residual [p - q]_+.  Proposals are tested in block order and the block stops at
// the first rejection.  When every proposal is accepted the block ends with a sample of the
// last target distribution (the counterpart of greedy verification's bonus); a matched EOS
// proposal ends the block as in greedy verification.
//
// p_i = softmax(logits[b, i] / temperature).  Random numbers: a counter-based uniform, the
// SplitMix64 finaliser (Steele, Lea & Flood, OOPSLA 2014) chained over (seed, counters...),
// top 23 bits plus one half times 2^-23 -- exact in fp32.  Acceptance of proposal i of
// request b draws U(seed, b, i, 0).  Samples use the exponential race: index v arrives at
// E_v / w_v with E_v = -ln U(seed, b, i, 1, v); the first arrival is an exact draw from
// w / sum(w) (lowest index on an exact tie), so no normalisation or prefix sum is needed.
//
// All softmax arithmetic runs in base 2 on the special-function unit: y = logit *
// log2(e) / temperature, p = 2^(y - max) / sum 2^(y - max).
// Kernel 1 (HBM-bound, one pass over every logits row): per (row, chunk) the maximum of y
//   and the sum of 2^(y - max), merged online (each 16-byte vector: its maximum first, one
//   rescale, then its exponentials).
// Kernel 2 (one warp per request): rows' (max, sum) from their chunks in chunk order; the
//   acceptance scan in block order (p(y) from the row's statistics, q(y) read directly);
//   writes the accepted proposals and which row, if any, is sampled.
// Kernel 3 (per (request, chunk)): the race over that row -- weights [p - q]_+ after a
//   rejection, p for the final sample -- to a (key, index) pair per chunk; a residual that
//   is zero everywhere (p == q, possible only through rounding) falls back to p, whose
//   race is run in the same pass from the same arrival draws.  Arrival E_v / w_v is ranked
//   as -log2(U_v) / w_v (the factor ln 2 is common to all v); the race of p is ranked as
//   y_v - log2(-log2 U_v), the logarithm of the reciprocal arrival up to constants (the
//   Gumbel form: no exponential, no division), which orders the indices identically.
// Kernel 4 (one thread per request): the first arrival over the chunks, in chunk order.
#include "common.cuh"
#include "internal.h"

namespace dflash {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// uniform in (0, 1) on the 2^-23 grid, exact in fp32
__device__ __forceinline__ float grid_uniform(uint64_t h) {
  return ((float)(uint32_t)(h >> 41) + 0.5f) * (1.0f / 8388608.0f);
}

template <typename T>
__device__ __forceinline__ float logit_at(const T* p, long i) {
  return to_f(p[i]);
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2f(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (max, sum of 2^(y - max)) merge
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * ex2f(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * ex2f(m2 - m);
  }
}

// the (max, sum) of n more values y[0..n-1] (a -inf value adds nothing)
template <int n>
__device__ __forceinline__ void push_n(float& m, float& s, const float* y) {
  float lm = y[0];
#pragma unroll
  for (int e = 1; e < n; ++e) lm = fmaxf(lm, y[e]);
  if (lm == -INFINITY) return;
  if (lm > m) {
    s = m == -INFINITY ? 0.f : s * ex2f(m - lm);
    m = lm;
  }
#pragma unroll
  for (int e = 0; e < n; ++e) s += ex2f(y[e] - m);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
softmax_stats_kernel(const T* __restrict__ logits, int V, int chunks, int chunk_len, bool vec_ok,
                     float inv_temp, float* __restrict__ part_m, float* __restrict__ part_s) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.y, chunk = blockIdx.x;
  const int c0 = chunk * chunk_len, c1 = min(V, c0 + chunk_len);
  const T* p = logits + (size_t)row * V;
  float m = -INFINITY, s = 0.f;
  int c = c0;
  if (vec_ok) {
    // 16-byte loads: 8 bf16 or 4 fp32 values
    constexpr int kVec = 16 / sizeof(T);
    const int nvec = (c1 - c0) / kVec;
    const uint4* pv = reinterpret_cast<const uint4*>(p + c0);
    for (int t = threadIdx.x; t < nvec; t += kThreads) {
      const uint4 u = __ldcs(pv + t);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      if constexpr (sizeof(T) == 2) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y[2 * e] = __uint_as_float(w[e] << 16) * inv_temp;
          y[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u) * inv_temp;
        }
        push_n<8>(m, s, y);
      } else {
        float y[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = __uint_as_float(w[e]) * inv_temp;
        push_n<4>(m, s, y);
      }
    }
    c = c0 + nvec * kVec;
  }
  for (int v = c + threadIdx.x; v < c1; v += kThreads) {
    const float y = logit_at(p, v) * inv_temp;
    push_n<1>(m, s, &y);
  }
  // block merge of the (max, sum) pairs, in a fixed order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    merge_ms(m, s, m2, s2);
  }
  __shared__ float sm[kThreads / 32], ss[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sm[warp] = m;
    ss[warp] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w2 = 1; w2 < kThreads / 32; ++w2) merge_ms(m, s, sm[w2], ss[w2]);
    part_m[(size_t)row * chunks + chunk] = m;
    part_s[(size_t)row * chunks + chunk] = s;
  }
}

struct SamplePlan {
  int row;    // row of the block to sample (-1: no sample, the block ended at an EOS)
  int mode;   // 0: residual [p - q]_+ after a rejection, 1: the final sample of p
  float m, z; // the row's softmax statistics
};

template <typename T>
__global__ void sampling_scan_kernel(const T* __restrict__ logits, const float* __restrict__ q,
                                     const float* __restrict__ part_m,
                                     const float* __restrict__ part_s, int chunks,
                                     const int32_t* __restrict__ draft, int B, int gamma, int V,
                                     float inv_temp, uint64_t seed, int32_t eos,
                                     int32_t* __restrict__ emitted,
                                     int32_t* __restrict__ num_emitted,
                                     int32_t* __restrict__ accepted, SamplePlan* __restrict__ plan,
                                     unsigned* status) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const int S = gamma + 1;
  const int32_t* d = draft + (size_t)b * gamma;
  int32_t* em = emitted + (size_t)b * S;
  const uint64_t hb = mix64(mix64(seed) ^ (uint64_t)(int64_t)b);
  int n = 0;
  int stop = S;     // first rejected proposal, S: none
  bool eos_stop = false;
  // lanes test the proposals in groups of 32; the first group with a rejection or an EOS
  // ends the scan (the outcome of every earlier proposal is an acceptance)
  for (int i0 = 0; i0 < gamma && stop == S && !eos_stop; i0 += 32) {
    const int i = i0 + lane;
    bool acc_i = false, is_eos = false;
    if (i < gamma) {
      const int y = d[i];
      if (y < 0 || y >= V) {
        report(status, kStatusCheck, kKernVerify);
      } else {
        float M = -INFINITY, Z = 0.f;
        const size_t row = (size_t)b * S + i;
        for (int c = 0; c < chunks; ++c) merge_ms(M, Z, part_m[row * chunks + c], part_s[row * chunks + c]);
        const float py = ex2f(logit_at(logits + row * V, y) * inv_temp - M) / Z;
        const float qy = q[((size_t)b * gamma + i) * V + y];
        const float u = grid_uniform(mix64(mix64(hb ^ (uint64_t)i) ^ 0ull));
        acc_i = u * qy < py;
        is_eos = eos >= 0 && y == eos;
      }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, i < gamma && !acc_i);
    const unsigned eosm = __ballot_sync(0xffffffffu, i < gamma && acc_i && is_eos);
    // the first stopping event in this group: a rejection at r, or an accepted EOS at e
    const int r = rej ? __ffs(rej) - 1 : 32;
    const int e = eosm ? __ffs(eosm) - 1 : 32;
    if (e < r) {
      n = i0 + e + 1;
      eos_stop = true;
    } else if (r < 32) {
      n = i0 + r;
      stop = i0 + r;
    } else {
      n = min(gamma, i0 + 32);
    }
  }
  for (int i = lane; i < n; i += 32) em[i] = d[i];
  if (lane == 0) {
    accepted[b] = n;
    SamplePlan sp;
    sp.row = -1;
    sp.mode = 1;
    sp.m = -INFINITY;
    sp.z = 0.f;
    if (!eos_stop) {
      sp.row = stop < S ? stop : gamma;
      sp.mode = stop < S ? 0 : 1;
      const size_t row = (size_t)b * S + sp.row;
      for (int c = 0; c < chunks; ++c) merge_ms(sp.m, sp.z, part_m[row * chunks + c], part_s[row * chunks + c]);
    }
    plan[b] = sp;
    num_emitted[b] = eos_stop ? n : n + 1;  // the sample fills slot n (kernel 4)
  }
  for (int i = (eos_stop ? n : n + 1) + lane; i < S; i += 32) em[i] = -1;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
race_kernel(const T* __restrict__ logits, const float* __restrict__ q,
            const SamplePlan* __restrict__ plan, int gamma, int V, int chunks, int chunk_len,
            bool vec_ok, float inv_temp, uint64_t seed, float* __restrict__ race_t,
            int* __restrict__ race_i, float* __restrict__ race_tp, int* __restrict__ race_ip) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y, chunk = blockIdx.x;
  const SamplePlan sp = plan[b];
  const size_t out = (size_t)b * chunks + chunk;
  if (sp.row < 0) {
    if (threadIdx.x == 0) {
      race_t[out] = INFINITY;
      race_i[out] = 0x7fffffff;
      race_tp[out] = INFINITY;
      race_ip[out] = 0x7fffffff;
    }
    return;
  }
  const int S = gamma + 1;
  const T* lrow = logits + ((size_t)b * S + sp.row) * V;
  const float* qrow = sp.mode == 0 ? q + ((size_t)b * gamma + sp.row) * V : nullptr;
  const uint64_t hr = mix64(mix64(mix64(mix64(seed) ^ (uint64_t)(int64_t)b) ^ (uint64_t)sp.row) ^ 1ull);
  const float inv_z = 1.f / sp.z;
  const int c0 = chunk * chunk_len, c1 = min(V, c0 + chunk_len);
  // ranking keys, smaller first: after a rejection -log2(U) / [p - q]_+ for the residual and
  // -(y - log2(-log2 U)) for the fallback race of p; for the final sample the latter alone.
  // Both from the same draw U_v.
  float bt = INFINITY, btp = INFINITY;
  int bi = 0x7fffffff, bip = 0x7fffffff;
  auto consider = [&](int v, float y, float qv) {
    if (y == -INFINITY) return;                         // p_v = 0
    const float nl = -lg2f(grid_uniform(mix64(hr ^ (uint64_t)v)));   // -log2 U > 0
    const float tp = lg2f(nl) - (y - sp.m);             // Gumbel form of the race of p
    if (qrow) {
      const float w = ex2f(y - sp.m) * inv_z - qv;
      if (w > 0.f) {
        const float t = __fdividef(nl, w);
        if (t < bt) { bt = t; bi = v; }   // a thread's indices increase: strict < keeps the lowest
      }
      if (tp < btp) { btp = tp; bip = v; }
    } else if (tp < bt) {
      bt = tp;
      bi = v;
    }
  };
  int v0 = c0;
  if constexpr (sizeof(T) == 2) {
    if (vec_ok) {
      // 8 consecutive entries per thread and step: one 16-byte load of logits (and two of q),
      // all loads of a step issued before the arithmetic
      const int nvec = (c1 - c0) / 8;
      for (int t = threadIdx.x; t < nvec; t += kThreads) {
        const int v = c0 + 8 * t;
        const uint4 u = __ldcs(reinterpret_cast<const uint4*>(lrow + v));
        float4 qa = make_float4(0.f, 0.f, 0.f, 0.f), qb = qa;
        if (qrow) {
          qa = __ldcs(reinterpret_cast<const float4*>(qrow + v));
          qb = __ldcs(reinterpret_cast<const float4*>(qrow + v + 4));
        }
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t bits = (e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16);
          consider(v + e, __uint_as_float(bits) * inv_temp, qv[e]);
        }
      }
      v0 = c0 + nvec * 8;
    }
  }
  for (int v = v0 + threadIdx.x; v < c1; v += kThreads)
    consider(v, logit_at(lrow, v) * inv_temp, qrow ? qrow[v] : 0.f);
  // block minimum of (time, index), lowest index on equal times
  __shared__ float st[kThreads / 32], stp[kThreads / 32];
  __shared__ int si[kThreads / 32], sip[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float t2 = __shfl_xor_sync(0xffffffffu, bt, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (t2 < bt || (t2 == bt && i2 < bi)) { bt = t2; bi = i2; }
    const float tp2 = __shfl_xor_sync(0xffffffffu, btp, o);
    const int ip2 = __shfl_xor_sync(0xffffffffu, bip, o);
    if (tp2 < btp || (tp2 == btp && ip2 < bip)) { btp = tp2; bip = ip2; }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    st[warp] = bt;
    si[warp] = bi;
    stp[warp] = btp;
    sip[warp] = bip;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w2 = 1; w2 < kThreads / 32; ++w2) {
      if (st[w2] < bt || (st[w2] == bt && si[w2] < bi)) { bt = st[w2]; bi = si[w2]; }
      if (stp[w2] < btp || (stp[w2] == btp && sip[w2] < bip)) { btp = stp[w2]; bip = sip[w2]; }
    }
    race_t[out] = bt;
    race_i[out] = bi;
    race_tp[out] = btp;
    race_ip[out] = bip;
  }
}

// One warp per request: lanes take chunks c = lane, lane + 32, ..., then a butterfly; the
// winner is the smallest key, the lowest index on equal keys -- the same whatever the order.
__global__ void race_finish_kernel(const SamplePlan* __restrict__ plan,
                                   const float* __restrict__ race_t, const int* __restrict__ race_i,
                                   const float* __restrict__ race_tp,
                                   const int* __restrict__ race_ip, int chunks, int B, int gamma,
                                   const int32_t* __restrict__ accepted,
                                   int32_t* __restrict__ emitted) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B || plan[b].row < 0) return;
  float bt = INFINITY, btp = INFINITY;
  int bi = 0x7fffffff, bip = 0x7fffffff;
  for (int c = lane; c < chunks; c += 32) {
    const size_t k = (size_t)b * chunks + c;
    const float t = race_t[k], tp = race_tp[k];
    const int i = race_i[k], ip = race_ip[k];
    if (t < bt || (t == bt && i < bi)) { bt = t; bi = i; }
    if (tp < btp || (tp == btp && ip < bip)) { btp = tp; bip = ip; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float t2 = __shfl_xor_sync(0xffffffffu, bt, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (t2 < bt || (t2 == bt && i2 < bi)) { bt = t2; bi = i2; }
    const float tp2 = __shfl_xor_sync(0xffffffffu, btp, o);
    const int ip2 = __shfl_xor_sync(0xffffffffu, bip, o);
    if (tp2 < btp || (tp2 == btp && ip2 < bip)) { btp = tp2; bip = ip2; }
  }
  if (lane == 0) {
    // an empty residual (p == q after rounding) samples p instead
    int tok = bi != 0x7fffffff ? bi : bip;
    if (tok == 0x7fffffff) tok = 0;
    emitted[(size_t)b * (gamma + 1) + accepted[b]] = tok;
  }
}

}  // namespace

SamplingPlan plan_sampling(int B, int gamma, int V, int num_sms) {
  SamplingPlan sp;
  const VerifyPlan vp = plan_verify(B, gamma, V, num_sms);
  sp.chunks = vp.chunks;
  sp.chunk_len = vp.chunk_len;
  // the race covers one row per request: about two waves of four resident 256-thread CTAs
  // per SM over all requests, at least 8192 vocab entries per chunk
  const long rows = B;
  long best = (2L * 4 * (num_sms > 0 ? num_sms : 1) + rows - 1) / rows;
  const long max_chunks = (V + 8191) / 8192;
  if (best > max_chunks) best = max_chunks;
  if (best < 1) best = 1;
  long len = (V + best - 1) / best;
  len = (len + 7) / 8 * 8;
  sp.race_chunk_len = (int)len;
  sp.race_chunks = (int)((V + len - 1) / len);
  const size_t srows = (size_t)B * (gamma + 1);
  sp.ws_bytes = srows * sp.chunks * 2 * sizeof(float) + (size_t)B * sizeof(SamplePlan) +
                (size_t)B * sp.race_chunks * 4 * sizeof(float) + 8 * 256;  // 7 carvings, 256-aligned
  return sp;
}

cudaError_t launch_verify_sampling(const void* logits, int dtype, float inv_temp, const float* q,
                                   const int32_t* draft, int B, int gamma, int V, uint64_t seed,
                                   int32_t eos, int32_t* emitted, int32_t* num_emitted,
                                   int32_t* accepted, void* ws, const SamplingPlan& sp,
                                   unsigned* status, cudaStream_t stream) {
  const size_t rows = (size_t)B * (gamma + 1);
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto take = [&](size_t bytes) {
    uint8_t* p = base;
    base += (bytes + 255) & ~(size_t)255;
    return p;
  };
  float* part_m = reinterpret_cast<float*>(take(rows * sp.chunks * sizeof(float)));
  float* part_s = reinterpret_cast<float*>(take(rows * sp.chunks * sizeof(float)));
  SamplePlan* plan = reinterpret_cast<SamplePlan*>(take((size_t)B * sizeof(SamplePlan)));
  const size_t rc = (size_t)B * sp.race_chunks;
  float* race_t = reinterpret_cast<float*>(take(rc * sizeof(float)));
  int* race_i = reinterpret_cast<int*>(take(rc * sizeof(int)));
  float* race_tp = reinterpret_cast<float*>(take(rc * sizeof(float)));
  int* race_ip = reinterpret_cast<int*>(take(rc * sizeof(int)));
  const bool bf16 = dtype == DFLASH_DTYPE_BF16;
  cudaError_t e;
  const dim3 g1(sp.chunks, (unsigned)rows);
  const size_t elem = bf16 ? 2 : 4;
  const bool vec_ok = ((uintptr_t)logits % 16 == 0) && ((size_t)V * elem % 16 == 0) &&
                      ((size_t)sp.chunk_len * elem % 16 == 0);
  e = bf16 ? launch_pdl(softmax_stats_kernel<__nv_bfloat16>, g1, dim3(kThreads), 0, stream,
                        (const __nv_bfloat16*)logits, V, sp.chunks, sp.chunk_len, vec_ok, inv_temp,
                        part_m, part_s)
           : launch_pdl(softmax_stats_kernel<float>, g1, dim3(kThreads), 0, stream,
                        (const float*)logits, V, sp.chunks, sp.chunk_len, vec_ok, inv_temp, part_m,
                        part_s);
  if (e != cudaSuccess) return e;
  const int warps = 4;
  const dim3 g2((B + warps - 1) / warps);
  e = bf16 ? launch_pdl(sampling_scan_kernel<__nv_bfloat16>, g2, dim3(warps * 32), 0, stream,
                        (const __nv_bfloat16*)logits, q, part_m, part_s, sp.chunks, draft, B, gamma,
                        V, inv_temp, seed, eos, emitted, num_emitted, accepted, plan, status)
           : launch_pdl(sampling_scan_kernel<float>, g2, dim3(warps * 32), 0, stream,
                        (const float*)logits, q, part_m, part_s, sp.chunks, draft, B, gamma, V,
                        inv_temp, seed, eos, emitted, num_emitted, accepted, plan, status);
  if (e != cudaSuccess) return e;
  const dim3 g3(sp.race_chunks, B);
  // 16-byte vectors: rows of bf16 logits and of fp32 q start 16-byte aligned, as do chunks
  const bool race_vec = bf16 && ((uintptr_t)logits % 16 == 0) && ((uintptr_t)q % 16 == 0) &&
                        (V % 8 == 0) && (sp.race_chunk_len % 8 == 0);
  e = bf16 ? launch_pdl(race_kernel<__nv_bfloat16>, g3, dim3(kThreads), 0, stream,
                        (const __nv_bfloat16*)logits, q, plan, gamma, V, sp.race_chunks,
                        sp.race_chunk_len, race_vec, inv_temp, seed, race_t, race_i, race_tp,
                        race_ip)
           : launch_pdl(race_kernel<float>, g3, dim3(kThreads), 0, stream, (const float*)logits,
                        q, plan, gamma, V, sp.race_chunks, sp.race_chunk_len, false, inv_temp,
                        seed, race_t, race_i, race_tp, race_ip);
  if (e != cudaSuccess) return e;
  e = launch_pdl(race_finish_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, plan, race_t,
                 race_i, race_tp, race_ip, sp.race_chunks, B, gamma, accepted, emitted);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dflash

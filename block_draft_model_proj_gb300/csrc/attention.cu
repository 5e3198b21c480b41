// Anchored block-sparse attention over dual-source K/V, CUDA-core version.
//
// "DFlash Draft Body", How It Works step 3: within a layer each block reads the target
// prefix before its anchor and all positions of the same block; it cannot read another
// block and does not update the target sequence.  "DFlash" (How it works): the target's
// projected K/V are attended alongside the draft tokens' own K/V.  "DFlash: drafting,
// verification, and speed" (One DFlash generation cycle): a predicted block must not read
// target features containing its future answers -- hence the strict prefix c < anchor.
//
// Key set of a valid slot of block (b, k) with anchor a: context positions c < min(a, L)
// with mask[b, c] != 0, then every valid slot of block (b, k).  Query head h reads KV head
// h / (Hq / Hkv).  Excluded keys are dropped by selection, never by adding -inf to a score,
// so whatever lies beyond the anchor cannot leak in even if it is not finite.
//
// One CTA per (block, KV head): its rows are the S slots x (Hq/Hkv) query heads.  Keys are
// streamed in tiles of kKT through shared memory with an fp32 online softmax.  This is the
// fp32 configuration's attention (every product and sum an fp32 FMA, no TF32); the bf16
// configuration uses the tensor-core kernel in attention_tc.cu on the same layouts.
#include "common.cuh"
#include "internal.h"

namespace dflash {

namespace {

constexpr int kKT = 32;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
attention_simt_kernel(const float* __restrict__ q, const float* __restrict__ kb,
                      const float* __restrict__ vbt, int ns_pad, const float* __restrict__ kv_layer,
                      const int32_t* __restrict__ anchors, const uint8_t* __restrict__ valid,
                      const uint8_t* __restrict__ mask, ActOut out, int N, int S, int L, int Hq,
                      int Hkv, int dh) {
  extern __shared__ float smem[];
  const int grp = Hq / Hkv;
  const int R = S * grp;           // rows: r = j * grp + hh
  float* Qs = smem;                // [R][dh]
  float* Os = Qs + R * dh;         // [R][dh]
  float* Ks = Os + R * dh;         // [kKT][dh + 1]
  float* Vs = Ks + kKT * (dh + 1); // [kKT][dh]
  float* Ps = Vs + kKT * dh;       // [R][kKT]
  float* mrow = Ps + R * kKT;      // [R]
  float* lrow = mrow + R;          // [R]
  float* alpha = lrow + R;         // [R]
  int* kok = reinterpret_cast<int*>(alpha + R);  // [kKT]

  const int blk = blockIdx.x;      // b * N + k
  const int g = blockIdx.y;
  const int b = blk / N;
  const int a = anchors[blk];
  const uint8_t* vrow = valid + (long)blk * S;
  const long t0 = (long)blk * S;   // first slot row of this block
  const int Dq = Hq * dh;
  const int k = blk - b * N;
  const long bg = (long)b * Hkv + g;
  const float* qblk = q + ((bg * N + k) * R) * (long)dh;     // rows r = j * grp + hh
  const float* kblk = kb + ((bg * N + k) * S) * (long)dh;    // [S][dh]
  const float* vblk = vbt + bg * dh * (long)ns_pad + (long)k * S;  // [dh][ns_pad] from key 0

  // queries (pre-scaled by 1/sqrt(dh)); invalid slots are zero rows and get zero output
  const float scale = rsqrtf((float)dh);
  for (int e = threadIdx.x; e < R * dh; e += kThreads) {
    const int r = e / dh;
    const int j = r / grp;
    const bool ok = a >= 0 && vrow[j];
    Qs[e] = ok ? qblk[e] * scale : 0.f;
    Os[e] = 0.f;
  }
  for (int r = threadIdx.x; r < R; r += kThreads) { mrow[r] = -INFINITY; lrow[r] = 0.f; }
  __syncthreads();

  const int n_ctx = a < 0 ? 0 : min(a, L);
  const int n_tiles_ctx = (n_ctx + kKT - 1) / kKT;
  const int n_tiles_blk = a < 0 ? 0 : (S + kKT - 1) / kKT;
  const float* Kc = kv_layer + (((long)b * 2 + 0) * Hkv + g) * (long)L * dh;   // [L][dh]
  const float* Vc = kv_layer + (((long)b * 2 + 1) * Hkv + g) * (long)L * dh;   // [dh][L]
  const uint8_t* mrow_b = mask + (long)b * L;

  for (int tile = 0; tile < n_tiles_ctx + n_tiles_blk; ++tile) {
    const bool is_ctx = tile < n_tiles_ctx;
    const int base = is_ctx ? tile * kKT : (tile - n_tiles_ctx) * kKT;
    for (int kk = threadIdx.x; kk < kKT; kk += kThreads) {
      const int key = base + kk;
      int ok;
      if (is_ctx) ok = key < n_ctx && mrow_b[key] != 0;
      else ok = key < S && vrow[key] != 0;
      kok[kk] = ok;
    }
    for (int e = threadIdx.x; e < kKT * dh; e += kThreads) {
      const int kk = e / dh, d = e - kk * dh;
      const int key = base + kk;
      float kvk = 0.f, kvv = 0.f;
      if (is_ctx) {
        if (key < n_ctx) { kvk = Kc[(long)key * dh + d]; kvv = Vc[(long)d * L + key]; }
      } else if (key < S) {
        kvk = kblk[(long)key * dh + d];
        kvv = vblk[(long)d * ns_pad + key];
      }
      Ks[kk * (dh + 1) + d] = kvk;
      Vs[kk * dh + d] = kvv;
    }
    __syncthreads();
    // scores
    for (int e = threadIdx.x; e < R * kKT; e += kThreads) {
      const int r = e / kKT, kk = e - r * kKT;
      float s = 0.f;
      const float* qr = Qs + r * dh;
      const float* kr = Ks + kk * (dh + 1);
      for (int d = 0; d < dh; ++d) s = fmaf(qr[d], kr[d], s);
      Ps[e] = s;
    }
    __syncthreads();
    // online softmax update per row
    for (int r = threadIdx.x; r < R; r += kThreads) {
      float mx = mrow[r];
      for (int kk = 0; kk < kKT; ++kk)
        if (kok[kk]) mx = fmaxf(mx, Ps[r * kKT + kk]);
      float al = 1.f, sum = 0.f;
      if (mx != -INFINITY) {
        al = mrow[r] == -INFINITY ? 0.f : expf(mrow[r] - mx);
        for (int kk = 0; kk < kKT; ++kk) {
          const float p = kok[kk] ? expf(Ps[r * kKT + kk] - mx) : 0.f;
          Ps[r * kKT + kk] = p;
          sum += p;
        }
      } else {
        for (int kk = 0; kk < kKT; ++kk) Ps[r * kKT + kk] = 0.f;
      }
      mrow[r] = mx;
      lrow[r] = lrow[r] * al + sum;
      alpha[r] = al;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < R * dh; e += kThreads) {
      const int r = e / dh, d = e - r * dh;
      float o = Os[e] * alpha[r];
      const float* pr = Ps + r * kKT;
      for (int kk = 0; kk < kKT; ++kk) o = fmaf(pr[kk], Vs[kk * dh + d], o);
      Os[e] = o;
    }
    __syncthreads();
  }
  for (int e = threadIdx.x; e < R * dh; e += kThreads) {
    const int r = e / dh, d = e - r * dh;
    const int j = r / grp, hh = g * grp + (r - j * grp);
    const bool ok = a >= 0 && vrow[j] && lrow[r] > 0.f;
    out.store((t0 + j) * Dq + (long)hh * dh + d, ok ? Os[e] / lrow[r] : 0.f);
  }
}

}  // namespace

size_t attention_simt_smem(int S, int grp, int dh) {
  const int R = S * grp;
  return sizeof(float) * ((size_t)2 * R * dh + (size_t)kKT * (dh + 1) + (size_t)kKT * dh +
                          (size_t)R * kKT + 3 * (size_t)R) + sizeof(int) * kKT;
}

cudaError_t launch_attention_simt(int dtype, const AttnArgs& a, cudaStream_t stream) {
  (void)dtype;
  const size_t smem = attention_simt_smem(a.S, a.Hq / a.Hkv, a.dh);
  dim3 grid(a.B * a.N, a.Hkv);
  cudaError_t e = cudaFuncSetAttribute(attention_simt_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  attention_simt_kernel<<<grid, kThreads, smem, stream>>>(a.q, a.kb, a.vbt, a.ns_pad, a.kv_layer,
                                                          a.anchors, a.valid, a.mask, a.out, a.N,
                                                          a.S, a.L, a.Hq, a.Hkv, a.dh);
  return cudaGetLastError();
}

}  // namespace dflash

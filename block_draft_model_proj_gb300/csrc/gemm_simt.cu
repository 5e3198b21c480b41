// CUDA-core GEMM with fp32 accumulation: C[z] = A[:, Kz] * B[:, Kz]^T.
//
// Used for the fp32 configuration (no TF32: every product and sum is an fp32 FMA), and for
// bf16 shapes the tensor-core kernel does not take (row strides that are not a multiple of
// 16 bytes).  64x64 output tile per CTA, 256 threads with a 4x4 micro-tile each, K staged
// through shared memory 16 at a time.  Optional K-split z = blockIdx.z writes its partial
// sum to its own C slice; the consumer adds the slices in order.
#include "common.cuh"
#include "internal.h"

namespace dflash {

namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <typename T>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const T* __restrict__ A, long lda, const T* __restrict__ B, long ldb,
                 float* __restrict__ C, long ldc, long M, int N, int K, int k_chunk) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const long m0 = (long)blockIdx.y * BM;
  const int n0 = blockIdx.x * BN;
  const int z = blockIdx.z;
  const int kbeg = z * k_chunk;
  const int kend = min(K, kbeg + k_chunk);
  float* Cz = C + (long)z * M * ldc;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = kbeg; k0 < kend; k0 += BK) {
    // 64x16 tile of A and of B: 1024 elements each, 4 per thread
    for (int e = threadIdx.x; e < BM * BK; e += 256) {
      const int r = e / BK, kk = e - r * BK;
      const long gm = m0 + r;
      const int gk = k0 + kk;
      As[kk][r] = (gm < M && gk < kend) ? to_f(A[gm * lda + gk]) : 0.f;
      const int gn = n0 + r;
      Bs[kk][r] = (gn < N && gk < kend) ? to_f(B[(long)gn * ldb + gk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn < N) Cz[gm * ldc + gn] = acc[i][j];
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt(int dtype, const void* A, long lda, const void* Bm, long ldb,
                             float* C, long ldc, long M, int N, int K, int splits,
                             cudaStream_t stream) {
  if (splits < 1) splits = 1;
  int k_chunk = (K + splits - 1) / splits;
  k_chunk = (k_chunk + BK - 1) / BK * BK;
  dim3 grid((N + BN - 1) / BN, (unsigned)((M + BM - 1) / BM), splits);
  if (dtype == DFLASH_DTYPE_BF16) {
    gemm_simt_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        (const __nv_bfloat16*)A, lda, (const __nv_bfloat16*)Bm, ldb, C, ldc, M, N, K, k_chunk);
  } else {
    gemm_simt_kernel<float><<<grid, 256, 0, stream>>>((const float*)A, lda, (const float*)Bm, ldb,
                                                      C, ldc, M, N, K, k_chunk);
  }
  return cudaGetLastError();
}

}  // namespace dflash

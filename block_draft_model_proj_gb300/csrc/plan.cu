// Anchor plan kernel: deterministic anchors, block validity, loss mask and position ids.
//
// "DFlash Draft Body", How It Works step 1: the plan is a function of (input mask, sample
// ids, optimizer step, seed); rows with the same sample id get the same anchors; a sample
// with no valid window contributes nothing.  Steps 2 and 4: a block is one anchor plus
// gamma draft positions; loss_mask excludes the anchor and invalid positions.
//
// Readings implemented here (identical in the fp64 oracle):
//  - candidate anchor a: mask[a] and mask[a+1] valid;
//  - sampling without replacement: the N candidates with the smallest (key, a), key a
//    chained SplitMix64 finaliser over (seed, step, sample id, a), emitted in position order;
//  - the lowest row with a given sample id draws; the others copy its anchor list, while
//    validity comes from each row's own mask.
//
// One CTA per row.  The N smallest keys are found by an 8-pass radix select on the 64-bit
// key (256-bin shared-memory histograms), then the selected positions are compacted in
// increasing position order with a block-wide ballot scan.  All integer: bit-exact.
#include "common.cuh"
#include "internal.h"

namespace dflash {

namespace {

constexpr int kPlanThreads = 512;

__device__ __forceinline__ uint64_t splitmix64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ bool is_cand(const uint8_t* m, int L, int a) {
  return a + 1 < L && m[a] != 0 && m[a + 1] != 0;
}

// Exclusive rank of this thread's flag among the block's flags (thread order), plus total.
__device__ __forceinline__ int block_ballot_scan(bool flag, int* warp_counts, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  __syncthreads();
  if (lane == 0) warp_counts[warp] = __popc(bal);
  __syncthreads();
  int before = 0, sum = 0;
  for (int w = 0; w < kPlanThreads / 32; ++w) {
    const int c = warp_counts[w];
    if (w < warp) before += c;
    sum += c;
  }
  *total = sum;
  return before + in_warp;
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const uint8_t* __restrict__ mask, const int64_t* __restrict__ sids, int B, int L,
            uint64_t step, uint64_t seed, int N, int S, int32_t* __restrict__ anchors,
            uint8_t* __restrict__ block_valid, uint8_t* __restrict__ loss_mask,
            int32_t* __restrict__ position_ids, int32_t* __restrict__ ctx_len) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned hist[256];
  __shared__ int warp_counts[kPlanThreads / 32];
  __shared__ int sh_sel_digit, sh_remaining, sh_cut, sh_equal;
  __shared__ int sh_anchor[1024];  // N <= 1024 (host-checked)

  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t sid = sids[b];
  int leader = b;
  for (int r = 0; r < b; ++r) {
    if (sids[r] == sid) { leader = r; break; }
  }
  const uint8_t* m = mask + (size_t)leader * L;
  const uint64_t prefix_hash =
      splitmix64_mix(splitmix64_mix(splitmix64_mix(seed) ^ step) ^ (uint64_t)sid);

  // number of candidates
  int local = 0;
  for (int a = tid; a < L; a += kPlanThreads) local += is_cand(m, L, a) ? 1 : 0;
  __shared__ int sh_count;
  if (tid == 0) sh_count = 0;
  __syncthreads();
  atomicAdd(&sh_count, local);
  __syncthreads();
  const int n_cand = sh_count;

  // threshold key T and how many candidates with key == T to take
  uint64_t prefix = 0, prefix_mask = 0;
  int remaining = N;          // candidates still to take at the current prefix
  bool take_all = n_cand <= N;
  if (!take_all) {
    for (int pass = 0; pass < 8; ++pass) {
      const int shift = 56 - 8 * pass;
      for (int i = tid; i < 256; i += kPlanThreads) hist[i] = 0u;
      __syncthreads();
      for (int a = tid; a < L; a += kPlanThreads) {
        if (!is_cand(m, L, a)) continue;
        const uint64_t key = splitmix64_mix(prefix_hash ^ (uint64_t)a);
        if ((key & prefix_mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // warp 0 finds the digit d where the running count of smaller digits first reaches
        // `remaining`: lane l owns bins 8l .. 8l+7
        const int lane = tid;
        int mine = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) mine += (int)hist[lane * 8 + q];
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int up = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += up;
        }
        const int excl = incl - mine;
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= remaining);
        const int owner = __ffs(hit) - 1;  // more candidates than anchors: always a hit
        if (lane == owner) {
          int cum = excl, d = lane * 8;
          for (; d < lane * 8 + 7; ++d) {
            if (cum + (int)hist[d] >= remaining) break;
            cum += (int)hist[d];
          }
          sh_sel_digit = d;
          sh_remaining = remaining - cum;
          sh_equal = (int)hist[d];
        }
      }
      __syncthreads();
      prefix |= (uint64_t)sh_sel_digit << shift;
      prefix_mask |= 0xFFull << shift;
      remaining = sh_remaining;
      __syncthreads();
    }
  }
  // Candidates with key < T are all taken.  Among those with key == T (a 64-bit collision,
  // practically never more than one) take the `remaining` lowest positions: find the cut.
  if (!take_all) {
    if (tid == 0 && sh_equal <= remaining) sh_cut = L;  // every key == T is taken
    if (tid == 0 && sh_equal > remaining) {
      int seen = 0, cut = -1;
      for (int a = 0; a < L && seen < remaining; ++a) {
        if (is_cand(m, L, a) && splitmix64_mix(prefix_hash ^ (uint64_t)a) == prefix) {
          ++seen;
          cut = a;
        }
      }
      sh_cut = cut;
    }
    __syncthreads();
  }
  const int cut = take_all ? L : sh_cut;

  // ordered compaction of the chosen positions
  int base = 0;
  for (int a0 = 0; a0 < L; a0 += kPlanThreads) {
    const int a = a0 + tid;
    bool sel = false;
    if (a < L && is_cand(m, L, a)) {
      if (take_all) {
        sel = true;
      } else {
        const uint64_t key = splitmix64_mix(prefix_hash ^ (uint64_t)a);
        sel = key < prefix || (key == prefix && a <= cut);
      }
    }
    int total;
    const int rank = block_ballot_scan(sel, warp_counts, &total);
    if (sel && base + rank < N) sh_anchor[base + rank] = a;
    base += total;
  }
  __syncthreads();
  const int n_sel = base < N ? base : N;

  // outputs, validity from this row's own mask
  const uint8_t* own = mask + (size_t)b * L;
  __shared__ int sh_ctx_len;
  if (tid == 0) sh_ctx_len = 0;
  __syncthreads();
  for (int k = tid; k < N; k += kPlanThreads) {
    anchors[(size_t)b * N + k] = k < n_sel ? sh_anchor[k] : -1;
  }
  for (int e = tid; e < N * S; e += kPlanThreads) {
    const int k = e / S, j = e - k * S;
    const size_t o = (size_t)b * N * S + e;
    if (k >= n_sel) {
      block_valid[o] = 0;
      loss_mask[o] = 0;
      position_ids[o] = -1;
      continue;
    }
    const int a = sh_anchor[k];
    const int p = a + j;
    const bool v = own[a] != 0 && p < L && own[p] != 0;
    block_valid[o] = v ? 1 : 0;
    loss_mask[o] = (v && j >= 1) ? 1 : 0;
    position_ids[o] = p;
    if (v) atomicMax(&sh_ctx_len, a);
  }
  if (ctx_len) {
    __syncthreads();
    if (tid == 0) ctx_len[b] = sh_ctx_len;
  }
}

}  // namespace

cudaError_t launch_plan(const uint8_t* mask, const int64_t* sids, int B, int L, uint64_t step,
                        uint64_t seed, int N, int S, int32_t* anchors, uint8_t* block_valid,
                        uint8_t* loss_mask, int32_t* position_ids, int32_t* ctx_len,
                        cudaStream_t stream) {
  {
    const cudaError_t le = launch_pdl(plan_kernel, dim3(B), dim3(kPlanThreads), 0, stream, mask,
        sids, B, L, step, seed, N, S, anchors, block_valid, loss_mask, position_ids, ctx_len);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace dflash

// Greedy verification without a caller workspace.
//
// dflash_verify_greedy needs a little scratch memory for the per-chunk argmax partials and
// takes it from a caller-provided workspace.  Some callers cannot provide one: code that
// runs inside a host framework which owns every byte of device memory through its own pool
// and forbids side allocations, or a latency-critical serving loop that must never call
// cudaMalloc / cudaFree (they can synchronize the device and stall every stream).  For
// them, dflash_verify_greedy_static uses a fixed scratch array that lives in this
// library's own device memory, so the call allocates nothing at all.
//
// The scratch array below is a file-scope __device__ array: every GPU that loads the
// library holds its 128 KiB until the process exits.  Host code cannot use the array's
// name as a device address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and caches it.
#include <stdio.h>

#include <atomic>

#include "../../include/dflash_testing.h"
#include "common.cuh"
#include "internal.h"

namespace dflash {

namespace {

// 16384 (value, index) partial pairs: 64 KiB of values + 64 KiB of indices.
constexpr size_t kStaticEntries = 16384;
constexpr size_t kStaticBytes = kStaticEntries * (sizeof(float) + sizeof(int));

static __device__ __align__(256) unsigned char g_verify_scratch[kStaticBytes];

constexpr int kMaxDevices = 64;
// Per-device address of the scratch array.  Host threads may make their first call on a
// device at the same time: each looks the address up and stores the same value, through an
// atomic, so the cache itself is free of data races.
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Looks up (once per device, with that device current) where the scratch array lives.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

int num_sms_current() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" {

int dflash_verify_greedy_static(const void* logits, int logits_dtype, const int32_t* draft, int B,
                                int gamma, int V, int32_t eos, int32_t* emitted,
                                int32_t* num_emitted, int32_t* accepted, int32_t* target_choices,
                                void* stream) {
  if (B < 1 || gamma < 0 || V < 1) {
    return set_error(DFLASH_ERR_INVALID_ARG,
                     "need B >= 1, gamma >= 0, V >= 1 (one target choice per draft token plus a "
                     "bonus)");
  }
  const long rows = (long)B * (gamma + 1);
  if (rows > (long)kStaticEntries) {
    return set_error(DFLASH_ERR_INVALID_ARG,
                     "B * (gamma + 1) = %ld exceeds the static scratch limit of %zu rows; use "
                     "dflash_verify_greedy with a workspace", rows, kStaticEntries);
  }
  if (gamma > kMaxVerifyGamma) {
    return set_error(DFLASH_ERR_INVALID_ARG, "gamma (%d) must be <= %d", gamma, kMaxVerifyGamma);
  }
  if (logits_dtype != DFLASH_DTYPE_BF16 && logits_dtype != DFLASH_DTYPE_F32) {
    return set_error(DFLASH_ERR_INVALID_ARG, "logits_dtype must be DFLASH_DTYPE_BF16 or _F32");
  }
  if (!logits || (!draft && gamma > 0) || !emitted || !num_emitted || !accepted) {
    return set_error(DFLASH_ERR_INVALID_ARG, "null pointer argument");
  }
  // the same split of each vocab row as the workspace variant, capped so that all partials
  // fit in the static array (fewer, longer chunks when there are many rows)
  const VerifyPlan vp =
      cap_verify_chunks(plan_verify(B, gamma, V, num_sms_current()), rows, V, (long)kStaticEntries);
  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) {
    return set_error(DFLASH_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
  }
  // every partial the second kernel reads is written by the first one in the same call, so
  // nothing in the array needs clearing
  float* part_v = static_cast<float*>(base);
  int* part_i = reinterpret_cast<int*>(static_cast<unsigned char*>(base) +
                                       kStaticEntries * sizeof(float));
  e = launch_verify(logits, logits_dtype, draft, B, gamma, V, eos, emitted, num_emitted, accepted,
                    target_choices, part_v, part_i, vp, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    return set_error(DFLASH_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  }
  return DFLASH_OK;
}

}  // extern "C"

// ---- testing hook: the chunk plan of both verification entry points, on the host ----
extern "C" int dflash_testing_verify_plan(int B, int gamma, int V, long resident_ctas,
                                          long static_entries, int* chunks, int* chunk_len) {
  if (B < 1 || gamma < 0 || V < 1 || resident_ctas < 1 || !chunks || !chunk_len)
    return set_error(DFLASH_ERR_INVALID_ARG, "bad verify plan query");
  const long rows = (long)B * (gamma + 1);
  VerifyPlan vp = plan_verify_for(rows, V, resident_ctas);
  if (static_entries > 0) {
    if (rows > static_entries)
      return set_error(DFLASH_ERR_INVALID_ARG, "more rows than static entries");
    vp = cap_verify_chunks(vp, rows, V, static_entries);
  }
  *chunks = vp.chunks;
  *chunk_len = vp.chunk_len;
  return DFLASH_OK;
}

// paged_decode_attn_noalloc: the decode step with its scratch memory in a
// fixed device array owned by the library, for callers that cannot allocate
// device memory.
//
// Who needs it: a caller whose device memory is all handed out by someone
// else -- a plug-in inside a host engine that owns every device buffer through
// its own pool and gives the plug-in no allocator, or a process that reserves
// the whole GPU at start-up so that a later cudaMalloc would fail -- and a
// caller on a latency-critical path that cannot afford cudaMalloc's cost or
// its implicit device-wide synchronisation.  Such a caller has its inputs and
// outputs already, but nowhere to put the step's partial results.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes
// (64 MiB).  Every GPU that loads the library holds it until the process
// exits.  In host code the array's name is only a host-side stand-in, never a
// device address, so the first call on each device looks up its real address
// with cudaGetSymbolAddress (with that device current) and caches it; that
// first call should come before any stream capture.  All calls share the one
// array and it keeps the last call's contents: the only part that must start
// at zero (the status word) is cleared by every call, and calls whose work
// overlaps on the GPU race on the array.  No cudaMalloc, cudaFree or other
// allocating routine is called.  kv_check_noalloc_status reads the status
// word (a bad block id or a timed-out wait) that the kernels record there.

#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace pkv {
namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).
kv_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return fail(KV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(KV_ERR_INVALID_ARG, "device %d beyond the %d supported", dev,
                kMaxDevices);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail(KV_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s",
                  cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" kv_status paged_decode_attn_noalloc(
    const void* q, const void* k_pool, const void* v_pool, int64_t num_blocks,
    const int32_t* block_tables, const int32_t* seq_lens,
    const int32_t* prefix_groups, int32_t n_groups, int32_t nb,
    int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t head_dim,
    int32_t block_size, float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* stream) {
  pkv::clear_error();
  if (!info) return pkv::fail(KV_ERR_INVALID_ARG, "null plan info");
  if (info->workspace_bytes < 0 ||
      (size_t)info->workspace_bytes > pkv::kNoAllocScratchBytes)
    return pkv::fail(KV_ERR_INVALID_ARG,
                     "this step needs %lld bytes of scratch; the built-in "
                     "scratch holds at most %zu (64 MiB): use "
                     "paged_decode_attn with a caller workspace",
                     (long long)info->workspace_bytes,
                     pkv::kNoAllocScratchBytes);
  void* scratch = nullptr;
  if (kv_status s = pkv::scratch_address(&scratch)) return s;
  return paged_decode_attn(q, k_pool, v_pool, num_blocks, block_tables,
                           seq_lens, prefix_groups, n_groups, nb, max_blocks,
                           Hq, Hkv, head_dim, block_size, scale, out, plan,
                           info, scratch, pkv::kNoAllocScratchBytes, stream);
}

extern "C" kv_status kv_check_noalloc_status(void* stream, int32_t* out_code,
                                             int32_t* out_detail) {
  pkv::clear_error();
  if (!out_code) return pkv::fail(KV_ERR_INVALID_ARG, "null out_code");
  void* scratch = nullptr;
  if (kv_status s = pkv::scratch_address(&scratch)) return s;
  return kv_check_device_status(scratch, stream, out_code, out_detail);
}

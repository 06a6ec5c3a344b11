// Data movement behind kv_append and kv_fork_branches.
//
// Pool layout: [layer][block][kv_head][16 slots][head_dim] bf16, so one
// (block, kv_head) is a contiguous 16 x d tile (4 KB at d = 128) and one
// token's row of one head is d contiguous values.  Both kernels move 16-byte
// vectors with grid-stride loops; destinations come from the host allocator
// and are passed by value (no device-side table).

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"

namespace pkv {
namespace {

constexpr int kMaxDst = 2048;  // blocks per launch (8 KB of parameters)

struct ScatterArgs {
  uint4* k_pool;
  uint4* v_pool;
  const uint4* k_new;
  const uint4* v_new;
  int64_t num_blocks;
  int L, Hkv, vec_per_row;  // vec_per_row = d / 8
  int n;                    // tokens in the whole append
  int tok_begin, tok_end;   // tokens [tok_begin, tok_end) of this launch
  int tok0;                 // branch length before the append
  int first_lblock;         // logical block of dst[0]
  int dst[kMaxDst];
};

// One 16-byte vector per thread-iteration: (layer, token, head, vec).
__global__ void append_scatter_kernel(const __grid_constant__ ScatterArgs a) {
  const int64_t toks = a.tok_end - a.tok_begin;
  const int64_t per_layer = toks * a.Hkv * a.vec_per_row;
  const int64_t total = per_layer * a.L;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t layer = i / per_layer;
    int64_t r = i - layer * per_layer;
    const int vec = (int)(r % a.vec_per_row);
    r /= a.vec_per_row;
    const int h = (int)(r % a.Hkv);
    const int tok = a.tok_begin + (int)(r / a.Hkv);  // token within the append
    const int t = a.tok0 + tok;                      // token within the branch
    const int blk = a.dst[t / 16 - a.first_lblock];
    const int slot = t % 16;
    const int64_t src =
        ((layer * a.n + tok) * a.Hkv + h) * (int64_t)a.vec_per_row + vec;
    const int64_t dst =
        (((layer * a.num_blocks + blk) * a.Hkv + h) * 16 + slot) *
            (int64_t)a.vec_per_row + vec;
    a.k_pool[dst] = a.k_new[src];
    a.v_pool[dst] = a.v_new[src];
  }
}

struct CopyArgs {
  uint4* k_pool;
  uint4* v_pool;
  int64_t num_blocks;
  int L;
  int vec_per_block;  // Hkv * 16 * d / 8 (one layer)
  int n;
  int src[kMaxDst / 2];
  int dst[kMaxDst / 2];
};

__global__ void block_copy_kernel(const __grid_constant__ CopyArgs a) {
  const int64_t per_pair = (int64_t)a.L * a.vec_per_block;
  const int64_t total = per_pair * a.n;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int pair = (int)(i / per_pair);
    int64_t r = i - pair * per_pair;
    const int64_t layer = r / a.vec_per_block;
    const int64_t vec = r - layer * a.vec_per_block;
    const int64_t layer_base = layer * a.num_blocks;
    const int64_t s = (layer_base + a.src[pair]) * a.vec_per_block + vec;
    const int64_t d = (layer_base + a.dst[pair]) * a.vec_per_block + vec;
    a.k_pool[d] = a.k_pool[s];
    a.v_pool[d] = a.v_pool[s];
  }
}

int grid_for(int64_t work) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (work + 255) / 256;
  return (int)std::max<int64_t>(1, std::min<int64_t>(blocks, (int64_t)sms * 8));
}

}  // namespace

int launch_append_scatter(void* k_pool, void* v_pool, const void* k_new,
                          const void* v_new, int64_t num_blocks, int L,
                          int Hkv, int d, int B, int n, int tok0,
                          const int32_t* dst_blocks, int n_dst,
                          void* stream) {
  (void)B;
  ScatterArgs a;
  a.k_pool = static_cast<uint4*>(k_pool);
  a.v_pool = static_cast<uint4*>(v_pool);
  a.k_new = static_cast<const uint4*>(k_new);
  a.v_new = static_cast<const uint4*>(v_new);
  a.num_blocks = num_blocks;
  a.L = L;
  a.Hkv = Hkv;
  a.vec_per_row = d / 8;
  a.n = n;
  a.tok0 = tok0;
  const int first_lb = tok0 / 16;
  // Launch over runs of tokens whose destination blocks fit the parameters.
  int tok = 0;
  while (tok < n) {
    const int lb_begin = (tok0 + tok) / 16;
    const int lb_last_allowed = lb_begin + kMaxDst - 1;
    const int tok_end = std::min(n, (lb_last_allowed + 1) * 16 - tok0);
    a.tok_begin = tok;
    a.tok_end = tok_end;
    a.first_lblock = lb_begin;
    const int lb_end = (tok0 + tok_end - 1) / 16;
    for (int lb = lb_begin; lb <= lb_end; ++lb)
      a.dst[lb - lb_begin] = dst_blocks[lb - first_lb];
    const int64_t work = (int64_t)(tok_end - tok) * Hkv * (d / 8) * L;
    append_scatter_kernel<<<grid_for(work), 256, 0, (cudaStream_t)stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    tok = tok_end;
  }
  (void)n_dst;
  return 0;
}

int launch_block_copy(void* k_pool, void* v_pool, int64_t num_blocks, int L,
                      int Hkv, int d, int B, const int32_t* src,
                      const int32_t* dst, int n, void* stream) {
  CopyArgs a;
  a.k_pool = static_cast<uint4*>(k_pool);
  a.v_pool = static_cast<uint4*>(v_pool);
  a.num_blocks = num_blocks;
  a.L = L;
  a.vec_per_block = Hkv * B * d / 8;
  for (int i0 = 0; i0 < n; i0 += kMaxDst / 2) {
    a.n = std::min(n - i0, kMaxDst / 2);
    for (int i = 0; i < a.n; ++i) {
      a.src[i] = src[i0 + i];
      a.dst[i] = dst[i0 + i];
    }
    const int64_t work = (int64_t)a.n * L * a.vec_per_block;
    block_copy_kernel<<<grid_for(work), 256, 0, (cudaStream_t)stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
  return 0;
}

}  // namespace pkv

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
#include <vector>

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

struct XferArgs {
  const uint4* src_k;
  const uint4* src_v;
  uint4* dst_k;
  uint4* dst_v;
  int64_t src_blocks, dst_blocks;
  int L;
  int vec_per_block;  // Hkv * 16 * d / 8 (one layer)
  int n;
  int src[kMaxDst / 2];
  int dst[kMaxDst / 2];
};

__global__ void block_transfer_kernel(const __grid_constant__ XferArgs a) {
  const int64_t per_pair = (int64_t)a.L * a.vec_per_block;
  const int64_t total = per_pair * a.n;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int pair = (int)(i / per_pair);
    const int64_t r = i - pair * per_pair;
    const int64_t layer = r / a.vec_per_block;
    const int64_t vec = r - layer * a.vec_per_block;
    const int64_t s = (layer * a.src_blocks + a.src[pair]) * a.vec_per_block + vec;
    const int64_t d = (layer * a.dst_blocks + a.dst[pair]) * a.vec_per_block + vec;
    a.dst_k[d] = a.src_k[s];
    a.dst_v[d] = a.src_v[s];
  }
}

constexpr int kMaxRuns = 128;
constexpr int kMaxRunDst = 1536;

struct RunDesc {
  int row, n, tok0, first_lb, dst_off;
};

struct BatchArgs {
  uint4* k_pool;
  uint4* v_pool;
  const uint4* k_new;
  const uint4* v_new;
  int64_t num_blocks;
  int L, Hkv, vec_per_row, total;
  int n_runs;
  RunDesc runs[kMaxRuns];
  int dst[kMaxRunDst];
};

// blockIdx.y = run; grid-stride over (layer, token, head, vec) of that run.
__global__ void append_batch_kernel(const __grid_constant__ BatchArgs a) {
  const RunDesc r = a.runs[blockIdx.y];
  const int64_t per_layer = (int64_t)r.n * a.Hkv * a.vec_per_row;
  const int64_t work = per_layer * a.L;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < work;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t layer = i / per_layer;
    int64_t rem = i - layer * per_layer;
    const int vec = (int)(rem % a.vec_per_row);
    rem /= a.vec_per_row;
    const int h = (int)(rem % a.Hkv);
    const int tok = (int)(rem / a.Hkv);
    const int t = r.tok0 + tok;
    const int blk = a.dst[r.dst_off + t / 16 - r.first_lb];
    const int64_t src =
        ((layer * a.total + r.row + tok) * a.Hkv + h) * (int64_t)a.vec_per_row + vec;
    const int64_t dst =
        (((layer * a.num_blocks + blk) * a.Hkv + h) * 16 + t % 16) *
            (int64_t)a.vec_per_row + vec;
    a.k_pool[dst] = a.k_new[src];
    a.v_pool[dst] = a.v_new[src];
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

int launch_append_batch(void* k_pool, void* v_pool, const void* k_new,
                        const void* v_new, int64_t num_blocks, int L, int Hkv,
                        int d, int32_t total, const std::vector<ScatterRun>& runs,
                        void* stream) {
  BatchArgs a;
  a.k_pool = static_cast<uint4*>(k_pool);
  a.v_pool = static_cast<uint4*>(v_pool);
  a.k_new = static_cast<const uint4*>(k_new);
  a.v_new = static_cast<const uint4*>(v_new);
  a.num_blocks = num_blocks;
  a.L = L;
  a.Hkv = Hkv;
  a.vec_per_row = d / 8;
  a.total = total;
  a.n_runs = 0;
  int n_dst = 0;
  int64_t max_work = 0;
  auto flush = [&]() -> int {
    if (a.n_runs == 0) return 0;
    const int gx = std::max(1, std::min(grid_for(max_work), 64));
    append_batch_kernel<<<dim3(gx, a.n_runs), 256, 0, (cudaStream_t)stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    a.n_runs = 0;
    n_dst = 0;
    max_work = 0;
    return (int)e;
  };
  for (const ScatterRun& run : runs) {
    // Split a run into pieces whose blocks fit the parameter space.
    int tok = 0;
    while (tok < run.n) {
      const int t0 = run.tok0 + tok;
      const int lb0 = t0 / 16;
      const int lb_cap = lb0 + kMaxRunDst / 2 - 1;
      const int tok_end = std::min(run.n, (lb_cap + 1) * 16 - run.tok0);
      const int lb1 = (run.tok0 + tok_end - 1) / 16;
      const int nb_piece = lb1 - lb0 + 1;
      if (a.n_runs == kMaxRuns || n_dst + nb_piece > kMaxRunDst) {
        if (int e = flush()) return e;
      }
      RunDesc& r = a.runs[a.n_runs++];
      r.row = run.row + tok;
      r.n = tok_end - tok;
      r.tok0 = t0;
      r.first_lb = lb0;
      r.dst_off = n_dst;
      for (int lb = lb0; lb <= lb1; ++lb)
        a.dst[n_dst++] = run.dst[lb - run.first_lblock];
      max_work = std::max<int64_t>(max_work, (int64_t)r.n * Hkv * (d / 8) * L);
      tok = tok_end;
    }
  }
  return flush();
}

int launch_block_transfer(const void* src_k, const void* src_v,
                          int64_t src_blocks, void* dst_k, void* dst_v,
                          int64_t dst_blocks, int L, int Hkv, int d,
                          const int32_t* src, const int32_t* dst, int n,
                          void* stream) {
  XferArgs a;
  a.src_k = static_cast<const uint4*>(src_k);
  a.src_v = static_cast<const uint4*>(src_v);
  a.dst_k = static_cast<uint4*>(dst_k);
  a.dst_v = static_cast<uint4*>(dst_v);
  a.src_blocks = src_blocks;
  a.dst_blocks = dst_blocks;
  a.L = L;
  a.vec_per_block = Hkv * 16 * d / 8;
  for (int i0 = 0; i0 < n; i0 += kMaxDst / 2) {
    a.n = std::min(n - i0, kMaxDst / 2);
    for (int i = 0; i < a.n; ++i) {
      a.src[i] = src[i0 + i];
      a.dst[i] = dst[i0 + i];
    }
    const int64_t work = (int64_t)a.n * L * a.vec_per_block;
    block_transfer_kernel<<<grid_for(work), 256, 0, (cudaStream_t)stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
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

// Data movement behind kv_append, kv_append_batch, kv_fork_branches,
// kv_spill and kv_restore.
//
// bf16 pool layout: [layer][block][kv_head][16 slots][head_dim], so one
// (block, kv_head) is a contiguous 16 x d tile (4 KB at d = 128) and one
// token's row of one head is d contiguous values.  e4m3 pools keep the same
// tile order with 1-byte codes in the tile layouts of pagedkv.h and a 16-byte
// scale record per tile.  Copies move 16-byte vectors with grid-stride loops;
// destinations come from the host allocator and are passed by value (no
// device-side table).

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <unordered_map>
#include <vector>

#include "device_common.cuh"
#include "e4m3.cuh"

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

// Whole-block moves (copy-on-write, spill, restore): for pair i, every
// layer's (block src[i]) bytes of K, V and the scale records of `from` go to
// block dst[i] of `to`, as 16-byte vectors.
struct MoveArgs {
  const uint4* from_k;
  const uint4* from_v;
  const uint4* from_s;
  uint4* to_k;
  uint4* to_v;
  uint4* to_s;
  int64_t from_blocks, to_blocks;
  int L;
  int kv_vecs;  // 16-byte vectors of one (layer, block) in K (and in V)
  int s_vecs;   // ... in the scale records (0 for bf16 pools)
  int n;
  int src[kMaxDst / 2];
  int dst[kMaxDst / 2];
};

// U independent vectors per thread and iteration (all loaded, then
// stored), so that U copies per thread are in flight over the CPU-GPU link.
template <int U>
__global__ void block_move_kernel(const __grid_constant__ MoveArgs a) {
  const int per_layer = 2 * a.kv_vecs + a.s_vecs;
  const int64_t per_pair = (int64_t)a.L * per_layer;
  const int64_t total = per_pair * a.n;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i0 < total;
       i0 += step * U) {
    uint4 v[U];
    uint4* d[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * step;
      d[u] = nullptr;
      if (i < total) {
        const int pair = (int)(i / per_pair);
        const int64_t r = i - pair * per_pair;
        const int64_t layer = r / per_layer;
        int vec = (int)(r - layer * per_layer);
        const int64_t fb = layer * a.from_blocks + a.src[pair];
        const int64_t tb = layer * a.to_blocks + a.dst[pair];
        if (vec < a.kv_vecs) {
          v[u] = a.from_k[fb * a.kv_vecs + vec];
          d[u] = a.to_k + tb * a.kv_vecs + vec;
        } else if ((vec -= a.kv_vecs) < a.kv_vecs) {
          v[u] = a.from_v[fb * a.kv_vecs + vec];
          d[u] = a.to_v + tb * a.kv_vecs + vec;
        } else {
          vec -= a.kv_vecs;
          v[u] = a.from_s[fb * a.s_vecs + vec];
          d[u] = a.to_s + tb * a.s_vecs + vec;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (d[u]) *d[u] = v[u];
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

int launch_block_move(const PoolBufs& from, const PoolBufs& to, int L,
                      int64_t kv_bytes, int64_t s_bytes, const int32_t* src,
                      const int32_t* dst, int n, void* stream) {
  MoveArgs a;
  a.from_k = static_cast<const uint4*>(from.k);
  a.from_v = static_cast<const uint4*>(from.v);
  a.from_s = static_cast<const uint4*>(from.s);
  a.to_k = static_cast<uint4*>(const_cast<void*>(to.k));
  a.to_v = static_cast<uint4*>(const_cast<void*>(to.v));
  a.to_s = static_cast<uint4*>(const_cast<void*>(to.s));
  a.from_blocks = from.blocks;
  a.to_blocks = to.blocks;
  a.L = L;
  a.kv_vecs = (int)(kv_bytes / 16);
  a.s_vecs = (int)(s_bytes / 16);
  // A light grid: one CTA for every four SMs, four 16-byte vectors in
  // flight per thread.  The moves that cross the CPU-GPU link (spill,
  // restore) need no more to run at the link's speed (restore 205 GB/s of
  // its 211).  A restore is also a prefetch that runs beside decode steps,
  // and the decode steps pay for the copy's footprint on the SMs: beside a
  // restore they took 37% longer with a grid filling every SM's thread
  // slots, 11% with a CTA per SM and 4% with this one.
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  for (int i0 = 0; i0 < n; i0 += kMaxDst / 2) {
    a.n = std::min(n - i0, kMaxDst / 2);
    for (int i = 0; i < a.n; ++i) {
      a.src[i] = src[i0 + i];
      a.dst[i] = dst[i0 + i];
    }
    const int64_t work = (int64_t)a.n * L * (2 * a.kv_vecs + a.s_vecs);
    const int grid = (int)std::min<int64_t>(std::max(sms / 4, 1),
                                            std::max<int64_t>(1, (work + 255) / 256));
    block_move_kernel<4><<<grid, 256, 0, (cudaStream_t)stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
  return 0;
}

// ---- e4m3 pools: quantising writes --------------------------------------------

namespace {

struct E4m3Group {
  int32_t phys, w0, nw, pad;  // block, its writes [w0, w0 + nw)
};
struct E4m3Write {
  int32_t s0, s1, row, pad;   // slots [s0, s1) <- input rows row ..
};
constexpr int kMaxE4m3Groups = 512;
constexpr int kMaxE4m3Writes = 1024;

struct E4m3AppendArgs {
  uint8_t* k8;
  uint8_t* v8;
  float4* scales;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int64_t num_blocks;
  int L, Hkv, d, total;
  E4m3Group groups[kMaxE4m3Groups];
  E4m3Write writes[kMaxE4m3Writes];
};

// grid (groups, layers, kv-heads); warp 0 writes K, warp 1 writes V.  A
// block's writes are applied in order by the same warp.
__global__ void __launch_bounds__(64)
    append_e4m3_kernel(const __grid_constant__ E4m3AppendArgs a) {
  const E4m3Group g = a.groups[blockIdx.x];
  const int layer = blockIdx.y, h = blockIdx.z;
  const bool is_v = threadIdx.x >= 32;
  const int lane = threadIdx.x & 31;
  const int64_t tile = ((int64_t)layer * a.num_blocks + g.phys) * a.Hkv + h;
  uint8_t* codes = (is_v ? a.v8 : a.k8) + tile * 16 * a.d;
  float* scale = reinterpret_cast<float*>(a.scales + tile) + (is_v ? 1 : 0);
  const __nv_bfloat16* src = is_v ? a.v_new : a.k_new;
  for (int w = g.w0; w < g.w0 + g.nw; ++w) {
    const E4m3Write wr = a.writes[w];
    const __nv_bfloat16* rows =
        src + (((int64_t)layer * a.total + wr.row) * a.Hkv + h) * a.d;
    e4m3_tile_write(codes, scale, wr.s0, wr.s1, rows, (int64_t)a.Hkv * a.d,
                    a.d, is_v, lane);
  }
}

struct E4m3StepArgs {
  uint8_t* k8;
  uint8_t* v8;
  float4* scales;
  const __nv_bfloat16* k_step;
  const __nv_bfloat16* v_step;
  const int32_t* tables;
  const int32_t* seq_lens;
  DeviceStatus* status;
  int64_t num_blocks;
  int Hkv, d, max_blocks;
};

// grid (nb, kv-heads): branch b's newest token into its slot.
__global__ void __launch_bounds__(64)
    append_step_e4m3_kernel(const E4m3StepArgs a) {
  const int b = blockIdx.x, h = blockIdx.y;
  const bool is_v = threadIdx.x >= 32;
  const int lane = threadIdx.x & 31;
  const int t = a.seq_lens[b] - 1;
  const int lb = t >> 4;
  const int phys = t >= 0 && lb < a.max_blocks
                       ? a.tables[(int64_t)b * a.max_blocks + lb] : -1;
  if (phys < 0 || (int64_t)phys >= a.num_blocks) {
    if (threadIdx.x == 0) record_status(a.status, KV_ERR_DEVICE, phys);
    return;
  }
  const int64_t tile = (int64_t)phys * a.Hkv + h;
  uint8_t* codes = (is_v ? a.v8 : a.k8) + tile * 16 * a.d;
  float* scale = reinterpret_cast<float*>(a.scales + tile) + (is_v ? 1 : 0);
  const __nv_bfloat16* row =
      (is_v ? a.v_step : a.k_step) + ((int64_t)b * a.Hkv + h) * a.d;
  e4m3_tile_write(codes, scale, t & 15, (t & 15) + 1, row, 0, a.d, is_v, lane);
}

}  // namespace

int launch_append_e4m3(void* k8, void* v8, void* scales, int64_t num_blocks,
                       int L, int Hkv, int d, const void* k_new,
                       const void* v_new, int32_t total,
                       const std::vector<ScatterRun>& runs, void* stream) {
  // Per-block write lists in program order.
  std::vector<int32_t> order;                       // distinct blocks
  std::vector<std::vector<E4m3Write>> per_block;    // parallel to order
  std::unordered_map<int32_t, int32_t> index;
  for (const ScatterRun& run : runs) {
    int tok = 0;
    while (tok < run.n) {
      const int t = run.tok0 + tok;
      const int lb = t / 16;
      const int s0 = t % 16;
      const int cnt = std::min(16 - s0, run.n - tok);
      const int32_t phys = run.dst[lb - run.first_lblock];
      auto it = index.find(phys);
      int32_t gi;
      if (it == index.end()) {
        gi = (int32_t)order.size();
        index.emplace(phys, gi);
        order.push_back(phys);
        per_block.emplace_back();
      } else {
        gi = it->second;
      }
      per_block[gi].push_back({s0, s0 + cnt, run.row + tok, 0});
      tok += cnt;
    }
  }
  E4m3AppendArgs a;
  a.k8 = static_cast<uint8_t*>(k8);
  a.v8 = static_cast<uint8_t*>(v8);
  a.scales = static_cast<float4*>(scales);
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.num_blocks = num_blocks;
  a.L = L;
  a.Hkv = Hkv;
  a.d = d;
  a.total = total;
  size_t gi = 0;
  while (gi < order.size()) {
    int ng = 0, nw = 0;
    while (gi < order.size() && ng < kMaxE4m3Groups) {
      const auto& ws = per_block[gi];
      if ((size_t)nw + ws.size() > (size_t)kMaxE4m3Writes) {
        if (ng > 0) break;
        return (int)cudaErrorInvalidValue;  // one block written > 1024 times
      }
      a.groups[ng] = {order[gi], nw, (int32_t)ws.size(), 0};
      for (const E4m3Write& w : ws) a.writes[nw++] = w;
      ++ng;
      ++gi;
    }
    append_e4m3_kernel<<<dim3(ng, L, Hkv), 64, 0, (cudaStream_t)stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
  return 0;
}

int launch_append_step_e4m3(void* k8, void* v8, void* scales,
                            int64_t num_blocks, int Hkv, int d,
                            const int32_t* tables, const int32_t* seq_lens,
                            int nb, int max_blocks, const void* k_step,
                            const void* v_step, DeviceStatus* status,
                            void* stream) {
  E4m3StepArgs a;
  a.k8 = static_cast<uint8_t*>(k8);
  a.v8 = static_cast<uint8_t*>(v8);
  a.scales = static_cast<float4*>(scales);
  a.k_step = static_cast<const __nv_bfloat16*>(k_step);
  a.v_step = static_cast<const __nv_bfloat16*>(v_step);
  a.tables = tables;
  a.seq_lens = seq_lens;
  a.status = status;
  a.num_blocks = num_blocks;
  a.Hkv = Hkv;
  a.d = d;
  a.max_blocks = max_blocks;
  append_step_e4m3_kernel<<<dim3(nb, Hkv), 64, 0, (cudaStream_t)stream>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace pkv

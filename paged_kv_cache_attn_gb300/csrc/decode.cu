// Decode attention over the paged pool: the split-KV kernel, the log-sum-exp
// merge, and the paged_decode_attn entry point.
//
// What is computed ("The Reasoning Engine Meltdown", §2.1): for each branch b
// and q-head h, softmax(scale * q K^T) V over the branch's cached tokens,
// token t read from block table[b][t / 16], slot t % 16 ("Dismantling the
// Memory Wall", PagedAttention section), kv-head h / (Hq / Hkv).
//
// Split-KV kernel (one CTA = one work item = up to 16 query rows x one
// kv-head x a range of logical blocks):
//  * 4 warps; warp w takes blocks w, w + 4, ... of the range.  Each warp runs
//    its own 2-stage ring, so that three CTAs fit on an SM (measured: three
//    CTAs with two stages beat two CTAs with three stages, since a third
//    item per SM hides more of each item's start-up and epilogue, which
//    dominate short items): per block, lanes 0-3 each
//    issue one 2-D TMA box (16 rows x 64 columns, 128-byte swizzle) of the
//    (block, kv-head) K and V tiles, completing on the stage's mbarrier; the
//    whole warp waits on it.
//  * S = Q K^T with mma.sync m16n8k16: query rows are M (16), the block's
//    16 tokens are N (two n8 tiles), head_dim is K.  The S accumulator layout
//    is the A-operand layout of the next product, so P never leaves
//    registers: O += P V with V read by ldmatrix.trans.
//  * Online softmax in base 2 (scores pre-multiplied by scale * log2(e)),
//    row maxima and sums reduced across the four lanes of a row with
//    shuffles.
//  * The four warps' (m, l, O) are combined through shared memory and written
//    as one unnormalised partial row per query row.
// The merge kernel combines each (branch, q-head)'s partial rows:
// m* = max m_i, l* = sum l_i 2^(m_i - m*), out = sum o_i 2^(m_i - m*) / l*.

#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "device_common.cuh"

namespace pkv {

template <int D, int NS>
struct SplitCfg {
  static constexpr int kWarps = 4;
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = 16 * D * 2;      // one (block, head) tile
  static constexpr int kStageBytes = 2 * kTileBytes;  // K + V
  static constexpr int kRingBytes = kWarps * NS * kStageBytes;
  static constexpr int kMergeBytes = kWarps * 16 * D * 4;
  static constexpr int kSmem =
      (kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes) + 1024;
};

// CTAs 0 .. n_long - 1 take items 0 .. n_long - 1 with all four warps; each
// later CTA takes four of the remaining (short) items, one per warp, and its
// warps write their partial rows themselves.
template <int D, int NS>
__global__ void __launch_bounds__(128, 3)
    splitkv_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const SplitParams p, int n_long, int n_items) {
  using C = SplitCfg<D, NS>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[C::kWarps][NS];
  __shared__ float m_sh[C::kWarps][16];
  __shared__ float l_sh[C::kWarps][16];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  float* base_ptr = reinterpret_cast<float*>(
      smem_raw + (base - smem_u32(smem_raw)));
  const bool per_warp = (int)blockIdx.x >= n_long;  // uniform in the CTA
  const int idx = per_warp ? n_long + 4 * ((int)blockIdx.x - n_long) + warp
                           : (int)blockIdx.x;
  WorkItem it = p.items[idx < n_items ? idx : 0];
  bool have = idx < n_items;
  if (have && !item_ok(it, p, 16)) {
    if (per_warp ? lane == 0 : threadIdx.x == 0)
      record_status(p.status, KV_ERR_DEVICE, -1 - idx);
    have = false;
  }
  if (!per_warp && !have) return;  // the whole CTA, before any barrier

  if (threadIdx.x == 0) {
    for (int w = 0; w < C::kWarps; ++w)
      for (int s = 0; s < NS; ++s) mbar_init(smem_u32(&bars[w][s]), 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  __syncthreads();

  if (!have) return;  // a warp without an item (no CTA barrier follows)
  const int G = p.G;
  const int seq_len = it.masked ? p.seq_lens[it.branch0] : 0x7fffffff;
  const int32_t* table = p.tables + (int64_t)it.branch0 * p.max_blocks;
  const int nblk = it.blk_end - it.blk_begin;
  // This warp's blocks of the item: first, first + stride, ...
  const int first = per_warp ? 0 : warp;
  const int stride = per_warp ? 1 : C::kWarps;
  const int my_n = nblk > first ? (nblk - first + stride - 1) / stride : 0;
  const uint32_t ring = base + warp * NS * C::kStageBytes;
  const uint32_t bar0 = smem_u32(&bars[warp][0]);

  // This warp's block-table entries, 32 at a time in registers (lane i holds
  // the entry of the warp's (32 * window + i)-th block): one coalesced load
  // per 32 blocks instead of a dependent load before every TMA issue.
  int tcache = 0, twin = -1;
  // Issue the loads of this warp's k-th block into stage k % NS.  Returns
  // whether the block id is inside the pool (uniform across the warp).
  auto issue = [&](int k) -> bool {
    if ((k >> 5) != twin) {
      twin = k >> 5;
      const int kk = (twin << 5) + lane;
      tcache = kk < my_n ? table[it.blk_begin + first + stride * kk] : 0;
    }
    const int phys = __shfl_sync(0xffffffffu, tcache, k & 31);
    const bool ok = phys >= 0 && (int64_t)phys < p.num_blocks;
    const int s = k % NS;
    const uint32_t st = ring + s * C::kStageBytes;
    const uint32_t bar = bar0 + s * 8;
    if (ok) {
      // Lane 0 arms the barrier; lanes 0 .. 2*kBoxes-1 then issue one box
      // each in a single instruction (K and V, each kBoxes column halves).
      fence_proxy_async_smem();
      if (lane == 0) mbar_expect_tx(bar, C::kStageBytes);
      __syncwarp();
      if (lane < 2 * C::kBoxes) {
        const int y = (phys * p.Hkv + it.g) * 16;
        const int bx = lane % C::kBoxes;
        const bool is_v = lane >= C::kBoxes;
        tma_load_2d(st + (is_v ? C::kTileBytes : 0) + bx * 2048,
                    is_v ? &tmV : &tmK, bx * 64, y, bar);
      }
    } else if (lane == 0) {
      record_status(p.status, KV_ERR_DEVICE, phys);
      mbar_arrive(bar);
    }
    return ok;
  };

  uint32_t bad = 0;  // bit s: the block in stage s is outside the pool
  const int pre = my_n < NS ? my_n : NS;
  for (int k = 0; k < pre; ++k) {
    if (!issue(k)) bad |= 1u << k;
  }

  // Query fragments (A operand, 16 rows x D): row r -> branch / q-head.
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t qa[D / 16][4];
  {
    const __nv_bfloat16* rowp[2] = {nullptr, nullptr};
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = gq + 8 * hr;
      if (r < it.nrows) {
        const int rr = it.row0 + r;
        const int b = it.branch0 + rr / G;
        const int qh = it.g * G + rr % G;
        rowp[hr] = p.q + ((int64_t)b * p.Hq + qh) * D;
      }
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int hr = i & 1;
        const int col = kk * 16 + 2 * tq + 8 * (i >> 1);
        qa[kk][i] = rowp[hr]
                        ? *reinterpret_cast<const uint32_t*>(rowp[hr] + col)
                        : 0u;
      }
    }
  }

  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[nt][i] = 0.f;

  const int mi = lane >> 3, ri = lane & 7;
  bool timed_out = false;
  int k = 0;
  for (; k < my_n; ++k) {
    const int s = k % NS;
    const uint32_t st = ring + s * C::kStageBytes;
    if (!mbar_wait(bar0 + s * 8, (k / NS) & 1)) {
      timed_out = true;
      break;
    }
    const int j = it.blk_begin + first + stride * k;
    if (!((bad >> s) & 1)) {
      int nv = seq_len - j * 16;
      nv = nv > 16 ? 16 : nv;
      const uint32_t kt = st, vt = st + C::kTileBytes;
      if (p.k_step && it.masked && nv < 17 && j * 16 + nv == seq_len) {
        // Fused append: the branch's newest token (slot nv - 1 of its last
        // block) comes from k_step / v_step; write it into the tile in shared
        // memory (swizzled) and into the pool.  Lanes 0-15: K, 16-31: V.
        const int slot = nv - 1;
        const int c = lane & 15;
        if (c < D / 8) {
          const bool is_v = lane >= 16;
          const int64_t src =
              ((int64_t)it.branch0 * p.Hkv + it.g) * (D / 8) + c;
          const uint4 v = is_v ? p.v_step[src] : p.k_step[src];
          const uint32_t a = (is_v ? vt : kt) + (c >> 3) * 2048 + slot * 128 +
                             (((c & 7) ^ (slot & 7)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a),
                       "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                       : "memory");
          const int phys = table[j];
          const int64_t dst =
              (((int64_t)phys * p.Hkv + it.g) * 16 + slot) * (D / 8) + c;
          (is_v ? p.v_pool : p.k_pool)[dst] = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // S = Q K^T for the block's 16 tokens.
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int token = ((mi >> 1) << 3) + ri;
        const int chunk = kk * 2 + (mi & 1);
        const uint32_t addr = kt + (chunk >> 3) * 2048 + token * 128 +
                              (((chunk & 7) ^ (token & 7)) << 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        mma_16816(sacc[0], qa[kk], b0, b1);
        mma_16816(sacc[1], qa[kk], b2, b3);
      }
      // Scale, mask tokens past the branch's length, online softmax.
      float x[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int tok = nt * 8 + 2 * tq + (i & 1);
          x[nt][i] = tok < nv ? sacc[nt][i] * p.scale_log2 : -INFINITY;
        }
      float pr[2][4];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float mx = fmaxf(fmaxf(x[0][2 * hr], x[0][2 * hr + 1]),
                         fmaxf(x[1][2 * hr], x[1][2 * hr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_r[hr], mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2(m_r[hr] - m_use);
        m_r[hr] = m_new;
        float sum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pv = ex2(x[nt][2 * hr + e] - m_use);
            pr[nt][2 * hr + e] = pv;
            sum += pv;
          }
        l_r[hr] = l_r[hr] * alpha + sum;
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
          o[nt][2 * hr] *= alpha;
          o[nt][2 * hr + 1] *= alpha;
        }
      }
      // Masked slots may hold anything (even NaN): zero their V rows so that
      // 0 * V stays 0 in the product below.
      if (nv < 16) {
        const int chunks = (16 - nv) * C::kBoxes * 8;
        for (int c = lane; c < chunks; c += 32) {
          const int row = nv + c / (C::kBoxes * 8);
          const int rem = c % (C::kBoxes * 8);
          st_shared_zero16(vt + (rem >> 3) * 2048 + row * 128 + (rem & 7) * 16);
        }
        // Order these generic-proxy writes before the TMA refill of the slot.
        fence_proxy_async_smem();
        __syncwarp();
      }
      uint32_t pa[4];
      pa[0] = pack_bf16(pr[0][0], pr[0][1]);
      pa[1] = pack_bf16(pr[0][2], pr[0][3]);
      pa[2] = pack_bf16(pr[1][0], pr[1][1]);
      pa[3] = pack_bf16(pr[1][2], pr[1][3]);
      // O += P V.
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        const int token = ((mi & 1) << 3) + ri;
        const int chunk = np * 2 + (mi >> 1);
        const uint32_t addr = vt + (chunk >> 3) * 2048 + token * 128 +
                              (((chunk & 7) ^ (token & 7)) << 4);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(addr, v0, v1, v2, v3);
        mma_16816(o[2 * np], pa, v0, v1);
        mma_16816(o[2 * np + 1], pa, v2, v3);
      }
    }
    __syncwarp();
    if (k + NS < my_n) {
      if (issue(k + NS))
        bad &= ~(1u << s);
      else
        bad |= 1u << s;
    }
  }
  if (timed_out) {
    if (lane == 0) record_status(p.status, KV_ERR_TIMEOUT, 1);
    // Let every copy still in flight land before the CTA can exit.
    for (int kk = k; kk < my_n && kk < k + NS; ++kk)
      mbar_wait(bar0 + (kk % NS) * 8, (kk / NS) & 1);
  }

  // Row sums across the four lanes of each row.
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 1);
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 2);
  }

  if (per_warp) {
    // The warp's own item: its state is the partial result.  Lane (gq, tq)
    // holds rows gq and gq + 8, columns 8 nt + 2 tq and + 1.
    float* dst = p.o + (int64_t)it.prow_base * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + 2 * tq;
      if (gq < it.nrows)
        *reinterpret_cast<float2*>(dst + gq * D + col) =
            make_float2(o[nt][0], o[nt][1]);
      if (gq + 8 < it.nrows)
        *reinterpret_cast<float2*>(dst + (gq + 8) * D + col) =
            make_float2(o[nt][2], o[nt][3]);
    }
    if (tq == 0) {
      if (gq < it.nrows) p.ml[it.prow_base + gq] = make_float2(m_r[0], l_r[0]);
      if (gq + 8 < it.nrows)
        p.ml[it.prow_base + gq + 8] = make_float2(m_r[1], l_r[1]);
    }
    return;
  }

  // Combine the four warps' partial states through shared memory.
  __syncthreads();  // every warp is done with its ring
  float* Ow = base_ptr + warp * 16 * D;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    const int col = nt * 8 + 2 * tq;
    *reinterpret_cast<float2*>(Ow + gq * D + col) = make_float2(o[nt][0], o[nt][1]);
    *reinterpret_cast<float2*>(Ow + (gq + 8) * D + col) =
        make_float2(o[nt][2], o[nt][3]);
  }
  if (tq == 0) {
    m_sh[warp][gq] = m_r[0];
    m_sh[warp][gq + 8] = m_r[1];
    l_sh[warp][gq] = l_r[0];
    l_sh[warp][gq + 8] = l_r[1];
  }
  __syncthreads();
  {
    const int row = threadIdx.x >> 3;          // 16 rows x 8 threads
    const int c0 = (threadIdx.x & 7) * (D / 8);
    if (row < it.nrows) {
      float mstar = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) mstar = fmaxf(mstar, m_sh[w][row]);
      const float muse = mstar == -INFINITY ? 0.f : mstar;
      float wgt[C::kWarps];
      float lstar = 0.f;
#pragma unroll
      for (int w = 0; w < C::kWarps; ++w) {
        wgt[w] = ex2(m_sh[w][row] - muse);
        lstar += wgt[w] * l_sh[w][row];
      }
      float* dst = p.o + (int64_t)(it.prow_base + row) * D + c0;
#pragma unroll
      for (int c = 0; c < D / 8; c += 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < C::kWarps; ++w) {
          const float4 v = *reinterpret_cast<const float4*>(
              base_ptr + (w * 16 + row) * D + c0 + c);
          acc.x += wgt[w] * v.x;
          acc.y += wgt[w] * v.y;
          acc.z += wgt[w] * v.z;
          acc.w += wgt[w] * v.w;
        }
        *reinterpret_cast<float4*>(dst + c) = acc;
      }
      if ((threadIdx.x & 7) == 0) p.ml[it.prow_base + row] = make_float2(mstar, lstar);
    }
  }
}

struct MergeParams {
  const int32_t* csr_ptr;
  const MergeEntry* csr;
  const float2* ml;
  const float* o;
  __nv_bfloat16* out;
  int nb, Hq, G;
  int64_t partial_rows;
};

// One warp per (branch, q-head).
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const MergeParams p) {
  constexpr int V = D / 32;  // values per lane
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.nb * p.Hq) return;
  const int b = gw / p.Hq, h = gw % p.Hq;
  const int g = h / p.G, r = h % p.G;
  const int e0 = p.csr_ptr[b], e1 = p.csr_ptr[b + 1];
  // One pass with a running maximum: m (base-2 log units), l, acc.
  float m = -INFINITY, lsum = 0.f;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  for (int e = e0; e < e1; ++e) {
    const MergeEntry me = p.csr[e];
    if (r < me.r_lo || r >= me.r_hi) continue;
    const int64_t row = me.base + (int64_t)g * me.stride + (r - me.r_lo);
    if (row < 0 || row >= p.partial_rows) continue;
    const float2 ml = p.ml[row];
    const float* src = p.o + (int64_t)row * D + lane * V;
    float v[V];
    if constexpr (V == 4) {
      const float4 t = *reinterpret_cast<const float4*>(src);
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
      const float2 t = *reinterpret_cast<const float2*>(src);
      v[0] = t.x; v[1] = t.y;
    }
    const float m_new = fmaxf(m, ml.x);
    const float a = m == -INFINITY ? 0.f : ex2(m - m_new);  // first entry: 0
    const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - m_new);
    lsum = lsum * a + w * ml.y;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = acc[i] * a + w * v[i];
    m = m_new;
  }
  const float inv = 1.f / lsum;
  __nv_bfloat16* dst = p.out + ((int64_t)b * p.Hq + h) * D + lane * V;
  if constexpr (V == 4) {
    uint2 pk;
    pk.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0] * inv, acc[1] * inv);
  }
}

// ---- host side ----------------------------------------------------------------

namespace {

constexpr int kStages = 2;

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D view of one layer's pool: rows = block * Hkv * 16 + head * 16 + slot,
// columns = head_dim; boxes of 16 rows x 64 columns, 128-byte swizzle.
kv_status make_pool_map(CUtensorMap* tm, const void* pool, int64_t rows, int d) {
  auto enc = get_encode();
  if (!enc) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(pool), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return KV_OK;
}

// 5-D view of one layer's pool (head_dim 128) in which one box is a whole
// (block, kv-head) tile of 16 rows x 128 columns:
//   x0: column within a 64-column half (2 bytes)   box 64
//   x1: row within a group of 8        (256 bytes) box 8
//   x2: column half                    (128 bytes) box 2
//   x3: group of 8 rows                (2048 bytes) box 2
//   x4: block * Hkv + head             (4096 bytes) box 1
// The strides are not nested (x2 steps inside a row), which a load allows;
// every coordinate inside the dims addresses the tile's own 4 KB.  With
// 128-byte swizzle the box lands as four 1 KB atoms of 8 rows x 64 columns,
// ordered (group 0, half 0), (0, 1), (1, 0), (1, 1): the canonical K-major
// layout with 8-row groups 2048 bytes apart and halves 1024 bytes apart.
kv_status make_pool_map_tiles(CUtensorMap* tm, const void* pool, int64_t nh) {
  auto enc = get_encode();
  if (!enc) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[5] = {64, 8, 2, 2, (cuuint64_t)nh};
  cuuint64_t strides[4] = {256, 128, 2048, 4096};
  cuuint32_t box[5] = {64, 8, 2, 2, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                   const_cast<void*>(pool), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled (tiles) failed (%d)", (int)r);
  return KV_OK;
}

template <int D>
cudaError_t launch_split(const CUtensorMap& tk, const CUtensorMap& tv,
                         const SplitParams& sp, int n_items, int n_warp_items,
                         cudaStream_t stream) {
  if (n_warp_items < 0 || n_warp_items > n_items) return cudaErrorInvalidValue;
  const int n_long = n_items - n_warp_items;
  using C = SplitCfg<D, kStages>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        splitkv_decode_kernel<D, kStages>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  splitkv_decode_kernel<D, kStages>
      <<<n_long + (n_warp_items + 3) / 4, 128, C::kSmem, stream>>>(
          tk, tv, sp, n_long, n_items);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_merge(const MergeParams& mp, cudaStream_t stream) {
  const int warps = mp.nb * mp.Hq;
  lse_merge_kernel<D><<<(warps + 7) / 8, 256, 0, stream>>>(mp);
  return cudaGetLastError();
}

}  // namespace

// Split-KV kernel over an e4m3 pool; defined in decode_e4m3.cu.
cudaError_t launch_split_e4m3(const SplitParams& sp, const void* k8,
                              const void* v8, const void* scales, int n_items,
                              int n_warp_items, int d, cudaStream_t stream);

// Tensor-core tile kernel over an e4m3 pool; defined in decode_tc_e4m3.cu.
cudaError_t launch_tile_e4m3(const SplitParams& sp, const WorkItem* items,
                             int n_items, const void* k8, const void* v8,
                             const void* scales, cudaStream_t stream);

// Tensor-core (tcgen05) kernel for 128-row tiles; defined in decode_tc.cu.
cudaError_t launch_tile_items(const CUtensorMap& tk, const CUtensorMap& tv,
                              const SplitParams& sp, const WorkItem* items,
                              int n_items, int d, cudaStream_t stream);

// Tensor-core kernel for items of up to 256 rows (two M-tiles sharing each
// K/V load); defined in decode_tc_wide.cu.
cudaError_t launch_tile_wide_items(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const SplitParams& sp, const WorkItem* items,
                                   int n_items, int d, cudaStream_t stream);

// Second stream (and fork / join events) per device: the tensor-core tile
// pass runs beside the split-KV pass so that the tile kernel's tensor work
// overlaps the split kernel's HBM streaming on the same SMs.
// A step with both 256-row and 128-row tile items runs the two tile kernels
// on two such streams, side by side.
struct SideStream {
  cudaStream_t stream = nullptr, stream2 = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr, join2 = nullptr;
};

kv_status side_stream(SideStream** out) {
  static std::mutex mu;
  static SideStream per_dev[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64)
    return fail(KV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(mu);
  SideStream& s = per_dev[dev];
  if (!s.stream) {
    // Highest priority: the tile pass has fewer, longer CTAs and sits on the
    // step's critical path, so its pending CTAs are dispatched first.
    int lo = 0, hi = 0;
    cudaDeviceGetStreamPriorityRange(&lo, &hi);
    e = cudaStreamCreateWithPriority(&s.stream, cudaStreamNonBlocking, hi);
    if (e == cudaSuccess)
      e = cudaStreamCreateWithPriority(&s.stream2, cudaStreamNonBlocking, hi);
    if (e == cudaSuccess)
      e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
    if (e == cudaSuccess)
      e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
    if (e == cudaSuccess)
      e = cudaEventCreateWithFlags(&s.join2, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      s.stream = nullptr;
      return fail(KV_ERR_CUDA, "side stream: %s", cudaGetErrorString(e));
    }
  }
  *out = &s;
  return KV_OK;
}

thread_local void* const* g_launch_events = nullptr;
thread_local int g_n_launch_events = 0;

inline void mark(int slot, cudaStream_t st) {
  if (slot < g_n_launch_events && g_launch_events[slot])
    cudaEventRecord(static_cast<cudaEvent_t>(g_launch_events[slot]), st);
}

}  // namespace pkv

using pkv::fail;

extern "C" kv_status kv_set_launch_events(void* const* events,
                                          int32_t n_events) {
  pkv::clear_error();
  pkv::g_launch_events = n_events > 0 ? events : nullptr;
  pkv::g_n_launch_events = events ? n_events : 0;
  return KV_OK;
}

// The newest tokens an e4m3 step quantises into the pool before attending
// (paged_decode_append_attn_e4m3).
struct E4m3Append {
  const void* k_step;
  const void* v_step;
  void* kv_scales;
};

static kv_status decode_impl(
    const void* q, const void* k_step, const void* v_step, const void* k_pool,
    const void* v_pool, const void* kv_scales, int64_t num_blocks,
    const int32_t* block_tables,
    const int32_t* seq_lens, const int32_t* prefix_groups, int32_t n_groups,
    int32_t nb, int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t d,
    int32_t block_size, float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* workspace, size_t ws_bytes,
    void* stream, const E4m3Append* pre = nullptr) {
  (void)prefix_groups;
  if (!q || !k_pool || !v_pool || !block_tables || !seq_lens || !out ||
      !plan || !info || !workspace)
    return fail(KV_ERR_INVALID_ARG, "null argument");
  if (n_groups < 0 || (n_groups > 0 && !prefix_groups))
    return fail(KV_ERR_INVALID_ARG, "bad prefix_groups");
  if (nb < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || max_blocks < 1)
    return fail(KV_ERR_INVALID_ARG, "bad nb/Hq/Hkv/max_blocks");
  if (d != 64 && d != 128) return fail(KV_ERR_INVALID_ARG, "head_dim 64 or 128");
  if (block_size != 16) return fail(KV_ERR_INVALID_ARG, "block_size must be 16");
  if (num_blocks < 1 || num_blocks * Hkv * 16 > (int64_t)INT32_MAX)
    return fail(KV_ERR_INVALID_ARG, "num_blocks out of range");
  if (((uintptr_t)q | (uintptr_t)k_pool | (uintptr_t)v_pool | (uintptr_t)out |
       (uintptr_t)kv_scales) & 15)
    return fail(KV_ERR_INVALID_ARG, "q, pools and out must be 16-byte aligned");
  const bool e4m3 = kv_scales != nullptr;
  if (e4m3 != ((info->flags & KV_PLAN_KV_E4M3) != 0))
    return fail(KV_ERR_INVALID_ARG, e4m3 ? "an e4m3 step needs a plan made "
                                           "with KV_PLAN_KV_E4M3"
                                         : "plan was made for an e4m3 pool");
  if (info->n_tile_items != 0 && d != 128)
    return fail(KV_ERR_INVALID_ARG, "tensor-core tiles need head_dim 128");
  if (info->n_tile_wide_items < 0 ||
      info->n_tile_wide_items > info->n_tile_items ||
      (e4m3 && info->n_tile_wide_items != 0))
    return fail(KV_ERR_INVALID_ARG, "plan info: bad n_tile_wide_items %d",
                info->n_tile_wide_items);
  if ((uintptr_t)workspace & 255)
    return fail(KV_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(KV_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (info->n_merge_rows != nb || info->partial_rows < 0)
    return fail(KV_ERR_INVALID_ARG, "plan info does not match nb");
  if (info->n_row_warp_items < 0 || info->n_row_warp_items > info->n_row_items)
    return fail(KV_ERR_INVALID_ARG, "plan info: bad n_row_warp_items %d",
                info->n_row_warp_items);
  const size_t need = pkv::ws_total(info->partial_rows, d);
  if (ws_bytes < need || (size_t)info->workspace_bytes != need)
    return fail(KV_ERR_INVALID_ARG, "workspace %zu bytes < %zu needed",
                ws_bytes, need);

  cudaStream_t st = (cudaStream_t)stream;
  CUtensorMap tk, tv, tk_tiles, tv_tiles;
  const int64_t rows = num_blocks * Hkv * 16;
  if (!e4m3) {
    if (kv_status s = pkv::make_pool_map(&tk, k_pool, rows, d)) return s;
    if (kv_status s = pkv::make_pool_map(&tv, v_pool, rows, d)) return s;
    if (info->n_tile_items > 0) {
      if (kv_status s = pkv::make_pool_map_tiles(&tk_tiles, k_pool, num_blocks * Hkv))
        return s;
      if (kv_status s = pkv::make_pool_map_tiles(&tv_tiles, v_pool, num_blocks * Hkv))
        return s;
    }
  }

  auto* ws = static_cast<uint8_t*>(workspace);
  pkv::SplitParams sp;
  sp.q = static_cast<const __nv_bfloat16*>(q);
  sp.tables = block_tables;
  sp.seq_lens = seq_lens;
  sp.ml = reinterpret_cast<float2*>(ws + pkv::ws_ml_offset());
  sp.o = reinterpret_cast<float*>(ws + pkv::ws_o_offset(info->partial_rows));
  sp.status = reinterpret_cast<pkv::DeviceStatus*>(ws);
  sp.nb = nb;
  sp.partial_rows = info->partial_rows;
  sp.Hq = Hq;
  sp.Hkv = Hkv;
  sp.G = Hq / Hkv;
  sp.max_blocks = max_blocks;
  sp.num_blocks = num_blocks;
  sp.scale_log2 = scale * 1.4426950408889634f;
  sp.k_step = static_cast<const uint4*>(k_step);
  sp.v_step = static_cast<const uint4*>(v_step);
  sp.k_pool = static_cast<uint4*>(const_cast<void*>(k_pool));
  sp.v_pool = static_cast<uint4*>(const_cast<void*>(v_pool));

  // The plan lives on the device; its layout is fixed by the host header
  // fields mirrored in *info.
  const int off_row = pkv::kPlanHeaderInts;
  const int off_tile = off_row + 8 * info->n_row_items;
  const int off_ptr = off_tile + 8 * info->n_tile_items;
  const int off_ent = off_ptr + nb + 1;

  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(pkv::DeviceStatus), st);
  if (e != cudaSuccess) return fail(KV_ERR_CUDA, "memset: %s", cudaGetErrorString(e));
  if (pre) {
    const int err = pkv::launch_append_step_e4m3(
        const_cast<void*>(k_pool), const_cast<void*>(v_pool), pre->kv_scales,
        num_blocks, Hkv, d, block_tables, seq_lens, nb, max_blocks,
        pre->k_step, pre->v_step, sp.status, st);
    if (err)
      return fail(KV_ERR_CUDA, "e4m3 append launch failed (cuda %d)", err);
  }
  // With both passes present the tile pass forks onto the side stream and
  // joins back before the merge; 256-row and 128-row tile items, when a step
  // has both, run on two side streams.
  pkv::SideStream* side = nullptr;
  const int n_wide = e4m3 ? 0 : info->n_tile_wide_items;
  const int n_narrow = info->n_tile_items - n_wide;
  const bool two_tile = n_wide > 0 && n_narrow > 0;
  const bool fork =
      info->n_tile_items > 0 && (info->n_row_items > 0 || two_tile);
  if (fork) {
    if (kv_status s2 = pkv::side_stream(&side)) return s2;
    e = cudaEventRecord(side->fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->fork, 0);
    if (e == cudaSuccess && two_tile)
      e = cudaStreamWaitEvent(side->stream2, side->fork, 0);
    if (e != cudaSuccess)
      return fail(KV_ERR_CUDA, "fork: %s", cudaGetErrorString(e));
  }
  if (info->n_tile_items > 0) {
    cudaStream_t ts = fork ? side->stream : st;
    pkv::mark(0, ts);
    const auto* titems = reinterpret_cast<const pkv::WorkItem*>(plan + off_tile);
    if (e4m3) {
      e = pkv::launch_tile_e4m3(sp, titems, info->n_tile_items, k_pool, v_pool,
                                kv_scales, ts);
    } else {
      e = cudaSuccess;
      if (n_wide > 0)
        e = pkv::launch_tile_wide_items(tk_tiles, tv_tiles, sp, titems, n_wide,
                                        d, ts);
      if (e == cudaSuccess && n_narrow > 0)
        e = pkv::launch_tile_items(tk_tiles, tv_tiles, sp, titems + n_wide,
                                   n_narrow, d, two_tile ? side->stream2 : ts);
      // The tile pass ends when both of its streams have.
      if (e == cudaSuccess && two_tile) {
        e = cudaEventRecord(side->join2, side->stream2);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ts, side->join2, 0);
      }
    }
    pkv::mark(1, ts);
    if (e != cudaSuccess)
      return fail(KV_ERR_CUDA, "tile kernel: %s", cudaGetErrorString(e));
    if (fork) {
      e = cudaEventRecord(side->join, ts);
      if (e != cudaSuccess)
        return fail(KV_ERR_CUDA, "join: %s", cudaGetErrorString(e));
    }
  }
  if (info->n_row_items > 0) {
    sp.items = reinterpret_cast<const pkv::WorkItem*>(plan + off_row);
    pkv::mark(2, st);
    if (e4m3)
      e = pkv::launch_split_e4m3(sp, k_pool, v_pool, kv_scales,
                                 info->n_row_items, info->n_row_warp_items, d,
                                 st);
    else
      e = d == 128 ? pkv::launch_split<128>(tk, tv, sp, info->n_row_items,
                                            info->n_row_warp_items, st)
                   : pkv::launch_split<64>(tk, tv, sp, info->n_row_items,
                                           info->n_row_warp_items, st);
    pkv::mark(3, st);
    if (e != cudaSuccess)
      return fail(KV_ERR_CUDA, "split-KV kernel: %s", cudaGetErrorString(e));
  }
  if (fork) {
    e = cudaStreamWaitEvent(st, side->join, 0);
    if (e != cudaSuccess)
      return fail(KV_ERR_CUDA, "join: %s", cudaGetErrorString(e));
  }
  pkv::MergeParams mp;
  mp.csr_ptr = plan + off_ptr;
  mp.csr = reinterpret_cast<const pkv::MergeEntry*>(plan + off_ent);
  mp.ml = sp.ml;
  mp.o = sp.o;
  mp.out = static_cast<__nv_bfloat16*>(out);
  mp.nb = nb;
  mp.Hq = Hq;
  mp.G = sp.G;
  mp.partial_rows = info->partial_rows;
  pkv::mark(4, st);
  e = d == 128 ? pkv::launch_merge<128>(mp, st) : pkv::launch_merge<64>(mp, st);
  pkv::mark(5, st);
  if (e != cudaSuccess)
    return fail(KV_ERR_CUDA, "merge kernel: %s", cudaGetErrorString(e));
  return KV_OK;
}

extern "C" kv_status paged_decode_attn(
    const void* q, const void* k_pool, const void* v_pool, int64_t num_blocks,
    const int32_t* block_tables, const int32_t* seq_lens,
    const int32_t* prefix_groups, int32_t n_groups, int32_t nb,
    int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
    float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* workspace, size_t ws_bytes,
    void* stream) {
  pkv::clear_error();
  return decode_impl(q, nullptr, nullptr, k_pool, v_pool, nullptr, num_blocks,
                     block_tables, seq_lens, prefix_groups, n_groups, nb,
                     max_blocks, Hq, Hkv, d, block_size, scale, out, plan, info,
                     workspace, ws_bytes, stream);
}

extern "C" kv_status paged_decode_attn_e4m3(
    const void* q, const void* k_pool, const void* v_pool,
    const void* kv_scales, int64_t num_blocks, const int32_t* block_tables,
    const int32_t* seq_lens, const int32_t* prefix_groups, int32_t n_groups,
    int32_t nb, int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t d,
    int32_t block_size, float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* workspace, size_t ws_bytes,
    void* stream) {
  pkv::clear_error();
  if (!kv_scales) return fail(KV_ERR_INVALID_ARG, "kv_scales required");
  return decode_impl(q, nullptr, nullptr, k_pool, v_pool, kv_scales,
                     num_blocks, block_tables, seq_lens, prefix_groups,
                     n_groups, nb, max_blocks, Hq, Hkv, d, block_size, scale,
                     out, plan, info, workspace, ws_bytes, stream);
}

extern "C" kv_status paged_decode_append_attn_e4m3(
    const void* q, const void* k_step, const void* v_step, const void* k_pool,
    const void* v_pool, void* kv_scales, int64_t num_blocks,
    const int32_t* block_tables, const int32_t* seq_lens,
    const int32_t* prefix_groups, int32_t n_groups, int32_t nb,
    int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t d,
    int32_t block_size, float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* workspace, size_t ws_bytes,
    void* stream) {
  pkv::clear_error();
  if (!k_step || !v_step || !kv_scales)
    return fail(KV_ERR_INVALID_ARG, "k_step, v_step and kv_scales required");
  if (((uintptr_t)k_step | (uintptr_t)v_step) & 15)
    return fail(KV_ERR_INVALID_ARG, "k_step / v_step must be 16-byte aligned");
  if (nb > 65535 * 64 || Hkv > 65535)
    return fail(KV_ERR_INVALID_ARG, "nb or Hkv too large for the append grid");
  const E4m3Append pre{k_step, v_step, kv_scales};
  return decode_impl(q, nullptr, nullptr, k_pool, v_pool, kv_scales,
                     num_blocks, block_tables, seq_lens, prefix_groups,
                     n_groups, nb, max_blocks, Hq, Hkv, d, block_size, scale,
                     out, plan, info, workspace, ws_bytes, stream, &pre);
}

extern "C" kv_status paged_decode_append_attn(
    const void* q, const void* k_step, const void* v_step, const void* k_pool,
    const void* v_pool, int64_t num_blocks, const int32_t* block_tables,
    const int32_t* seq_lens, const int32_t* prefix_groups, int32_t n_groups,
    int32_t nb, int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t d,
    int32_t block_size, float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* workspace, size_t ws_bytes,
    void* stream) {
  pkv::clear_error();
  if (!k_step || !v_step)
    return fail(KV_ERR_INVALID_ARG, "k_step / v_step required");
  if (((uintptr_t)k_step | (uintptr_t)v_step) & 15)
    return fail(KV_ERR_INVALID_ARG, "k_step / v_step must be 16-byte aligned");
  return decode_impl(q, k_step, v_step, k_pool, v_pool, nullptr, num_blocks,
                     block_tables, seq_lens, prefix_groups, n_groups, nb,
                     max_blocks, Hq, Hkv, d, block_size, scale, out, plan, info,
                     workspace, ws_bytes, stream);
}

namespace pkv {
namespace {
// One thread waits on an mbarrier that nothing completes, with the same
// bounded wait the attention kernels use, then records the timeout.
__global__ void selftest_timeout_kernel(DeviceStatus* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  if (!mbar_wait_for(smem_u32(&bar), 0, limit))
    record_status(status, KV_ERR_TIMEOUT, 99);
}
}  // namespace
}  // namespace pkv

extern "C" kv_status kv_selftest_timeout(void* workspace, int64_t wait_cycles,
                                         void* stream) {
  pkv::clear_error();
  if (!workspace || ((uintptr_t)workspace & 255))
    return fail(KV_ERR_INVALID_ARG, "workspace: non-null, 256-byte aligned");
  if (wait_cycles < 1 || wait_cycles > pkv::kWaitCycles)
    return fail(KV_ERR_INVALID_ARG, "wait_cycles outside [1, 2^31]");
  pkv::selftest_timeout_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(
      static_cast<pkv::DeviceStatus*>(workspace), wait_cycles);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return fail(KV_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return KV_OK;
}

extern "C" kv_status kv_check_device_status(void* workspace, void* stream,
                                            int32_t* out_code,
                                            int32_t* out_detail) {
  pkv::clear_error();
  if (!workspace || !out_code) return fail(KV_ERR_INVALID_ARG, "null argument");
  pkv::DeviceStatus h{};
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof h,
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof h, st);
  if (e != cudaSuccess)
    return fail(KV_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  *out_code = (int32_t)h.code;
  if (out_detail) *out_detail = h.detail;
  return KV_OK;
}

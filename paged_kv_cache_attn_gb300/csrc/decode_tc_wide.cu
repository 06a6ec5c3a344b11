// Shared-prefix tile kernel for segments of more than 128 query rows: one CTA
// computes two 128-row M-tiles (up to 256 rows) from every K/V tile it loads.
//
// A segment's blocks are read once per item for all of its rows -- the
// cross-branch re-read that paging removes ("Dismantling the Memory Wall",
// copy-on-write section; RKSC summary §1.1 on cross-branch KV waste).  With
// 128-row items a 256-row segment is loaded twice; here it is loaded once,
// and each byte an SM takes in serves twice the rows.
//
// TMEM (512 columns): S of M-tile 0 in 0..127, S of M-tile 1 in 128..255
// (each P written as bf16 pairs over the first 64 columns of its own S), O of
// M-tile 0 in 256..383, O of M-tile 1 in 384..511.  Q has no room there: both
// M-tiles' Q sit in shared memory in the canonical K-major 128-byte-swizzle
// layout (the layout a K tile lands in) and feed QK as a shared-memory A
// operand.
//
// Per 128-token KV tile j (8 blocks of 16), the MMA thread issues, for each
// M-tile m in turn, PV_m(j - 1) (once the rows of m have written P(j - 1))
// and then QK_m(j).  The MMAs of one thread run in issue order and a commit
// tracks all of the thread's earlier MMAs, so when S_m(j) is reported full,
// PV_m(j - 1) -- which read P from the same columns and wrote O_m -- is done:
// the rows may overwrite S_m with P(j) and rescale O_m without another wait.
// The softmax of one M-tile overlaps the other M-tile's MMAs.
//
//   warps 0-7  (rows):  warp w owns row 32 (w % 4) + lane of M-tile w / 4
//                       (TMEM lane = row): maximum, P = 2^(s - m) in bf16,
//                       base-2 online softmax with a lazy maximum (O and l
//                       rescaled only when the row maximum grows by more
//                       than 8) -> p_full[m]
//   warp 8     (MMA):   QK (M=128, N=128, K=128; A = Q from shared memory)
//                       and PV (M=128, N=128, K=128; A = P from TMEM, V an
//                       MN-major shared-memory operand)
//   warps 9-10 (TMA):   K (warp 9) and V (warp 10), one box per (block,
//                       kv-head) tile, eight boxes per instruction; K ring
//                       of 3 stages, V ring of 2 (shared memory: 64 KB of Q
//                       + 96 KB + 64 KB)
// At the end the rows read O from TMEM and write unnormalised partials
// (o, m, l), merged with the other passes by log-sum-exp.  Tokens of a tile
// past the item's range come from TMA loads at an out-of-range row (zero
// fill) and are masked out of the softmax.

#include "device_common.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace tcw {

using tc::fence_after_sync;
using tc::fence_before_sync;
using tc::idesc;
using tc::rescale_o_row;
using tc::sdesc;
using tc::softmax_tile;
using tc::store_o_row;
using tc::tma_load_5d;
using tc::tmem_wait_st;
using tc::umma_commit;
using tc::umma_ss;
using tc::umma_ts;

constexpr int kT = 128;                  // tokens per KV tile
constexpr int kTB = kT / 16;             // blocks per KV tile
constexpr int kNSK = 3;                  // K ring stages
constexpr int kNSV = 2;                  // V ring stages
constexpr int kBlk = 16 * 128 * 2;       // one (block, kv-head) tile: a box
constexpr int kKV = kT * 128 * 2;        // K (or V) tile, head_dim 128
constexpr int kQ = 128 * 128 * 2;        // Q of one M-tile
constexpr int kSmem = 2 * kQ + (kNSK + kNSV) * kKV + 1024;
constexpr int kRowWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kThreads = 11 * 32;        // warps 0-7 rows, 8 MMA, 9-10 TMA
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kRescale = 8.f;          // lazy-max threshold (log2 units)
constexpr int kTblWin = 64;              // block-table entries staged at once
constexpr int kMaxRows = 256;

// Named barrier 1: the eight row warps and the MMA warp (Q is in shared
// memory).
__device__ __forceinline__ void q_ready_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"((kRowWarps + 1) * 32) : "memory");
}

struct Bars {
  uint64_t k_full[kNSK], k_empty[kNSK], v_full[kNSV], v_empty[kNSV], s_full[2],
      p_full[2], o_ready, drain;
};

__global__ void __launch_bounds__(kThreads, 1)
    tile_wide_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV,
                     const SplitParams p, const WorkItem* items, int oob_tile) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int tbl_sh[2][kTblWin];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;                        // Q, M-tile 0 then 1
  const uint32_t sK = sQ + 2 * kQ;                 // K ring
  const uint32_t sV = sK + kNSK * kKV;             // V ring
  WorkItem it = items[blockIdx.x];
  // A malformed item is recorded and runs with no rows and no tiles.
  if (!item_ok(it, p, kMaxRows)) {
    if (threadIdx.x == 0)
      record_status(p.status, KV_ERR_DEVICE, -1 - (int)blockIdx.x);
    it.nrows = 0;
    it.blk_begin = it.blk_end = 0;
    it.branch0 = 0;
  }
  const int nblk = it.blk_end - it.blk_begin;
  const int ntile = (nblk + kTB - 1) / kTB;
  const int n_m = it.nrows > 128 ? 2 : 1;  // M-tiles with rows
  const int32_t* table = p.tables + (int64_t)it.branch0 * p.max_blocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNSK; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);   // the K producer warp
      mbar_init(smem_u32(&bars.k_empty[s]), 1);  // the MMA issuer's commit
    }
    for (int s = 0; s < kNSV; ++s) {
      mbar_init(smem_u32(&bars.v_full[s]), 1);   // the V producer warp
      mbar_init(smem_u32(&bars.v_empty[s]), 1);
    }
    for (int m = 0; m < 2; ++m) {
      mbar_init(smem_u32(&bars.s_full[m]), 1);
      mbar_init(smem_u32(&bars.p_full[m]), 4);   // the M-tile's four row warps
    }
    mbar_init(smem_u32(&bars.o_ready), 1);
    mbar_init(smem_u32(&bars.drain), 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::
            "r"(smem_u32(&tmem_base_sh)),
        "r"(kTmemCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                     : "memory");
  }
  if (warp == kMmaWarp + 1 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  if (warp < kRowWarps) {
    // Q of this thread's row into shared memory, in the layout a K tile
    // lands in: 8-row group g at 2048 g, column half h at + 1024 h, row i of
    // the group at + 128 i, 16-byte chunk c of the half-row at + 16 (c ^ i).
    const int m = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint4* src = nullptr;
    if (m * 128 + r < it.nrows) {
      const int rr = it.row0 + m * 128 + r;
      const int b = it.branch0 + rr / p.G;
      const int qh = it.g * p.G + rr % p.G;
      src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + qh) * 128);
    }
    const uint32_t qrow = sQ + m * kQ + (r >> 3) * 2048 + (r & 7) * 128;
    // A half-row's eight loads are all issued before its stores (a volatile
    // shared store would otherwise order each load after the one before).
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        v[c] = src ? src[h * 8 + c] : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < 8; ++c)
        tc::st_shared_v4(qrow + h * 1024 + ((c ^ (r & 7)) << 4), v[c].x,
                         v[c].y, v[c].z, v[c].w);
    }
    // Generic-proxy writes, read by the tensor cores (async proxy).
    fence_proxy_async_smem();
  }
  // Q must be in shared memory before the first QK product is issued; the
  // producer warps do not wait for it and start loading K and V at once.
  if (warp <= kMmaWarp) {
    q_ready_barrier();
    fence_after_sync();
  }

  if (warp > kMmaWarp) {
    // ---- TMA producers: warp 9 = K, warp 10 = V, the eight blocks of a tile
    // from lanes 0-7 in one instruction.  A K stage frees once both M-tiles'
    // QK products are done, a V stage once both PV products are.
    const int pw = warp - (kMmaWarp + 1);
    const bool is_v = pw == 1;
    const int ns = is_v ? kNSV : kNSK;
    const CUtensorMap* tm = is_v ? &tmV : &tmK;
    uint64_t* full = is_v ? bars.v_full : bars.k_full;
    uint64_t* empty = is_v ? bars.v_empty : bars.k_empty;
    const uint32_t ring = is_v ? sV : sK;
    int* tbl = tbl_sh[pw];
    int issued = 0, win = -1;
    bool ok = true;
    for (int j = 0; j < ntile && ok; ++j) {
      if (win < 0 || j * kTB + kTB > win + kTblWin) {
        __syncwarp();
        win = j * kTB;
        for (int i = lane; i < kTblWin; i += 32) {
          const int jb = it.blk_begin + win + i;
          tbl[i] = jb < it.blk_end ? table[jb] : -1;
        }
        __syncwarp();
      }
      const int s = j % ns;
      if (lane == 0) {
        if (*(volatile int*)&abort_sh ||
            (j >= ns && !mbar_wait(smem_u32(&empty[s]), ((j / ns) - 1) & 1)))
          ok = false;
        else
          mbar_expect_tx(smem_u32(&full[s]), kKV);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane < kTB) {
        const int bi = lane;
        const int rel = j * kTB + bi;
        int y = oob_tile;  // zero fill past the range
        if (it.blk_begin + rel < it.blk_end) {
          const int phys = tbl[rel - win];
          if (phys >= 0 && (int64_t)phys < p.num_blocks)
            y = phys * p.Hkv + it.g;
          else if (pw == 0)
            record_status(p.status, KV_ERR_DEVICE, phys);
        }
        tma_load_5d(ring + s * kKV + bi * kBlk, tm, y, smem_u32(&full[s]));
      }
      __syncwarp();
      issued = j + 1;
    }
    if (lane == 0) {
      if (!ok && !*(volatile int*)&abort_sh) {
        record_status(p.status, KV_ERR_TIMEOUT, 20);
        atomicExch(&abort_sh, 1);
      }
      // Let every load this warp issued land before the CTA can exit.
      for (int j = issued > ns ? issued - ns : 0; j < issued; ++j)
        mbar_wait(smem_u32(&full[j % ns]), (j / ns) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer ------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc(128, kT, false);
      constexpr uint32_t id_pv = idesc(128, 128, true);
      bool ok = true;
      // O_m += P_m(jp) V(jp); the V stage is waited for by the first M-tile.
      auto pv = [&](int m, int jp) {
        const int s = jp % kNSV;
        if (!mbar_wait(smem_u32(&bars.p_full[m]), jp & 1)) return false;
        if (m == 0 &&
            !mbar_wait(smem_u32(&bars.v_full[s]), (jp / kNSV) & 1))
          return false;
        fence_after_sync();
        const uint32_t vst = sV + s * kKV;
#pragma unroll
        for (int kt = 0; kt < kT / 16; ++kt) {
          const uint64_t bd = sdesc(vst + kt * kBlk, 1024, 2048);
          umma_ts(tmem + kColO + m * 128, tmem + m * 128 + kt * 8, bd, id_pv,
                  (jp > 0 || kt > 0) ? 1u : 0u);
        }
        return true;
      };
      // S_m = Q_m K(j)^T.
      auto qk = [&](int m, int j) {
        const uint32_t kst = sK + (j % kNSK) * kKV;
        const uint32_t qst = sQ + m * kQ;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 32;
          umma_ss(tmem + m * 128, sdesc(qst + off, 16, 2048),
                  sdesc(kst + off, 16, 2048), id_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars.s_full[m]));
      };
      for (int j = 0; j < ntile && ok; ++j) {
        if (!mbar_wait(smem_u32(&bars.k_full[j % kNSK]), (j / kNSK) & 1)) {
          ok = false;
          break;
        }
        fence_after_sync();
        for (int m = 0; m < n_m; ++m) {
          if (j > 0) {
            if (!pv(m, j - 1)) {
              ok = false;
              break;
            }
            if (m == n_m - 1) umma_commit(smem_u32(&bars.v_empty[(j - 1) % kNSV]));
          }
          qk(m, j);
        }
        if (!ok) break;
        umma_commit(smem_u32(&bars.k_empty[j % kNSK]));
      }
      for (int m = 0; m < n_m && ok && ntile > 0; ++m) ok = pv(m, ntile - 1);
      if (!ok) {
        record_status(p.status, KV_ERR_TIMEOUT, 21);
        atomicExch(&abort_sh, 1);
      }
      umma_commit(smem_u32(&bars.o_ready));
      // Drain: every MMA this thread issued has finished once this lands.
      umma_commit(smem_u32(&bars.drain));
      mbar_wait(smem_u32(&bars.drain), 0);
    }
  } else {
    // ---- softmax rows (warps 0-7; thread <-> TMEM lane of its M-tile) ------
    const int m = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t srow = lane_base + m * 128;
    const uint32_t orow = lane_base + kColO + m * 128;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntile && m < n_m; ++j) {
      // Warp-uniform: the TMEM accesses below are warp-collective.
      if (!__all_sync(0xffffffffu,
                      mbar_wait(smem_u32(&bars.s_full[m]), j & 1))) {
        ok = false;
        break;
      }
      fence_after_sync();
      const int valid = min(kT, (it.blk_end - (it.blk_begin + j * kTB)) * 16);
      float alpha;
      const bool need =
          softmax_tile(srow, valid, p.scale_log2, kRescale, m_used, l, alpha);
      // O_m holds PV up to tile j - 1, all of it done (see the header).
      if (__any_sync(0xffffffffu, need) && j > 0) rescale_o_row(orow, alpha);
      tmem_wait_st();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.p_full[m]));
    }
    if (!ok) {
      if (lane == 0) record_status(p.status, KV_ERR_TIMEOUT, 22);
      atomicExch(&abort_sh, 1);
    }
    // Epilogue: O row from TMEM -> unnormalised partial row.
    const bool done = mbar_wait(smem_u32(&bars.o_ready), 0);
    fence_after_sync();
    // tcgen05.ld is warp-collective: decide once per warp.
    const int row = m * 128 + r;
    if (m < n_m &&
        __all_sync(0xffffffffu, done && ok && !*(volatile int*)&abort_sh)) {
      store_o_row(orow, p.o + (int64_t)(it.prow_base + row) * 128,
                  row < it.nrows);
      if (row < it.nrows) p.ml[it.prow_base + row] = make_float2(m_used, l);
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kMmaWarp) {
    asm volatile(
        "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
        "r"(kTmemCols)
        : "memory");
  }
}

}  // namespace tcw

cudaError_t launch_tile_wide_items(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const SplitParams& sp,
                                   const WorkItem* items, int n_items, int d,
                                   cudaStream_t stream) {
  if (d != 128) return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        tcw::tile_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        tcw::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // A (block, head) index past the end of the pool: TMA fills with zeros.
  if ((int64_t)sp.num_blocks * sp.Hkv > INT32_MAX - 1) return cudaErrorInvalidValue;
  const int oob_tile = (int)((int64_t)sp.num_blocks * sp.Hkv);
  tcw::tile_wide_kernel<<<n_items, tcw::kThreads, tcw::kSmem, stream>>>(
      tk, tv, sp, items, oob_tile);
  return cudaGetLastError();
}

}  // namespace pkv

// Shared-prefix tile kernel on the 5th-generation tensor cores (tcgen05).
//
// One CTA = one tile item: 128 query rows of a shared-prefix segment (the
// branches x GQA heads that share the segment's blocks, stacked as M) x one
// kv-head x a range of the segment's logical blocks.  Every block of the
// range is read from HBM once for all 128 rows -- the cross-branch re-read
// that paging removes ("Dismantling the Memory Wall", copy-on-write section;
// RKSC summary §1.1 on cross-branch KV waste) -- and the contraction is dense
// enough (up to 128 flops per KV byte) to belong on the tensor cores.
//
// Pipeline per 128-token KV tile j (8 blocks of 16):
//   warps 5-8 (TMA):   K and V, each a box per (block, kv-head) tile (16
//                      rows x 128 cols as four 1 KB atoms of 8 rows x 64
//                      cols, 128-byte swizzle), into stage j % kNS ->
//                      k_full / v_full
//   warp 4  (MMA):     S[j%2] = Q K^T  (M=128, N=128, K=128; Q and S in
//                      TMEM) -> s_full, k_empty; then O += P(j-1) V(j-1)
//                      (M=128, N=128, K=128; P in TMEM, V as an MN-major
//                      shared-memory operand) -> v_empty, pv_done
//   warps 0-3 (rows):  thread r owns row r: two passes over its S row in
//                      TMEM (maximum, then P = 2^(s - m) as bf16 pairs over
//                      the first 64 columns of the same S buffer), base-2
//                      online softmax with a lazy maximum (O and l are
//                      rescaled only when the row maximum grows by more than
//                      8, so p <= 256) -> p_full.  Only a rescale of O waits
//                      for PV(j-1); otherwise the softmax of tile j overlaps
//                      it.  The MMAs of one thread run in issue order, so
//                      QK(j+2), which overwrites S[j%2], follows PV(j).
// An MMA of M=128, K=16 costs about the same ~95 cycles for N=64 and N=128
// on this part, so 128-token tiles halve the QK cost per token.
// At the end the rows read O from TMEM and write unnormalised partials
// (o, m, l), merged with the other passes by log-sum-exp.
//
// Tokens of a tile past the item's range come from TMA loads at an
// out-of-range row (zero fill) and are masked out of the softmax.

#include "device_common.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace tc {

constexpr int kT = 128;                  // tokens per KV tile
constexpr int kTB = kT / 16;             // blocks per KV tile
constexpr int kNS = 3;                   // stages of each of the K and V rings
constexpr int kBlk = 16 * 128 * 2;       // one (block, kv-head) tile: a box
constexpr int kBox = kT * 128;           // bytes a producer warp loads a tile
constexpr int kKV = 2 * kBox;            // K (or V) tile, head_dim 128
constexpr int kSmem = 2 * kNS * kKV + 1024;
constexpr int kThreads = 288;            // warps 0-3 rows, 4 MMA, 5-8 TMA
constexpr int kMmaWarp = 4;
// TMEM columns (fp32 unless noted): S[0] 0..127, S[1] 128..255 (P of a tile
// overwrites the first 64 columns of its S buffer as bf16 pairs), O
// 320..447, Q 448..511 (bf16 pairs).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 320, kColQ = 448;
constexpr float kRescale = 8.f;          // lazy-max threshold (log2 units)
constexpr int kTblWin = 128;             // block-table entries staged at once

// Named barrier 1: the four softmax warps and the MMA warp (Q is in TMEM).
__device__ __forceinline__ void q_ready_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"(5 * 32) : "memory");
}

struct Bars {
  uint64_t k_full[kNS], k_empty[kNS], v_full[kNS], v_empty[kNS], s_full[2],
      p_full[2], pv_done, o_ready, drain;
};

__global__ void __launch_bounds__(kThreads, 1)
    tile_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const SplitParams p, const WorkItem* items,
                       int oob_tile) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int tbl_sh[4][kTblWin];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = base;                        // K ring
  const uint32_t sV = sK + kNS * kKV;              // V ring
  WorkItem it = items[blockIdx.x];
  // A malformed item is recorded and runs with no rows and no tiles.
  if (!item_ok(it, p, 128)) {
    if (threadIdx.x == 0)
      record_status(p.status, KV_ERR_DEVICE, -1 - (int)blockIdx.x);
    it.nrows = 0;
    it.blk_begin = it.blk_end = 0;
    it.branch0 = 0;
  }
  const int nblk = it.blk_end - it.blk_begin;
  const int ntile = (nblk + kTB - 1) / kTB;
  const int32_t* table = p.tables + (int64_t)it.branch0 * p.max_blocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 2);   // two K producer warps
      mbar_init(smem_u32(&bars.k_empty[s]), 1);  // the MMA issuer's commit
      mbar_init(smem_u32(&bars.v_full[s]), 2);   // two V producer warps
      mbar_init(smem_u32(&bars.v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&bars.s_full[b]), 1);
    // P of tile j is reported on p_full[j % 2]: a softmax warp that runs a
    // tile ahead arrives on the other barrier, so it cannot complete the
    // phase PV(j) waits for before the slowest warp's P(j) is written.
    for (int b = 0; b < 2; ++b) mbar_init(smem_u32(&bars.p_full[b]), 4);
    mbar_init(smem_u32(&bars.pv_done), 1);
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
  if (warp == 5 && lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // Q tile into TMEM columns kColQ.. (lane r = row r = (branch, q-head) of
  // the segment; column c holds elements 2c and 2c + 1).
  if (threadIdx.x < 128) {
    const int r = threadIdx.x;
    const uint4* src = nullptr;
    if (r < it.nrows) {
      const int rr = it.row0 + r;
      const int b = it.branch0 + rr / p.G;
      const int qh = it.g * p.G + rr % p.G;
      src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + qh) * 128);
    }
    const uint32_t lane_base = tmem_base_sh + ((uint32_t)(warp * 32) << 16);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t qv[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = src ? src[h * 8 + c] : make_uint4(0, 0, 0, 0);
        qv[4 * c] = v.x;
        qv[4 * c + 1] = v.y;
        qv[4 * c + 2] = v.z;
        qv[4 * c + 3] = v.w;
      }
      tmem_st32(lane_base + kColQ + h * 32, qv);
    }
    tmem_wait_st();
  }
  // Q must be in TMEM before the first QK product is issued; the producer
  // warps do not wait for it and start loading K and V at once.
  if (warp <= kMmaWarp) {
    fence_before_sync();
    q_ready_barrier();
    fence_after_sync();
  }
  const uint32_t tmem = tmem_base_sh;

  if (warp >= 5) {
    // ---- TMA producers: warps 5 / 6 = K blocks 0-3 / 4-7 of a tile, warps
    // 7 / 8 = V.  One box is a whole (block, kv-head) tile of 4 KB; a warp
    // issues its blocks from lanes 0-3 in one instruction.  A K stage frees
    // as soon as its QK product is done, a V stage after its PV product; K
    // and V producers run independently.
    // Block-table entries are staged in shared memory, kTblWin at a time,
    // with coalesced loads.
    const int pw = warp - 5;
    const bool is_v = pw >= 2;
    const int half = pw & 1;
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
      const int s = j % kNS;
      if (lane == 0) {
        if (*(volatile int*)&abort_sh ||
            (j >= kNS && !mbar_wait(smem_u32(&empty[s]), ((j / kNS) - 1) & 1)))
          ok = false;
        else
          mbar_expect_tx(smem_u32(&full[s]), kBox);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane < kTB / 2) {
        const int bi = half * (kTB / 2) + lane;
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
        record_status(p.status, KV_ERR_TIMEOUT, 10);
        atomicExch(&abort_sh, 1);
      }
      // Let every load this warp issued land before the CTA can exit.
      for (int j = issued > kNS ? issued - kNS : 0; j < issued; ++j)
        mbar_wait(smem_u32(&full[j % kNS]), (j / kNS) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer ------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc(128, kT, false);
      constexpr uint32_t id_pv = idesc(128, 128, true);
      bool ok = true;
      auto pv = [&](int jp) {
        const int s = jp % kNS;
        if (!mbar_wait(smem_u32(&bars.p_full[jp & 1]), (jp >> 1) & 1))
          return false;
        if (!mbar_wait(smem_u32(&bars.v_full[s]), (jp / kNS) & 1)) return false;
        fence_after_sync();
        const uint32_t vst = sV + s * kKV;
#pragma unroll
        for (int kt = 0; kt < kT / 16; ++kt) {
          const uint64_t bd = sdesc(vst + kt * kBlk, 1024, 2048);
          umma_ts(tmem + kColO, tmem + (jp & 1) * kT + kt * 8, bd, id_pv,
                  (jp > 0 || kt > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars.v_empty[s]));
        umma_commit(smem_u32(&bars.pv_done));
        return true;
      };
      for (int j = 0; j < ntile && ok; ++j) {
        const int s = j % kNS, b = j & 1;
        if (!mbar_wait(smem_u32(&bars.k_full[s]), (j / kNS) & 1)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t kst = sK + s * kKV;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = sdesc(kst + (kk >> 2) * 1024 + (kk & 3) * 32, 16,
                                    2048);
          umma_ts(tmem + b * kT, tmem + kColQ + kk * 8, bd, id_qk,
                  kk > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars.k_empty[s]));
        umma_commit(smem_u32(&bars.s_full[b]));
        if (j >= 1) ok = pv(j - 1);
      }
      if (ok && ntile > 0) ok = pv(ntile - 1);
      if (!ok) {
        record_status(p.status, KV_ERR_TIMEOUT, 11);
        atomicExch(&abort_sh, 1);
      }
      umma_commit(smem_u32(&bars.o_ready));
      // Drain: every MMA this thread issued has finished once this lands.
      umma_commit(smem_u32(&bars.drain));
      mbar_wait(smem_u32(&bars.drain), 0);
    }
  } else {
    // ---- softmax rows (warps 0-3; thread r <-> TMEM lane r) ----------------
    const int r = threadIdx.x;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < ntile; ++j) {
      const int b = j & 1;
      // Warp-uniform: the TMEM accesses below are warp-collective.
      if (!__all_sync(0xffffffffu,
                      mbar_wait(smem_u32(&bars.s_full[b]), (j >> 1) & 1))) {
        ok = false;
        break;
      }
      fence_after_sync();
      const uint32_t srow = lane_base + b * kT;
      const int valid = min(kT, (it.blk_end - (it.blk_begin + j * kTB)) * 16);
      float alpha;
      const bool need =
          softmax_tile(srow, valid, p.scale_log2, kRescale, m_used, l, alpha);
      if (__any_sync(0xffffffffu, need) && j > 0) {
        // Rescale this row of O (it holds PV up to tile j - 1) once PV(j - 1)
        // is done.  PV(j) cannot have started (it waits for this tile's P),
        // so the barrier has completed j - 1 or j phases and the parity wait
        // is exact.
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&bars.pv_done), (j - 1) & 1))) {
          ok = false;
          break;
        }
        fence_after_sync();
        rescale_o_row(lane_base + kColO, alpha);
      }
      tmem_wait_st();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.p_full[b]));
    }
    if (!ok) {
      if (lane == 0) record_status(p.status, KV_ERR_TIMEOUT, 12);
      atomicExch(&abort_sh, 1);
    }
    // Epilogue: O row from TMEM -> unnormalised partial row.
    const bool done = mbar_wait(smem_u32(&bars.o_ready), 0);
    fence_after_sync();
    // tcgen05.ld is warp-collective: decide once per warp.
    if (__all_sync(0xffffffffu,
                   done && ok && !*(volatile int*)&abort_sh)) {
      store_o_row(lane_base + kColO, p.o + (int64_t)(it.prow_base + r) * 128,
                  r < it.nrows);
      if (r < it.nrows) p.ml[it.prow_base + r] = make_float2(m_used, l);
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

}  // namespace tc

cudaError_t launch_tile_items(const CUtensorMap& tk, const CUtensorMap& tv,
                              const SplitParams& sp, const WorkItem* items,
                              int n_items, int d, cudaStream_t stream) {
  if (d != 128) return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        tc::tile_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        tc::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // A (block, head) index past the end of the pool: TMA fills with zeros.
  if ((int64_t)sp.num_blocks * sp.Hkv > INT32_MAX - 1) return cudaErrorInvalidValue;
  const int oob_tile = (int)((int64_t)sp.num_blocks * sp.Hkv);
  tc::tile_decode_kernel<<<n_items, tc::kThreads, tc::kSmem, stream>>>(
      tk, tv, sp, items, oob_tile);
  return cudaGetLastError();
}

}  // namespace pkv

// Shared-prefix tile kernel for e4m3 pools on the tcgen05 tensor cores.
//
// One CTA = one tile item: up to 128 query rows of a shared-prefix segment x
// one kv-head x a range of the segment's blocks, every block read once for
// all rows ("Dismantling the Memory Wall", copy-on-write section: shared
// prefixes are stored once; RKSC summary §1.1: the cross-branch re-read is
// the waste).  Every e4m3 value is exactly an f16, so the codes are widened
// in shared memory and both products run as kind::f16:
//
//   S = Q K^T  A = Q in TMEM (f16; each row scaled by a power of two so that
//              its largest magnitude lies in [2^14, 2^15), which keeps every
//              bf16 query element exact), B = the K tile in f16.  Two
//              converter warps widen the pool's K rows (128 codes in the
//              canonical 128-byte-swizzle K-major layout) into two 64-column
//              halves of the same layout in f16.
//   O += P V   A = P (f16 pairs in TMEM: the P of S columns 32c .. 32c + 31
//              goes over columns 32c + 16 .. 32c + 31 of the same S buffer),
//              B = V^T in f16, widened by two more
//              converter warps from the transposed V tiles.  Tokens past the
//              range are zeros in both operands.
//   softmax    two threads per row (TMEM lane = row), each over 64 of a
//              tile's 128 columns, the row maximum exchanged through shared
//              memory; base 2, lazy maximum (O, l rescaled only when the row
//              maximum grows by more than 2^8).  The per-block K scale folds into the score factor; the
//              per-block V scale folds into P relative to the largest V scale
//              seen so far (O is rescaled when that grows).  Only a rescale
//              waits for the previous PV; otherwise the softmax of tile j
//              overlaps it.  The MMAs of one thread run in issue order, so
//              QK(j+2), which overwrites S[j%2], follows PV(j).
//
// Warps: 0-7 softmax rows (they also load Q into TMEM), 8 MMA issuer, 9 K
// producer and 10 V producer (8 bulk copies of 2 KB per tile each), 11 scale
// producer (the tile's 16-byte scale records into a 4-stage ring; a bulk copy
// costs ~130 cycles to issue whatever its size, so the records get a warp of
// their own), 12-13 V converters, 14-15 K converters.  Partial rows (o, m, l) go to the workspace and are merged by
// log-sum-exp with the other passes, exactly as for the bf16 tile kernel.

#include <cuda_fp16.h>

#include "device_common.cuh"
#include "e4m3.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace tc8 {

using tc::fence_after_sync;
using tc::fence_before_sync;
using tc::idesc_k0;
using tc::sdesc;
using tc::tmem_ld32;
using tc::tmem_st16;
using tc::tmem_st32;
using tc::tmem_wait_ld;
using tc::tmem_wait_st;
using tc::umma_commit;
using tc::umma_ts;

constexpr int kT = 128;                   // tokens per tile
constexpr int kTB = kT / 16;              // blocks per tile
constexpr int kNSK = 3;                   // stages of the K code ring
constexpr int kNSV = 2;                   // stages of the V code ring
constexpr int kNFK = 2;                   // f16 K buffers (conversion || QK)
constexpr int kNFV = 2;                   // f16 V^T buffers (conversion || PV)
constexpr int kSC = 4;                    // stages of the scale-record ring
constexpr int kTile8 = kT * 128;          // 8 blocks' K (or V) codes: 16 KB
constexpr int kHalfF = 128 * 128;         // an f16 operand half: 128 rows x 128 B
constexpr int kTileF = 2 * kHalfF;        // an f16 K or V^T tile: 32 KB
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kNSK * kTile8;
constexpr int kOffKF = kOffV + kNSV * kTile8;
constexpr int kOffVF = kOffKF + kNFK * kTileF;
constexpr int kOffS = kOffVF + kNFV * kTileF;
constexpr int kSmem = kOffS + kSC * kTB * 16 + 1024;
constexpr int kThreads = 512;
constexpr int kMmaWarp = 8, kKWarp = 9, kVWarp = 10, kScWarp = 11,
              kVCvtWarp = 12, kKCvtWarp = 14;
static_assert(kVWarp == kKWarp + 1 && kScWarp == kKWarp + 2,
              "a producer's role is its warp index minus kKWarp");
// TMEM columns: S[0] 0..127, S[1] 128..255 (fp32; P of a tile overwrites
// half of its S buffer as f16 pairs, see p_col), O 320..447 (fp32), Q
// 448..511 (f16 pairs).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 320, kColQ = 448;
constexpr float kRescale = 8.f;

// TMEM column (within an S buffer) of the P of tokens 16 kt .. 16 kt + 15:
// the P of S columns 32c .. 32c + 31 (tokens of k-steps 2c and 2c + 1) lies in
// columns 32c + 16 .. 32c + 31, which only the thread that read them writes.
__host__ __device__ constexpr uint32_t p_col(int kt) {
  return 32u * (uint32_t)(kt >> 1) + 16u + 8u * (uint32_t)(kt & 1);
}

struct Bars {
  uint64_t k_full[kNSK], k_empty[kNSK], v_full[kNSV], v_empty[kNSV],
      kf_full[kNFK], kf_empty[kNFK], vf_full[kNFV], vf_empty[kNFV],
      sc_full[kSC], sc_empty[kSC],
      s_full[2], p_full, pv_done, o_ready, drain, xch[2];
};

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Named barrier 1: the softmax warps (they write Q) and the MMA warp.
__device__ __forceinline__ void q_ready_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"(9 * 32) : "memory");
}

// Named barrier 2: the softmax warps (the two halves of a Q row).
__device__ __forceinline__ void rows_barrier() {
  asm volatile("bar.sync 2, %0;" ::"r"(8 * 32) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    tile_e4m3_kernel(const SplitParams p, const WorkItem* items,
                     const uint8_t* __restrict__ k8,
                     const uint8_t* __restrict__ v8,
                     const float4* __restrict__ scales) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  // Per row: the two halves' maxima of Q, then of each tile (double-buffered
  // by tile), and the final (m, l) pieces for the epilogue.
  __shared__ float qmax_sh[2][128];
  __shared__ float xmax_sh[2][2][128];
  __shared__ float xl_sh[2][128];
  __shared__ float xm_sh[128];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = base + kOffK, sV = base + kOffV, sKF = base + kOffKF,
                 sVF = base + kOffVF, sS = base + kOffS;
  WorkItem it = items[blockIdx.x];
  if (!item_ok(it, p, 128)) {
    if (threadIdx.x == 0)
      record_status(p.status, KV_ERR_DEVICE, -1 - (int)blockIdx.x);
    it.nrows = 0;
    it.blk_begin = it.blk_end = 0;
    it.branch0 = 0;
    it.g = 0;
  }
  const int nblk = it.blk_end - it.blk_begin;
  const int ntile = (nblk + kTB - 1) / kTB;
  const int32_t* table = p.tables + (int64_t)it.branch0 * p.max_blocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNSK; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.k_empty[s]), 2);    // both K converter warps
    }
    for (int s = 0; s < kNSV; ++s) {
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.v_empty[s]), 2);    // both V converter warps
    }
    for (int s = 0; s < kNFK; ++s) {
      mbar_init(smem_u32(&bars.kf_full[s]), 2);    // both K converter warps
      mbar_init(smem_u32(&bars.kf_empty[s]), 1);   // the MMA's commit
    }
    for (int s = 0; s < kNFV; ++s) {
      mbar_init(smem_u32(&bars.vf_full[s]), 2);    // both V converter warps
      mbar_init(smem_u32(&bars.vf_empty[s]), 1);   // the MMA's commit
    }
    for (int s = 0; s < 2; ++s) mbar_init(smem_u32(&bars.s_full[s]), 1);
    for (int s = 0; s < kSC; ++s) {
      mbar_init(smem_u32(&bars.sc_full[s]), 1);
      mbar_init(smem_u32(&bars.sc_empty[s]), 8);   // every softmax warp
    }
    mbar_init(smem_u32(&bars.p_full), 8);           // every softmax warp
    for (int b = 0; b < 2; ++b)
      mbar_init(smem_u32(&bars.xch[b]), 256);       // every softmax thread
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
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  // Q rows -> TMEM columns kColQ.. as f16 pairs (lane r = row r; column c
  // holds elements 2c and 2c + 1); thread (h, r) of the softmax warps writes
  // elements 64h .. 64h + 63.  Row r is scaled by 2^-sq so that its largest
  // magnitude lies in [2^14, 2^15): f16 then holds every bf16 element of the
  // row exactly down to 2^-31 of the largest (below that, within the f16
  // subnormal spacing 2^-24).
  float fsc = 0.f;  // scale_log2 * 2^sq of this thread's row
  if (warp < 8) {
    const int h = threadIdx.x >> 7, r = threadIdx.x & 127;
    const uint4* src = nullptr;
    if (r < it.nrows) {
      const int rr = it.row0 + r;
      const int b = it.branch0 + rr / p.G;
      const int qh = it.g * p.G + rr % p.G;
      src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + qh) * 128) +
            h * 8;
    }
    uint4 qw[8];
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      qw[c] = src ? src[c] : make_uint4(0, 0, 0, 0);
      const uint32_t w[4] = {qw[c].x, qw[c].y, qw[c].z, qw[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                                 fabsf(__uint_as_float(w[i] & 0xffff0000u))));
    }
    qmax_sh[h][r] = amax;
    rows_barrier();
    amax = fmaxf(qmax_sh[0][r], qmax_sh[1][r]);
    int sq = amax > 0.f ? scale_exponent(amax) - 14 : 0;
    sq = sq < -100 ? -100 : sq;
    const float mul = pow2f(-sq);
    fsc = p.scale_log2 * pow2f(sq);
    uint32_t qv[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t w[4] = {qw[c].x, qw[c].y, qw[c].z, qw[c].w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        qv[4 * c + i] = pack_f16(__uint_as_float(w[i] << 16) * mul,
                                 __uint_as_float(w[i] & 0xffff0000u) * mul);
    }
    tmem_st32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + kColQ + h * 32, qv);
    tmem_wait_st();
  }
  // Q must be in TMEM before the first QK product is issued; the producer
  // and converter warps do not wait for it.
  if (warp <= kMmaWarp) {
    fence_before_sync();
    q_ready_barrier();
    fence_after_sync();
  }

  if (warp >= kKWarp && warp <= kScWarp) {
    // ---- producers: one bulk copy per block of a tile, from lanes 0-7 --
    // the K codes, the V codes, or the (block, kv-head) scale records.
    // Block-table entries come 32 at a time (4 tiles) in registers, the next
    // window prefetched.  A code stage frees once both converter warps of its
    // kind are done, a record stage once every softmax warp has read it.
    const int role = warp - kKWarp;  // 0 K codes, 1 V codes, 2 records
    const int nst = role == 0 ? kNSK : role == 1 ? kNSV : kSC;
    uint64_t* full = role == 0 ? bars.k_full : role == 1 ? bars.v_full
                                                         : bars.sc_full;
    uint64_t* empty = role == 0 ? bars.k_empty : role == 1 ? bars.v_empty
                                                           : bars.sc_empty;
    const uint32_t ring = role == 0 ? sK : role == 1 ? sV : sS;
    const uint32_t stage_bytes = role == 2 ? kTB * 16 : kTile8;
    const uint32_t copy_bytes = role == 2 ? 16 : 2048;
    const uint8_t* pool = role == 0 ? k8 : role == 1
                              ? v8 : reinterpret_cast<const uint8_t*>(scales);
    auto win_load = [&](int w) -> int {
      const int idx = w * 32 + lane;
      return idx < nblk ? table[it.blk_begin + idx] : -1;
    };
    int tcur = 0, tnext = 0, wcur = -1;
    int issued = 0;
    bool ok = true;
    for (int j = 0; j < ntile && ok; ++j) {
      const int w = j >> 2;
      if (w != wcur) {
        tcur = (wcur == w - 1 && wcur >= 0) ? tnext : win_load(w);
        tnext = win_load(w + 1);
        wcur = w;
      }
      const int s = j % nst;
      const int nb_in = min(kTB, nblk - j * kTB);
      if (lane == 0) {
        if (*(volatile int*)&abort_sh ||
            (j >= nst && !mbar_wait(smem_u32(&empty[s]), ((j / nst) - 1) & 1)))
          ok = false;
        else
          mbar_expect_tx(smem_u32(&full[s]), nb_in * copy_bytes);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      int phys = __shfl_sync(0xffffffffu, tcur, ((j & 3) << 3) + (lane & 7));
      if (lane < nb_in) {
        if (phys < 0 || (int64_t)phys >= p.num_blocks) {
          if (role == 0) record_status(p.status, KV_ERR_DEVICE, phys);
          phys = 0;  // any block in the pool: the output is unspecified now
        }
        const int64_t tile = (int64_t)phys * p.Hkv + it.g;
        bulk_load(ring + s * stage_bytes + lane * copy_bytes,
                  pool + tile * copy_bytes, copy_bytes, smem_u32(&full[s]));
      }
      __syncwarp();
      issued = j + 1;
    }
    if (lane == 0) {
      if (!ok && !*(volatile int*)&abort_sh) {
        record_status(p.status, KV_ERR_TIMEOUT, 20);
        atomicExch(&abort_sh, 1);
      }
      // Let every copy this warp issued land before the CTA can exit.
      for (int j = issued > nst ? issued - nst : 0; j < issued; ++j)
        mbar_wait(smem_u32(&full[j % nst]), (j / nst) & 1);
    }
  } else if (warp >= kVCvtWarp && warp < kKCvtWarp) {
    // ---- V converters: raw V^T tile (8 blocks x [128 dims][16 slots]) ->
    // f16 V^T in two 64-token halves, each 128 rows (dims) x 128 bytes,
    // 16-byte chunk c of row d at (c ^ (d % 8)) * 16.  Warp cw takes
    // dimensions 64 cw .. 64 cw + 63.
    const int cw = warp - kVCvtWarp;
    bool ok = true;
    for (int j = 0; j < ntile && ok; ++j) {
      const int s = j % kNSV, f = j % kNFV;
      if (*(volatile int*)&abort_sh ||
          !mbar_wait(smem_u32(&bars.v_full[s]), (j / kNSV) & 1) ||
          (j >= kNFV &&
           !mbar_wait(smem_u32(&bars.vf_empty[f]), ((j / kNFV) - 1) & 1))) {
        ok = false;
        break;
      }
      const int nb_in = min(kTB, nblk - j * kTB);
      const uint32_t raw = sV + s * kTile8;
      const uint32_t dstt = sVF + f * kTileF;
      // All 16 loads first, so that they are in flight together.
      uint4 wv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int dim = cw * 64 + lane + 32 * (i & 1);
        wv[i] = (i >> 1) < nb_in ? lds128(raw + (i >> 1) * 2048 + dim * 16)
                                 : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int dim = cw * 64 + lane + 32 * (i & 1);
        const int blk = i >> 1;
        const uint4 w = wv[i];
        uint32_t h[8];
        e4m3x4_to_f16x2x2(w.x, h[0], h[1]);
        e4m3x4_to_f16x2x2(w.y, h[2], h[3]);
        e4m3x4_to_f16x2x2(w.z, h[4], h[5]);
        e4m3x4_to_f16x2x2(w.w, h[6], h[7]);
        const uint32_t row = dstt + (blk >> 2) * kHalfF + dim * 128;
        const uint32_t c0 = 2 * (blk & 3);
        tc::st_shared_v4(row + (((c0) ^ (dim & 7)) << 4), h[0], h[1], h[2], h[3]);
        tc::st_shared_v4(row + (((c0 + 1) ^ (dim & 7)) << 4), h[4], h[5], h[6],
                         h[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars.vf_full[f]));
        mbar_arrive(smem_u32(&bars.v_empty[s]));
      }
    }
    if (!ok && lane == 0) {
      if (!*(volatile int*)&abort_sh) record_status(p.status, KV_ERR_TIMEOUT, 21);
      atomicExch(&abort_sh, 1);
    }
  } else if (warp >= kKCvtWarp) {
    // ---- K converters: raw K tile (128 token rows of 128 codes, 16-byte
    // chunk c of row t at (c ^ (t % 8)) * 16) -> f16 K in two 64-dimension
    // halves, each 128 rows (tokens) x 128 bytes, 16-byte chunk cc of row t
    // at (cc ^ (t % 8)) * 16.  Warp kw writes half kw: code chunks 4 kw ..
    // 4 kw + 3, each becoming two f16 chunks.  Rows past the range: zeros.
    const int kw = warp - kKCvtWarp;
    bool ok = true;
    for (int j = 0; j < ntile && ok; ++j) {
      const int s = j % kNSK, f = j % kNFK;
      if (*(volatile int*)&abort_sh ||
          !mbar_wait(smem_u32(&bars.k_full[s]), (j / kNSK) & 1) ||
          (j >= kNFK &&
           !mbar_wait(smem_u32(&bars.kf_empty[f]), ((j / kNFK) - 1) & 1))) {
        ok = false;
        break;
      }
      const int rows_in = min(kTB, nblk - j * kTB) * 16;
      const uint32_t raw = sK + s * kTile8;
      const uint32_t dsth = sKF + f * kTileF + kw * kHalfF;
      // All 16 loads first, so that they are in flight together.
      uint4 wv[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = lane + 32 * (i & 3);
        const int c = 4 * kw + (i >> 2);
        wv[i] = t < rows_in ? lds128(raw + t * 128 + ((c ^ (t & 7)) << 4))
                            : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = lane + 32 * (i & 3);
        const int c = 4 * kw + (i >> 2);
        const uint4 w = wv[i];
        uint32_t h[8];
        e4m3x4_to_f16x2x2(w.x, h[0], h[1]);
        e4m3x4_to_f16x2x2(w.y, h[2], h[3]);
        e4m3x4_to_f16x2x2(w.z, h[4], h[5]);
        e4m3x4_to_f16x2x2(w.w, h[6], h[7]);
        const uint32_t row = dsth + t * 128;
        const uint32_t c0 = 2 * (c & 3);
        tc::st_shared_v4(row + ((c0 ^ (t & 7)) << 4), h[0], h[1], h[2], h[3]);
        tc::st_shared_v4(row + (((c0 + 1) ^ (t & 7)) << 4), h[4], h[5], h[6],
                         h[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars.kf_full[f]));
        mbar_arrive(smem_u32(&bars.k_empty[s]));
      }
    }
    if (!ok && lane == 0) {
      if (!*(volatile int*)&abort_sh) record_status(p.status, KV_ERR_TIMEOUT, 24);
      atomicExch(&abort_sh, 1);
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer --------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t id = idesc_k0(128, kT);  // f16 A and B, M = N = 128
      bool ok = true;
      auto pv = [&](int jp) {
        const int f = jp % kNFV;
        if (!mbar_wait(smem_u32(&bars.p_full), jp & 1)) return false;
        if (!mbar_wait(smem_u32(&bars.vf_full[f]), (jp / kNFV) & 1)) return false;
        fence_after_sync();
        const uint32_t fst = sVF + f * kTileF;
#pragma unroll
        for (int kt = 0; kt < kT / 16; ++kt) {
          const uint64_t bd =
              sdesc(fst + (kt >> 2) * kHalfF + (kt & 3) * 32, 16, 1024);
          umma_ts(tmem + kColO, tmem + (jp & 1) * kT + p_col(kt), bd, id,
                  (jp > 0 || kt > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars.vf_empty[f]));
        umma_commit(smem_u32(&bars.pv_done));
        return true;
      };
      for (int j = 0; j < ntile && ok; ++j) {
        const int f = j % kNFK, b = j & 1;
        if (*(volatile int*)&abort_sh ||
            !mbar_wait(smem_u32(&bars.kf_full[f]), (j / kNFK) & 1)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t kst = sKF + f * kTileF;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd =
              sdesc(kst + (kk >> 2) * kHalfF + (kk & 3) * 32, 16, 1024);
          umma_ts(tmem + b * kT, tmem + kColQ + kk * 8, bd, id,
                  kk > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars.kf_empty[f]));
        umma_commit(smem_u32(&bars.s_full[b]));
        if (j >= 1) ok = pv(j - 1);
      }
      if (ok && ntile > 0) ok = pv(ntile - 1);
      if (!ok) {
        record_status(p.status, KV_ERR_TIMEOUT, 22);
        atomicExch(&abort_sh, 1);
      }
      umma_commit(smem_u32(&bars.o_ready));
      umma_commit(smem_u32(&bars.drain));
      mbar_wait(smem_u32(&bars.drain), 0);
    }
  } else {
    // ---- softmax rows: two threads per row (warps 0-7).  Thread t holds row
    // r = t % 128 (TMEM lane r; warp w reaches lanes 32 (w % 4) ..) and the
    // 64 columns of half h = t / 128 of each S tile, i.e. blocks 4h .. 4h + 3.
    const int h = threadIdx.x >> 7;
    const int r = threadIdx.x & 127;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    float m_used = -INFINITY, l = 0.f, vref = 0.f;
    bool ok = true;
    for (int j = 0; j < ntile; ++j) {
      const int b = j & 1, sc = j % kSC;
      if (*(volatile int*)&abort_sh ||
          !mbar_wait(smem_u32(&bars.s_full[b]), (j >> 1) & 1) ||
          !mbar_wait(smem_u32(&bars.sc_full[sc]), (j / kSC) & 1)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const int valid = min(kT, (nblk - j * kTB) * 16);
      const int nvb = (valid + 15) >> 4;
      // Scale records: every block's V scale (for vref), this half's blocks'
      // K factors and V scales.
      const uint32_t rec = sS + sc * (kTB * 16);
      float vmax = 0.f;
#pragma unroll
      for (int bb = 0; bb < kTB; ++bb)
        vmax = fmaxf(vmax, bb < nvb ? lds64f(rec + bb * 16).y : 0.f);
      float kf[4], vsc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int bb = 4 * h + q;
        const float2 sr = lds64f(rec + bb * 16);
        kf[q] = bb < nvb ? fsc * sr.x : 0.f;
        vsc[q] = bb < nvb ? sr.y : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.sc_empty[sc]));
      float vfac = 1.f;
      if (vmax > vref) {
        vfac = vref / vmax;
        vref = vmax;
      }
      const uint32_t srow = lane_base + b * kT + h * 64;
      const int hv = valid - h * 64;  // valid columns of this half (may be <= 0)
      // Pass 1: maximum over this half's valid tokens.  The K scale factor of
      // a block is positive, so the maximum of the scaled scores of a block is
      // the factor times the maximum of its raw scores.  Blocks past the
      // item's range have no record in this stage (the slot holds whatever an
      // earlier tile or kernel left there) and are skipped.
      float mx = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t sv[32];
        tmem_ld32(srow + cc * 32, sv);
        tmem_wait_ld();
        float bm[2] = {-INFINITY, -INFINITY};
        if (hv >= (cc + 1) * 32) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            bm[i >> 4] = fmaxf(bm[i >> 4], __uint_as_float(sv[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (cc * 32 + i < hv)
              bm[i >> 4] = fmaxf(bm[i >> 4], __uint_as_float(sv[i]));
        }
        if (4 * h + 2 * cc < nvb) mx = fmaxf(mx, bm[0] * kf[2 * cc]);
        if (4 * h + 2 * cc + 1 < nvb) mx = fmaxf(mx, bm[1] * kf[2 * cc + 1]);
      }
      // The row maximum: both halves of the row publish theirs.
      xmax_sh[b][h][r] = mx;
      mbar_arrive(smem_u32(&bars.xch[b]));
      if (!mbar_wait(smem_u32(&bars.xch[b]), (j >> 1) & 1)) {
        ok = false;
        break;
      }
      mx = fmaxf(xmax_sh[b][0][r], xmax_sh[b][1][r]);
      const bool need = mx > m_used + kRescale;
      const float m_new = need ? mx : m_used;
      const float alpha = need ? ex2(m_used - m_new) : 1.f;
      l *= alpha;
      m_used = m_new;
      // Pass 2: P' = 2^(x - m + log2(vs / vref)) as f16 -- the V scale of the
      // block relative to vref (a power of two, at most 1) folded into the
      // exponent -- and l += P' * (vref / vs) per block.  Blocks whose V scale
      // is below 2^-64 of vref keep the factor 2^-64 (their V values are
      // negligible next to the largest; l stays exact).  The P of a 32-column
      // chunk goes over the chunk's own last 16 columns, already read.
      float lv[4], il[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = 4 * h + q < nvb
                          ? scale_exponent(vsc[q]) - scale_exponent(vref)
                          : 0;
        const int ec = e < -64 ? -64 : e;
        lv[q] = (float)ec - m_used;
        il[q] = pow2f(-ec);
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t sv[32];
        tmem_ld32(srow + cc * 32, sv);
        tmem_wait_ld();
        const float f0 = kf[2 * cc], f1 = kf[2 * cc + 1];
        const float a0 = lv[2 * cc], a1 = lv[2 * cc + 1];
        float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        uint32_t pk[16];
        if (hv >= (cc + 1) * 32) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const bool lo = i < 8;
            const float p0 = ex2(fmaf(__uint_as_float(sv[2 * i]), lo ? f0 : f1,
                                      lo ? a0 : a1));
            const float p1 = ex2(fmaf(__uint_as_float(sv[2 * i + 1]),
                                      lo ? f0 : f1, lo ? a0 : a1));
            acc[i >> 3][i & 1] += p0 + p1;
            pk[i] = pack_f16(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const bool lo = i < 8;
            const int t0 = cc * 32 + 2 * i;
            float p0 = ex2(fmaf(__uint_as_float(sv[2 * i]), lo ? f0 : f1,
                                lo ? a0 : a1));
            float p1 = ex2(fmaf(__uint_as_float(sv[2 * i + 1]), lo ? f0 : f1,
                                lo ? a0 : a1));
            p0 = t0 < hv ? p0 : 0.f;
            p1 = t0 + 1 < hv ? p1 : 0.f;
            acc[i >> 3][i & 1] += p0 + p1;
            pk[i] = pack_f16(p0, p1);
          }
        }
        l = fmaf(acc[0][0] + acc[0][1], il[2 * cc],
                 fmaf(acc[1][0] + acc[1][1], il[2 * cc + 1], l));
        tmem_st16(srow + cc * 32 + 16, pk);
      }
      if (j > 0 && (__any_sync(0xffffffffu, need) || vfac != 1.f)) {
        // Rescale this half of the row of O (it holds PV up to tile j - 1)
        // once PV(j - 1) is done.  PV(j) cannot have started (it waits for
        // this tile's P), so the barrier has completed j - 1 or j phases and
        // the parity wait is exact.
        if (!mbar_wait(smem_u32(&bars.pv_done), (j - 1) & 1)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const float f = alpha * vfac;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t ov[32];
          tmem_ld32(lane_base + kColO + h * 64 + cc * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
          tmem_st32(lane_base + kColO + h * 64 + cc * 32, ov);
        }
      }
      tmem_wait_st();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.p_full));
    }
    if (!ok) {
      if (lane == 0) record_status(p.status, KV_ERR_TIMEOUT, 23);
      atomicExch(&abort_sh, 1);
    }
    xl_sh[h][r] = l;
    if (h == 0) xm_sh[r] = m_used;
    // Epilogue: this half of the O row from TMEM -> unnormalised partial row
    // (the row's (m, l) is written after the block-wide barrier below).
    const bool done = mbar_wait(smem_u32(&bars.o_ready), 0);
    fence_after_sync();
    if (__all_sync(0xffffffffu, done && ok && !*(volatile int*)&abort_sh)) {
      float* dst = p.o + (int64_t)(it.prow_base + r) * 128 + h * 64;
      const float oscale = vref;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t ov[32];
        tmem_ld32(lane_base + kColO + h * 64 + cc * 32, ov);
        tmem_wait_ld();
        if (r < it.nrows) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + cc * 32 + i) =
                make_float4(__uint_as_float(ov[i]) * oscale,
                            __uint_as_float(ov[i + 1]) * oscale,
                            __uint_as_float(ov[i + 2]) * oscale,
                            __uint_as_float(ov[i + 3]) * oscale);
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (threadIdx.x < it.nrows && !*(volatile int*)&abort_sh)
    p.ml[it.prow_base + threadIdx.x] = make_float2(
        xm_sh[threadIdx.x], xl_sh[0][threadIdx.x] + xl_sh[1][threadIdx.x]);
  if (warp == kMmaWarp) {
    asm volatile(
        "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
        "r"(kTmemCols)
        : "memory");
  }
}

}  // namespace tc8

cudaError_t launch_tile_e4m3(const SplitParams& sp, const WorkItem* items,
                             int n_items, const void* k8, const void* v8,
                             const void* scales, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(
        tc8::tile_e4m3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        tc8::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  tc8::tile_e4m3_kernel<<<n_items, tc8::kThreads, tc8::kSmem, stream>>>(
      sp, items, static_cast<const uint8_t*>(k8),
      static_cast<const uint8_t*>(v8), static_cast<const float4*>(scales));
  return cudaGetLastError();
}

}  // namespace pkv

// Shared-prefix tile kernel for e4m3 pools on the tcgen05 tensor cores.
//
// One CTA = one tile item: up to 128 query rows of a shared-prefix segment x
// one kv-head x a range of the segment's blocks, every block read once for
// all rows ("Dismantling the Memory Wall", copy-on-write section: shared
// prefixes are stored once; RKSC summary §1.1: the cross-branch re-read is
// the waste).  The e4m3 codes go to the tensor cores as they are stored:
//
//   S = Q K^T  tcgen05.mma kind::f8f6f4, A = Q, B = the K codes.  The pool's
//              K tile (16 rows of 128 bytes, 16-byte chunks XOR-swizzled by
//              row) is already the canonical 128-byte-swizzle K-major layout,
//              so the 8 tiles of a 128-token tile, copied back to back, are
//              the B operand.  Q is carried as three e4m3 parts (hi + mid +
//              lo, after a per-row power-of-two scaling; relative error about
//              2^-12) whose products accumulate into one S.
//   O += P V   tcgen05.mma kind::f16: A = P (f16 pairs in TMEM), B = V^T in
//              f16.  Two converter warps widen each transposed V tile
//              (exact) into the 128-byte-swizzle K-major layout, tokens past
//              the range as zeros.
//   softmax    one thread per row (TMEM lane = row), base 2, lazy maximum
//              (O, l rescaled only when the row maximum grows by more than
//              2^8).  The per-block K scale folds into the score factor; the
//              per-block V scale folds into P relative to the largest V scale
//              seen so far (O is rescaled when that grows).
//
// Warps: 0-3 softmax rows (they also split Q into its parts), 4 MMA issuer,
// 5 K producer (8 bulk copies of 2 KB per tile, and the tiles' 16-byte scale
// records into a 4-stage ring), 6 V producer, 7-8 V converters.
// Partial rows (o, m, l) go to the workspace and are merged by log-sum-exp
// with the other passes, exactly as for the bf16 tile kernel.

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
using tc::umma_f8;
using tc::umma_ts;

constexpr int kT = 128;                   // tokens per tile
constexpr int kTB = kT / 16;              // blocks per tile
constexpr int kNS = 2;                    // stages of the K and raw V rings
constexpr int kSC = 4;                    // stages of the scale-record ring
constexpr int kTile8 = kT * 128;          // 8 blocks' K (or V) codes: 16 KB
constexpr int kHalfF = 128 * 128;         // f16 V^T, 64 tokens x 128 dims
constexpr int kTileF = 2 * kHalfF;        // f16 V^T tile: 32 KB
constexpr int kQPart = 128 * 128;         // one e4m3 part of Q: 16 KB
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kNS * kTile8;
constexpr int kOffF = kOffV + kNS * kTile8;
constexpr int kOffQ = kOffF + 2 * kTileF;
constexpr int kOffS = kOffQ + 3 * kQPart;
constexpr int kSmem = kOffS + kSC * kTB * 16 + 1024;
constexpr int kThreads = 288;
constexpr int kMmaWarp = 4, kKWarp = 5, kVWarp = 6, kCvtWarp = 7;
// TMEM columns: S[0] 0..127, S[1] 128..255 (fp32), P 256..319 (f16 pairs),
// O 320..447 (fp32).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColP = 256, kColO = 320;
constexpr float kRescale = 8.f;

struct Bars {
  uint64_t k_full[kNS], k_empty[kNS], v_full[kNS], v_empty[kNS], f_full[2],
      f_empty[2], sc_full[kSC], sc_empty[kSC], s_full[2], p_full, pv_done,
      o_ready, drain;
};

// Two floats -> two e4m3 codes (lower byte = lo): nearest, ties to even,
// saturating at +-448.
__device__ __forceinline__ uint32_t to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two e4m3 codes (lower byte first) -> their values, exactly.
__device__ __forceinline__ float2 from_e4m3x2(uint32_t two) {
  uint32_t lo, hi;
  e4m3x4_to_f16x2x2(two, lo, hi);
  return __half22float2(*reinterpret_cast<const __half2*>(&lo));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void q_ready_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"(5 * 32) : "memory");
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

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sK = base + kOffK, sV = base + kOffV, sF = base + kOffF,
                 sQ = base + kOffQ, sS = base + kOffS;
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
    for (int s = 0; s < kNS; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.k_empty[s]), 1);    // the MMA's commit
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.v_empty[s]), 2);    // both converter warps
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars.f_full[s]), 2);     // both converter warps
      mbar_init(smem_u32(&bars.f_empty[s]), 1);    // the MMA's commit
      mbar_init(smem_u32(&bars.s_full[s]), 1);
    }
    for (int s = 0; s < kSC; ++s) {
      mbar_init(smem_u32(&bars.sc_full[s]), 1);
      mbar_init(smem_u32(&bars.sc_empty[s]), 4);   // the four softmax warps
    }
    mbar_init(smem_u32(&bars.p_full), 4);
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

  // Q rows -> three e4m3 parts in shared memory (128-byte-swizzle K-major:
  // row r at r * 128, 16-byte chunk c at (c ^ (r % 8)) * 16).  Row r is
  // scaled by 2^-sq so that its largest magnitude lies in [128, 256).
  float fsc = 0.f;  // scale_log2 * 2^sq of this thread's row
  if (threadIdx.x < 128) {
    const int r = threadIdx.x;
    const uint4* src = nullptr;
    if (r < it.nrows) {
      const int rr = it.row0 + r;
      const int b = it.branch0 + rr / p.G;
      const int qh = it.g * p.G + rr % p.G;
      src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.Hq + qh) * 128);
    }
    float amax = 0.f;
    if (src) {
#pragma unroll 4
      for (int c = 0; c < 16; ++c) {
        const uint4 v = src[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                                   fabsf(__uint_as_float(w[i] & 0xffff0000u))));
      }
    }
    int sq = amax > 0.f ? scale_exponent(amax) - 7 : 0;
    sq = sq < -100 ? -100 : (sq > 120 ? 120 : sq);
    const float mul = pow2f(-sq);
    fsc = p.scale_log2 * pow2f(sq);
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {           // 16 dimensions per chunk
      uint32_t part[3][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 v = src ? src[2 * c + h] : make_uint4(0, 0, 0, 0);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t e[3][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x0 = __uint_as_float(w[i] << 16) * mul;
          const float x1 = __uint_as_float(w[i] & 0xffff0000u) * mul;
          const uint32_t c0 = to_e4m3x2(x0, x1);
          const float2 d0 = from_e4m3x2(c0);
          const float r0 = x0 - d0.x, r1 = x1 - d0.y;
          const uint32_t c1 = to_e4m3x2(r0, r1);
          const float2 d1 = from_e4m3x2(c1);
          const uint32_t c2 = to_e4m3x2(r0 - d1.x, r1 - d1.y);
          e[0][i] = c0;
          e[1][i] = c1;
          e[2][i] = c2;
        }
#pragma unroll
        for (int pt = 0; pt < 3; ++pt) {
          part[pt][2 * h] = e[pt][0] | (e[pt][1] << 16);
          part[pt][2 * h + 1] = e[pt][2] | (e[pt][3] << 16);
        }
      }
      const uint32_t off = (uint32_t)r * 128 + (((uint32_t)c ^ (r & 7)) << 4);
#pragma unroll
      for (int pt = 0; pt < 3; ++pt)
        tc::st_shared_v4(sQ + pt * kQPart + off, part[pt][0], part[pt][1],
                         part[pt][2], part[pt][3]);
    }
    fence_proxy_async_smem();
  }
  if (warp <= kMmaWarp) {
    fence_before_sync();
    q_ready_barrier();
    fence_after_sync();
  }

  if (warp == kKWarp || warp == kVWarp) {
    // ---- producers: 8 bulk copies of a tile's blocks, one per lane; the K
    // producer also copies the blocks' scale records.  Block-table entries
    // come 32 at a time (4 tiles) in registers, the next window prefetched.
    const bool is_k = warp == kKWarp;
    uint64_t* full = is_k ? bars.k_full : bars.v_full;
    uint64_t* empty = is_k ? bars.k_empty : bars.v_empty;
    const uint32_t ring = is_k ? sK : sV;
    const uint8_t* pool = is_k ? k8 : v8;
    auto win_load = [&](int w) -> int {
      const int idx = w * 32 + lane;
      return idx < nblk ? table[it.blk_begin + idx] : -1;
    };
    int tcur = 0, tnext = 0, wcur = -1;
    int issued = 0, issued_sc = 0;
    bool ok = true;
    for (int j = 0; j < ntile && ok; ++j) {
      const int w = j >> 2;
      if (w != wcur) {
        tcur = (wcur == w - 1 && wcur >= 0) ? tnext : win_load(w);
        tnext = win_load(w + 1);
        wcur = w;
      }
      const int s = j % kNS, sc = j % kSC;
      const int nb_in = min(kTB, nblk - j * kTB);
      if (lane == 0) {
        if (*(volatile int*)&abort_sh ||
            (j >= kNS && !mbar_wait(smem_u32(&empty[s]), ((j / kNS) - 1) & 1)) ||
            (is_k && j >= kSC &&
             !mbar_wait(smem_u32(&bars.sc_empty[sc]), ((j / kSC) - 1) & 1))) {
          ok = false;
        } else {
          mbar_expect_tx(smem_u32(&full[s]), nb_in * 2048);
          if (is_k) mbar_expect_tx(smem_u32(&bars.sc_full[sc]), nb_in * 16);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      int phys = __shfl_sync(0xffffffffu, tcur, ((j & 3) << 3) + (lane & 7));
      if (lane < nb_in) {
        if (phys < 0 || (int64_t)phys >= p.num_blocks) {
          if (is_k) record_status(p.status, KV_ERR_DEVICE, phys);
          phys = 0;  // any block in the pool: the output is unspecified now
        }
        const int64_t tile = (int64_t)phys * p.Hkv + it.g;
        bulk_load(ring + s * kTile8 + lane * 2048, pool + tile * 2048, 2048,
                  smem_u32(&full[s]));
        if (is_k)
          bulk_load(sS + sc * (kTB * 16) + lane * 16, scales + tile, 16,
                    smem_u32(&bars.sc_full[sc]));
      }
      __syncwarp();
      issued = j + 1;
      if (is_k) issued_sc = j + 1;
    }
    if (lane == 0) {
      if (!ok && !*(volatile int*)&abort_sh) {
        record_status(p.status, KV_ERR_TIMEOUT, 20);
        atomicExch(&abort_sh, 1);
      }
      // Let every copy this warp issued land before the CTA can exit.
      for (int j = issued > kNS ? issued - kNS : 0; j < issued; ++j)
        mbar_wait(smem_u32(&full[j % kNS]), (j / kNS) & 1);
      for (int j = issued_sc > kSC ? issued_sc - kSC : 0; j < issued_sc; ++j)
        mbar_wait(smem_u32(&bars.sc_full[j % kSC]), (j / kSC) & 1);
    }
  } else if (warp >= kCvtWarp) {
    // ---- converters: raw V^T tile (8 blocks x [128 dims][16 slots]) ->
    // f16 V^T in two 64-token halves, each 128 rows (dims) x 128 bytes,
    // 16-byte chunk c of row d at (c ^ (d % 8)) * 16.  Warp cw takes
    // dimensions 64 cw .. 64 cw + 63.
    const int cw = warp - kCvtWarp;
    bool ok = true;
    for (int j = 0; j < ntile && ok; ++j) {
      const int s = j % kNS, f = j & 1;
      if (*(volatile int*)&abort_sh ||
          !mbar_wait(smem_u32(&bars.v_full[s]), (j / kNS) & 1) ||
          (j >= 2 && !mbar_wait(smem_u32(&bars.f_empty[f]), ((j >> 1) - 1) & 1))) {
        ok = false;
        break;
      }
      const int nb_in = min(kTB, nblk - j * kTB);
      const uint32_t raw = sV + s * kTile8;
      const uint32_t dstt = sF + f * kTileF;
#pragma unroll 4
      for (int i = 0; i < 16; ++i) {
        const int dim = cw * 64 + lane + 32 * (i & 1);
        const int blk = i >> 1;
        uint32_t h[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (blk < nb_in) {
          const uint4 w = lds128(raw + blk * 2048 + dim * 16);
          e4m3x4_to_f16x2x2(w.x, h[0], h[1]);
          e4m3x4_to_f16x2x2(w.y, h[2], h[3]);
          e4m3x4_to_f16x2x2(w.z, h[4], h[5]);
          e4m3x4_to_f16x2x2(w.w, h[6], h[7]);
        }
        const uint32_t row = dstt + (blk >> 2) * kHalfF + dim * 128;
        const uint32_t c0 = 2 * (blk & 3);
        tc::st_shared_v4(row + (((c0) ^ (dim & 7)) << 4), h[0], h[1], h[2], h[3]);
        tc::st_shared_v4(row + (((c0 + 1) ^ (dim & 7)) << 4), h[4], h[5], h[6],
                         h[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&bars.f_full[f]));
        mbar_arrive(smem_u32(&bars.v_empty[s]));
      }
    }
    if (!ok && lane == 0) {
      if (!*(volatile int*)&abort_sh) record_status(p.status, KV_ERR_TIMEOUT, 21);
      atomicExch(&abort_sh, 1);
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer --------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t id = idesc_k0(128, kT);  // M = N = 128
      bool ok = true;
      auto pv = [&](int jp) {
        const int f = jp & 1;
        if (!mbar_wait(smem_u32(&bars.p_full), jp & 1)) return false;
        if (!mbar_wait(smem_u32(&bars.f_full[f]), (jp >> 1) & 1)) return false;
        fence_after_sync();
        const uint32_t fst = sF + f * kTileF;
#pragma unroll
        for (int kt = 0; kt < kT / 16; ++kt) {
          const uint64_t bd =
              sdesc(fst + (kt >> 2) * kHalfF + (kt & 3) * 32, 16, 1024);
          umma_ts(tmem + kColO, tmem + kColP + kt * 8, bd, id,
                  (jp > 0 || kt > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars.f_empty[f]));
        umma_commit(smem_u32(&bars.pv_done));
        return true;
      };
      for (int j = 0; j < ntile && ok; ++j) {
        const int s = j % kNS, b = j & 1;
        if (*(volatile int*)&abort_sh ||
            !mbar_wait(smem_u32(&bars.k_full[s]), (j / kNS) & 1)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t kst = sK + s * kTile8;
#pragma unroll
        for (int pt = 0; pt < 3; ++pt)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = sdesc(sQ + pt * kQPart + kk * 32, 16, 1024);
            const uint64_t bd = sdesc(kst + kk * 32, 16, 1024);
            umma_f8(tmem + b * kT, ad, bd, id, (pt | kk) ? 1u : 0u);
          }
        umma_commit(smem_u32(&bars.k_empty[s]));
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
    // ---- softmax rows (warps 0-3; thread r <-> TMEM lane r) ----------------
    const int r = threadIdx.x;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
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
      float kf[kTB], vsc[kTB];
      float vmax = 0.f;
#pragma unroll
      for (int bb = 0; bb < kTB; ++bb) {
        const float2 sr = lds64f(sS + sc * (kTB * 16) + bb * 16);
        kf[bb] = bb < nvb ? fsc * sr.x : 0.f;
        vsc[bb] = bb < nvb ? sr.y : 0.f;
        vmax = fmaxf(vmax, vsc[bb]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.sc_empty[sc]));
      float vfac = 1.f;
      if (vmax > vref) {
        vfac = vref / vmax;
        vref = vmax;
      }
      const uint32_t srow = lane_base + b * kT;
      // Pass 1: row maximum over the valid tokens.  The K scale factor of a
      // block is positive, so the maximum of the scaled scores of a block is
      // the factor times the maximum of its raw scores.
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < kT / 32; ++c) {
        uint32_t sv[32];
        tmem_ld32(srow + c * 32, sv);
        tmem_wait_ld();
        float bm[2] = {-INFINITY, -INFINITY};
        if (valid >= (c + 1) * 32) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            bm[i >> 4] = fmaxf(bm[i >> 4], __uint_as_float(sv[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i < valid)
              bm[i >> 4] = fmaxf(bm[i >> 4], __uint_as_float(sv[i]));
        }
        // Blocks past the item's range have no record in this stage (the
        // slot holds whatever an earlier tile or kernel left there).
        if (2 * c < nvb) mx = fmaxf(mx, bm[0] * kf[2 * c]);
        if (2 * c + 1 < nvb) mx = fmaxf(mx, bm[1] * kf[2 * c + 1]);
      }
      const bool need = mx > m_used + kRescale;
      const float m_new = need ? mx : m_used;
      const float alpha = need ? ex2(m_used - m_new) : 1.f;
      l *= alpha;
      m_used = m_new;
      // Pass 2: P' = 2^(x - m + log2(vs / vref)) as f16 -- the V scale of the
      // block relative to vref (a power of two, at most 1) folded into the
      // exponent -- and l += P' * (vref / vs) per block.  Blocks whose V scale
      // is below 2^-64 of vref keep the factor 2^-64 (their V values are
      // negligible next to the largest; l stays exact).
      float lv[kTB], il[kTB];
#pragma unroll
      for (int bb = 0; bb < kTB; ++bb) {
        const int e = bb < nvb ? scale_exponent(vsc[bb]) - scale_exponent(vref)
                               : 0;
        const int ec = e < -64 ? -64 : e;
        lv[bb] = (float)ec - m_used;
        il[bb] = pow2f(-ec);
      }
      uint32_t pk[kT / 2];
#pragma unroll
      for (int c = 0; c < kT / 32; ++c) {
        uint32_t sv[32];
        tmem_ld32(srow + c * 32, sv);
        tmem_wait_ld();
        const float f0 = kf[2 * c], f1 = kf[2 * c + 1];
        const float a0 = lv[2 * c], a1 = lv[2 * c + 1];
        float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        if (valid >= (c + 1) * 32) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const bool lo = i < 8;
            const float p0 = ex2(fmaf(__uint_as_float(sv[2 * i]), lo ? f0 : f1,
                                      lo ? a0 : a1));
            const float p1 = ex2(fmaf(__uint_as_float(sv[2 * i + 1]),
                                      lo ? f0 : f1, lo ? a0 : a1));
            acc[i >> 3][i & 1] += p0 + p1;
            pk[c * 16 + i] = pack_f16(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const bool lo = i < 8;
            const int t0 = c * 32 + 2 * i;
            float p0 = ex2(fmaf(__uint_as_float(sv[2 * i]), lo ? f0 : f1,
                                lo ? a0 : a1));
            float p1 = ex2(fmaf(__uint_as_float(sv[2 * i + 1]), lo ? f0 : f1,
                                lo ? a0 : a1));
            p0 = t0 < valid ? p0 : 0.f;
            p1 = t0 + 1 < valid ? p1 : 0.f;
            acc[i >> 3][i & 1] += p0 + p1;
            pk[c * 16 + i] = pack_f16(p0, p1);
          }
        }
        l = fmaf(acc[0][0] + acc[0][1], il[2 * c],
                 fmaf(acc[1][0] + acc[1][1], il[2 * c + 1], l));
      }
      if (j > 0 && !mbar_wait(smem_u32(&bars.pv_done), (j - 1) & 1)) {
        ok = false;
        break;
      }
      fence_after_sync();
      if (j > 0 && (__any_sync(0xffffffffu, need) || vfac != 1.f)) {
        const float f = alpha * vfac;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          tmem_ld32(lane_base + kColO + c * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
          tmem_st32(lane_base + kColO + c * 32, ov);
        }
      }
#pragma unroll
      for (int c = 0; c < kT / 32; ++c) {
        uint32_t q16[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) q16[i] = pk[c * 16 + i];
        tmem_st16(lane_base + kColP + c * 16, q16);
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
    const bool done = mbar_wait(smem_u32(&bars.o_ready), 0);
    fence_after_sync();
    if (__all_sync(0xffffffffu, done && ok && !*(volatile int*)&abort_sh)) {
      float* dst = p.o + (int64_t)(it.prow_base + r) * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        tmem_ld32(lane_base + kColO + c * 32, ov);
        tmem_wait_ld();
        if (r < it.nrows) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + c * 32 + i) =
                make_float4(__uint_as_float(ov[i]) * vref,
                            __uint_as_float(ov[i + 1]) * vref,
                            __uint_as_float(ov[i + 2]) * vref,
                            __uint_as_float(ov[i + 3]) * vref);
        }
      }
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

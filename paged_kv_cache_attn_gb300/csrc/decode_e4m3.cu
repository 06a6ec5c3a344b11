// Split-KV decode kernel for e4m3 pools.
//
// Same work items, partial rows and merge as the bf16 split-KV kernel in
// decode.cu; what differs is how a (block, kv-head) tile reaches the tensor
// cores.  The tile layouts of an e4m3 pool (pagedkv.h) are chosen so that
// every lane's 16-byte shared-memory load already holds its mma.sync operand
// fragments, conflict-free, with no transpose:
//  * Tiles arrive with three 1-D bulk copies per block (K codes, V codes, the
//    16-byte scale record), completing on the stage's mbarrier; each of the
//    4 warps runs its own 4-stage ring (three CTAs per SM).
//  * S = Q K^T with mma.sync m16n8k16 in f16: lane (n = lane / 4, q = lane %
//    4) of n-tile j reads token 4(n / 2) + 2j + n % 2 and the head-dimension
//    slice [q d / 4, (q + 1) d / 4); k-step s of that lane uses dimensions
//    q d / 4 + 4s .. + 3.  Q is loaded with the same dimension order, so the
//    dot products are exact permutations of the plain ones.  The K tile's
//    XOR chunk swizzle (head_dim 128) makes the eight rows of a load phase
//    hit eight different bank groups.
//  * With that token order, a lane's S accumulator columns are tokens
//    4q .. 4q + 3, which is the A operand of O += P V; the V tile is stored
//    transposed (16 slots per dimension), so those four tokens of the lane's
//    dimension are one aligned 32-bit word: one load per n-tile, and the 32
//    lanes of a load read 128 contiguous bytes.
//  * Each warp takes two of its blocks per iteration: four independent QK
//    accumulation chains, one softmax update over 32 tokens.  The softmax
//    keeps a lazy reference maximum per row that moves (rescaling O and l)
//    only when a block raises the row maximum by more than 2^8.
//  * Codes widen to f16 exactly (cvt e4m3x2 -> f16x2).  The K scale folds
//    into the per-row score multiplier; the V scale folds into P relative to
//    a running power-of-two reference (O is rescaled when a larger V scale
//    arrives), so P stays below 2^8 in f16.  q is scaled per row by a power
//    of two so its largest element lies in [2^14, 2^15) before the f16
//    conversion, and the factor is folded back into the scores.
//  * Masked slots may hold any code (NaN included): their scores are -inf
//    by selection and their V bytes are masked to zero in registers.

#include <cmath>

#include "device_common.cuh"
#include "e4m3.cuh"

namespace pkv {

namespace {

__device__ __forceinline__ void mma_16816_f16(float (&c)[4],
                                              const uint32_t (&a)[4],
                                              uint32_t b0, uint32_t b1) {
  // Not volatile: no side effects, so the compiler may move it around the
  // (volatile) shared-memory loads and overlap their latency.
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int D, int NS>
struct E4m3Cfg {
  static constexpr int kWarps = 4;
  static constexpr int kTile = 16 * D;          // bytes of one K (or V) tile
  static constexpr int kStage = 2 * kTile + 128;  // K, V, scale record, pad
  static constexpr int kRing = kWarps * NS * kStage;
  static constexpr int kMerge = kWarps * 16 * D * 4;
  static constexpr int kSmem = (kRing > kMerge ? kRing : kMerge) + 128;
  static constexpr int kChunks = D / 64;        // K chunks per lane and row
};

constexpr int kE4m3Stages = 4;

// kPerWarp: every warp takes a (short) item of its own, item
// item_base + 4 * blockIdx.x + warp, and writes its partial rows itself; a
// separate instantiation so that the CTA-wide one keeps its registers.
template <int D, int NS, bool kPerWarp>
__global__ void __launch_bounds__(128, 3)
    splitkv_e4m3_kernel(const SplitParams p, const uint8_t* __restrict__ k8,
                        const uint8_t* __restrict__ v8,
                        const float4* __restrict__ scales, int item_base,
                        int n_items) {
  using C = E4m3Cfg<D, NS>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[C::kWarps][NS];
  __shared__ float m_sh[C::kWarps][16];
  __shared__ float l_sh[C::kWarps][16];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(smem_raw) + 127u) & ~127u;
  float* base_ptr =
      reinterpret_cast<float*>(smem_raw + (base - smem_u32(smem_raw)));
  const int idx = kPerWarp ? item_base + 4 * (int)blockIdx.x + warp
                           : item_base + (int)blockIdx.x;
  const WorkItem it = p.items[idx < n_items ? idx : 0];
  bool have = idx < n_items;
  if (have && !item_ok(it, p, 16)) {
    if (kPerWarp ? lane == 0 : threadIdx.x == 0)
      record_status(p.status, KV_ERR_DEVICE, -1 - idx);
    have = false;
  }
  if (!kPerWarp && !have) return;  // the whole CTA, before any barrier
  if (threadIdx.x == 0) {
    for (int w = 0; w < C::kWarps; ++w)
      for (int s = 0; s < NS; ++s) mbar_init(smem_u32(&bars[w][s]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (!have) return;  // a warp without an item (no CTA barrier follows)

  const int G = p.G;
  const int seq_len = it.masked ? p.seq_lens[it.branch0] : 0x7fffffff;
  const int32_t* table = p.tables + (int64_t)it.branch0 * p.max_blocks;
  const int nblk = it.blk_end - it.blk_begin;
  // This warp's blocks of the item: first, first + stride, ...
  const int first = kPerWarp ? 0 : warp;
  constexpr int stride = kPerWarp ? 1 : C::kWarps;
  const int my_n = nblk > first ? (nblk - first + stride - 1) / stride : 0;
  const uint32_t ring = base + warp * NS * C::kStage;
  const uint32_t bar0 = smem_u32(&bars[warp][0]);

  // Block-table entries of this warp's blocks, 32 at a time in registers.
  int tcache = 0, twin = -1;
  auto issue = [&](int k) -> bool {
    if ((k >> 5) != twin) {
      twin = k >> 5;
      const int kk = (twin << 5) + lane;
      tcache = kk < my_n ? table[it.blk_begin + first + stride * kk] : 0;
    }
    const int phys = __shfl_sync(0xffffffffu, tcache, k & 31);
    const bool ok = phys >= 0 && (int64_t)phys < p.num_blocks;
    const int s = k % NS;
    const uint32_t st = ring + s * C::kStage;
    const uint32_t bar = bar0 + s * 8;
    if (ok) {
      fence_proxy_async_smem();
      if (lane == 0) mbar_expect_tx(bar, 2 * C::kTile + 16);
      __syncwarp();
      if (lane < 3) {
        const int64_t tile = (int64_t)phys * p.Hkv + it.g;
        const void* src = lane == 0   ? (const void*)(k8 + tile * C::kTile)
                          : lane == 1 ? (const void*)(v8 + tile * C::kTile)
                                      : (const void*)(scales + tile);
        bulk_load(st + lane * C::kTile, src, lane == 2 ? 16 : C::kTile, bar);
      }
    } else if (lane == 0) {
      record_status(p.status, KV_ERR_DEVICE, phys);
      mbar_arrive(bar);
    }
    return ok;
  };

  uint32_t bad = 0;  // bit s: the block in stage s is outside the pool
  const int pre = my_n < NS ? my_n : NS;
  for (int k = 0; k < pre; ++k)
    if (!issue(k)) bad |= 1u << k;

  // Query fragments in f16, in the lane's dimension order (see above), each
  // row scaled by 2^-sq so that its largest magnitude lies in [2^14, 2^15).
  const int gq = lane >> 2, tq = lane & 3;
  constexpr int kDimsPerLane = D / 4;
  uint32_t qa[D / 16][4];
  float fsc[2];
  {
    float qv[2][kDimsPerLane];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = gq + 8 * hr;
      const __nv_bfloat16* rowp = nullptr;
      if (r < it.nrows) {
        const int rr = it.row0 + r;
        const int b = it.branch0 + rr / G;
        const int qh = it.g * G + rr % G;
        rowp = p.q + ((int64_t)b * p.Hq + qh) * D + tq * kDimsPerLane;
      }
      float amax = 0.f;
#pragma unroll
      for (int v = 0; v < kDimsPerLane / 8; ++v) {
        uint4 w = rowp ? *reinterpret_cast<const uint4*>(rowp + 8 * v)
                       : make_uint4(0, 0, 0, 0);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float lo = __uint_as_float(ws[i] << 16);
          const float hi = __uint_as_float(ws[i] & 0xffff0000u);
          qv[hr][8 * v + 2 * i] = lo;
          qv[hr][8 * v + 2 * i + 1] = hi;
          amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
        }
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      int sq = amax > 0.f ? scale_exponent(amax) - 14 : 0;
      sq = sq < -100 ? -100 : sq;
      const float mul = pow2f(-sq);
#pragma unroll
      for (int i = 0; i < kDimsPerLane; ++i) qv[hr][i] *= mul;
      fsc[hr] = p.scale_log2 * pow2f(sq);
    }
#pragma unroll
    for (int s = 0; s < D / 16; ++s) {
      qa[s][0] = pack_f16(qv[0][4 * s], qv[0][4 * s + 1]);
      qa[s][1] = pack_f16(qv[1][4 * s], qv[1][4 * s + 1]);
      qa[s][2] = pack_f16(qv[0][4 * s + 2], qv[0][4 * s + 3]);
      qa[s][3] = pack_f16(qv[1][4 * s + 2], qv[1][4 * s + 3]);
    }
  }

  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};
  float vref = 0.f;  // O is held in units of vref (a power of two)
  float o[D / 8][4];
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[nt][i] = 0.f;

  bool timed_out = false;
  int k = 0;
  // An item of at most 8 rows (one branch at G <= 8) leaves rows 8-15 of the
  // 16-row MMA tile empty: their softmax is skipped (uniform in the warp),
  // and their P is zero.
  const bool lo_only = it.nrows <= 8;
  // Two of the warp's blocks per iteration (a and a + 1 of its sequence):
  // four independent QK accumulation chains and one softmax update over 32
  // tokens.  m_r is a lazy reference maximum: it moves (and O, l are
  // rescaled) only when a row's maximum exceeds it by more than 2^8, so the
  // weights 2^(x - m_r) stay below 2^8 and f16 P keeps them.
  for (; k < my_n; k += 2) {
    const int nblk2 = k + 1 < my_n ? 2 : 1;
    int stg[2], nv[2];
    bool use[2];
    float2 scl[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      stg[u] = (k + u) % NS;
      use[u] = false;
      nv[u] = 0;
      scl[u] = make_float2(0.f, 0.f);
      if (u < nblk2) {
        if (!mbar_wait(bar0 + stg[u] * 8, ((k + u) / NS) & 1)) timed_out = true;
        use[u] = !((bad >> stg[u]) & 1);
        const int j = it.blk_begin + first + stride * (k + u);
        const int n = seq_len - j * 16;
        nv[u] = use[u] ? (n > 16 ? 16 : n) : 0;
        if (use[u]) scl[u] = lds64f(ring + stg[u] * C::kStage + 2 * C::kTile);
      }
    }
    if (timed_out) break;

    // S = Q K^T for both blocks.
    float sacc[2][2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int jn = 0; jn < 2; ++jn)
#pragma unroll
        for (int i = 0; i < 4; ++i) sacc[u][jn][i] = 0.f;
#pragma unroll
    for (int kq = 0; kq < C::kChunks; ++kq) {
      uint4 w[2][2];
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int jn = 0; jn < 2; ++jn) {
          const int tk = 4 * (gq >> 1) + 2 * jn + (gq & 1);
          const int c = D == 128 ? 2 * tq + kq : tq;
          const int pc = D == 128 ? (c ^ (tk & 7)) : c;
          w[u][jn] = use[u] ? lds128(ring + stg[u] * C::kStage + tk * D + pc * 16)
                            : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int jn = 0; jn < 2; ++jn) {
            const uint32_t wd = i == 0   ? w[u][jn].x
                                : i == 1 ? w[u][jn].y
                                : i == 2 ? w[u][jn].z
                                         : w[u][jn].w;
            uint32_t b0, b1;
            e4m3x4_to_f16x2x2(wd, b0, b1);
            mma_16816_f16(sacc[u][jn], qa[4 * kq + i], b0, b1);
          }
    }
    // Scale, mask (tokens past nv, and blocks not in use).
    float x[2][2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float f0 = fsc[0] * scl[u].x, f1 = fsc[1] * scl[u].x;
#pragma unroll
      for (int jn = 0; jn < 2; ++jn)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          x[u][jn][i] = sacc[u][jn][i] * (i < 2 ? f0 : f1);
      if (nv[u] < 16) {
#pragma unroll
        for (int jn = 0; jn < 2; ++jn)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (4 * tq + 2 * jn + (i & 1) >= nv[u]) x[u][jn][i] = -INFINITY;
      }
    }
    // V scale reference: the largest V scale seen so far.
    const float vmax = fmaxf(scl[0].y, scl[1].y);
    float vfac = 1.f;
    if (vmax > vref) {
      vfac = vref / vmax;
      vref = vmax;
    }
    float alpha[2] = {1.f, 1.f};
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      if (hr == 1 && lo_only) break;
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < 2; ++u)
        mx = fmaxf(mx, fmaxf(fmaxf(x[u][0][2 * hr], x[u][0][2 * hr + 1]),
                             fmaxf(x[u][1][2 * hr], x[u][1][2 * hr + 1])));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (mx > m_r[hr] + 8.f) {  // also when m_r is -inf and mx finite
        alpha[hr] = ex2(m_r[hr] - mx);
        m_r[hr] = mx;
      }
    }
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f) ||
        vfac != 1.f) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        l_r[hr] *= alpha[hr];
        const float f = alpha[hr] * vfac;
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
          o[nt][2 * hr] *= f;
          o[nt][2 * hr + 1] *= f;
        }
      }
    }
    uint32_t pa[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float pfac = use[u] ? scl[u].y / vref : 0.f;
      float pr[2][4];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        if (hr == 1 && lo_only) {
          pr[0][2] = pr[0][3] = pr[1][2] = pr[1][3] = 0.f;
          break;
        }
        const float m_use = m_r[hr] == -INFINITY ? 0.f : m_r[hr];
        float sum = 0.f;
#pragma unroll
        for (int jn = 0; jn < 2; ++jn)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float pv = ex2(x[u][jn][2 * hr + e] - m_use);
            pr[jn][2 * hr + e] = pv * pfac;
            sum += pv;
          }
        l_r[hr] += sum;
      }
      pa[u][0] = pack_f16(pr[0][0], pr[0][1]);
      pa[u][1] = pack_f16(pr[0][2], pr[0][3]);
      pa[u][2] = pack_f16(pr[1][0], pr[1][1]);
      pa[u][3] = pack_f16(pr[1][2], pr[1][3]);
    }
    // O += P V for each block in use; bytes of tokens at or past nv are
    // zeroed before widening (masked slots may hold NaN codes).
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!use[u]) continue;
      int keep = nv[u] - 4 * tq;
      keep = keep < 0 ? 0 : (keep > 4 ? 4 : keep);
      const uint32_t vmask = keep == 4 ? 0xffffffffu : ((1u << (8 * keep)) - 1u);
      const uint32_t vt =
          ring + stg[u] * C::kStage + C::kTile + gq * 16 + tq * 4;
      const bool partial = nv[u] < 16;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        uint32_t w = lds32(vt + nt * 128);  // dimension 8 nt + gq
        if (partial) w &= vmask;
        uint32_t b0, b1;
        e4m3x4_to_f16x2x2(w, b0, b1);
        mma_16816_f16(o[nt], pa[u], b0, b1);
      }
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u < nblk2 && k + u + NS < my_n) {
        if (issue(k + u + NS))
          bad &= ~(1u << stg[u]);
        else
          bad |= 1u << stg[u];
      }
    }
  }
  if (timed_out) {
    if (lane == 0) record_status(p.status, KV_ERR_TIMEOUT, 2);
    for (int kk = k; kk < my_n && kk < k + NS; ++kk)
      mbar_wait(bar0 + (kk % NS) * 8, (kk / NS) & 1);
  }

#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 1);
    l_r[hr] += __shfl_xor_sync(0xffffffffu, l_r[hr], 2);
  }

  if (kPerWarp) {
    // The warp's own item: its state is the partial result (O back to plain
    // units, x vref).  Lane (gq, tq) holds rows gq and gq + 8, columns
    // 8 nt + 2 tq and + 1.
    float* dst = p.o + (int64_t)it.prow_base * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + 2 * tq;
      if (gq < it.nrows)
        *reinterpret_cast<float2*>(dst + gq * D + col) =
            make_float2(o[nt][0] * vref, o[nt][1] * vref);
      if (gq + 8 < it.nrows)
        *reinterpret_cast<float2*>(dst + (gq + 8) * D + col) =
            make_float2(o[nt][2] * vref, o[nt][3] * vref);
    }
    if (tq == 0) {
      if (gq < it.nrows) p.ml[it.prow_base + gq] = make_float2(m_r[0], l_r[0]);
      if (gq + 8 < it.nrows)
        p.ml[it.prow_base + gq + 8] = make_float2(m_r[1], l_r[1]);
    }
    return;
  }

  // Combine the four warps' partial states through shared memory; O goes
  // back to plain units (x vref).
  __syncthreads();
  float* Ow = base_ptr + warp * 16 * D;
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    const int col = nt * 8 + 2 * tq;
    *reinterpret_cast<float2*>(Ow + gq * D + col) =
        make_float2(o[nt][0] * vref, o[nt][1] * vref);
    *reinterpret_cast<float2*>(Ow + (gq + 8) * D + col) =
        make_float2(o[nt][2] * vref, o[nt][3] * vref);
  }
  if (tq == 0) {
    m_sh[warp][gq] = m_r[0];
    m_sh[warp][gq + 8] = m_r[1];
    l_sh[warp][gq] = l_r[0];
    l_sh[warp][gq + 8] = l_r[1];
  }
  __syncthreads();
  {
    const int row = threadIdx.x >> 3;  // 16 rows x 8 threads
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
      if ((threadIdx.x & 7) == 0)
        p.ml[it.prow_base + row] = make_float2(mstar, lstar);
    }
  }
}

// The long items one per CTA, then the last n_warp_items (short) one per
// warp, four to a CTA, on the same stream.
template <int D>
cudaError_t launch_t(const SplitParams& sp, const void* k8, const void* v8,
                     const void* scales, int n_items, int n_warp_items,
                     cudaStream_t stream) {
  using C = E4m3Cfg<D, kE4m3Stages>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        splitkv_e4m3_kernel<D, kE4m3Stages, false>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(splitkv_e4m3_kernel<D, kE4m3Stages, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (n_warp_items < 0 || n_warp_items > n_items) return cudaErrorInvalidValue;
  const int n_long = n_items - n_warp_items;
  const auto* k = static_cast<const uint8_t*>(k8);
  const auto* v = static_cast<const uint8_t*>(v8);
  const auto* s = static_cast<const float4*>(scales);
  if (n_long > 0)
    splitkv_e4m3_kernel<D, kE4m3Stages, false>
        <<<n_long, 128, C::kSmem, stream>>>(sp, k, v, s, 0, n_items);
  if (n_warp_items > 0)
    splitkv_e4m3_kernel<D, kE4m3Stages, true>
        <<<(n_warp_items + 3) / 4, 128, C::kSmem, stream>>>(sp, k, v, s,
                                                            n_long, n_items);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_split_e4m3(const SplitParams& sp, const void* k8,
                              const void* v8, const void* scales, int n_items,
                              int n_warp_items, int d, cudaStream_t stream) {
  return d == 128 ? launch_t<128>(sp, k8, v8, scales, n_items, n_warp_items,
                                  stream)
                  : launch_t<64>(sp, k8, v8, scales, n_items, n_warp_items,
                                 stream);
}

}  // namespace pkv

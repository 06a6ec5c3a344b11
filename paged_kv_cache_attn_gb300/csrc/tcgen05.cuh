// tcgen05 / TMEM / TMA helpers shared by the tensor-core decode kernels.
// Inline PTX for sm_103a.
#pragma once

#include "device_common.cuh"

namespace pkv {
namespace tc {

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 format: start
// address >> 4 in bits 0-13, leading byte offset >> 4 in 16-29, stride byte
// offset >> 4 in 32-45, version 1 in 46-47, layout type 2 in 61-63).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo,
                                          uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) |
         ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A
// K-major, B K-major or MN-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (+)= A B, kind::f16, with A read from tensor memory (16-bit A: two
// elements per column) and B from a shared-memory descriptor.
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a,
                                        uint64_t b, uint32_t id,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
          tmem_d),
      "r"(tmem_a), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

// D (+)= A B, kind::f16, with A and B both from shared-memory descriptors.
__device__ __forceinline__ void umma_ss(uint32_t tmem_d, uint64_t a, uint64_t b,
                                        uint32_t id, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::f16 with A and B both K-major and f16
// (format code 0), fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_k0(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 5-D TMA load (coordinates x0..x4) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* tm,
                                            int x4, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::"
      "bytes [%0], [%1, {%2, %2, %2, %2, %3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(0), "r"(x4), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

#define PKV_R32(a)                                                           \
  "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]),    \
      "=r"(a[6]), "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]),           \
      "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),       \
      "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]),       \
      "=r"(a[21]), "=r"(a[22]), "=r"(a[23]), "=r"(a[24]), "=r"(a[25]),       \
      "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]),       \
      "=r"(a[31])
#define PKV_W32(a)                                                           \
  "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]),          \
      "r"(a[6]), "r"(a[7]), "r"(a[8]), "r"(a[9]), "r"(a[10]), "r"(a[11]),    \
      "r"(a[12]), "r"(a[13]), "r"(a[14]), "r"(a[15]), "r"(a[16]),            \
      "r"(a[17]), "r"(a[18]), "r"(a[19]), "r"(a[20]), "r"(a[21]),            \
      "r"(a[22]), "r"(a[23]), "r"(a[24]), "r"(a[25]), "r"(a[26]),            \
      "r"(a[27]), "r"(a[28]), "r"(a[29]), "r"(a[30]), "r"(a[31])

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, "
      "[%32];"
      : PKV_R32(v)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr,
                                          const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      PKV_W32(v)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr,
                                          const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
      "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
      "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a,
                                             uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}

// ---- the softmax rows of the tcgen05 tile kernels ---------------------------
// One thread owns one query row (its TMEM lane).  S of a 128-token tile sits
// in 128 fp32 columns at `srow`; `valid` of its tokens count.

// Base-2 online softmax over one tile, with a lazy maximum: the row's
// reference m moves (and O, l are rescaled by the returned alpha) only when
// the tile's maximum exceeds it by more than `lazy` (log2 units), so every
// weight stays below 2^lazy.  P = 2^(s * scale_log2 - m) is written as bf16
// pairs over the first 64 columns of the same S: chunk c of P lands on
// columns 16c .. 16c + 15, which this thread has already read.  Returns
// whether m moved.
__device__ __forceinline__ bool softmax_tile(uint32_t srow, int valid,
                                             float scale_log2, float lazy,
                                             float& m_used, float& l,
                                             float& alpha) {
  // Pass 1: row maximum over the tile's valid tokens.
  float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t sv[32];
    tmem_ld32(srow + c * 32, sv);
    tmem_wait_ld();
    if (valid >= (c + 1) * 32) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(sv[i]));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (c * 32 + i < valid)
          mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(sv[i]));
    }
  }
  const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
  const float m_tile = mx * scale_log2;
  const bool need = m_tile > m_used + lazy;
  const float m_new = need ? m_tile : m_used;
  alpha = need ? ex2(m_used - m_new) : 1.f;
  l *= alpha;
  m_used = m_new;
  // Pass 2: P, and its sum into l.
  const float neg_m = -m_used;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t sv[32];
    tmem_ld32(srow + c * 32, sv);
    tmem_wait_ld();
    float acc4[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int t0 = c * 32 + 2 * i;
      float p0 = ex2(fmaf(__uint_as_float(sv[2 * i]), scale_log2, neg_m));
      float p1 = ex2(fmaf(__uint_as_float(sv[2 * i + 1]), scale_log2, neg_m));
      p0 = t0 < valid ? p0 : 0.f;
      p1 = t0 + 1 < valid ? p1 : 0.f;
      acc4[i & 3] += p0 + p1;
      pk[i] = pack_bf16(p0, p1);
    }
    l += (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
    tmem_st16(srow + c * 16, pk);
  }
  return need;
}

// This thread's row of O (128 fp32 columns at `orow`) times alpha.
__device__ __forceinline__ void rescale_o_row(uint32_t orow, float alpha) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t ov[32];
    tmem_ld32(orow + c * 32, ov);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i)
      ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
    tmem_st32(orow + c * 32, ov);
  }
}

// The row's unnormalised partial result: O (128 fp32 columns at `orow`) to
// dst (skipped for a row past the item's rows; the TMEM loads are
// warp-collective, so every lane of the warp calls this).
__device__ __forceinline__ void store_o_row(uint32_t orow, float* dst,
                                            bool row_valid) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t ov[32];
    tmem_ld32(orow + c * 32, ov);
    tmem_wait_ld();
    if (row_valid) {
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + c * 32 + i) =
            make_float4(__uint_as_float(ov[i]), __uint_as_float(ov[i + 1]),
                        __uint_as_float(ov[i + 2]), __uint_as_float(ov[i + 3]));
    }
  }
}

}  // namespace tc
}  // namespace pkv

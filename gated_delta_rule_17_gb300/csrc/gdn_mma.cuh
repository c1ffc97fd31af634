// Warp-level fp16 tensor-core tiles (mma.sync m16n8k16, fp32 accumulate) for the
// backward's chunk contractions.
//
// The backward's per-chunk products come in every orientation (A K^T, A^T B,
// A B^T with the same shared-memory tiles), are small (64 x 64 to 128 x 128
// outputs, 64 or 128 deep) and sit between elementwise epilogues. They are
// written here as warp tiles over plain row-major fp16 tiles in shared memory;
// `ldmatrix` (with or without .trans) loads each operand in whichever
// orientation the product needs, so one stored tile serves as A, A^T, B or B^T.
//
// Tiles are row-major with a leading dimension of (columns + 8) halves: rows stay
// 16-byte aligned for ldmatrix, and the 8 row addresses of one 8 x 8 matrix fall
// in 8 different bank groups.
//
// Accumulator fragment of an m16n8 tile, lane = 4 g + t:
//   c[0], c[1] -> (row g,     columns 2t, 2t + 1)
//   c[2], c[3] -> (row g + 8, columns 2t, 2t + 1)
#pragma once
#include <cuda_fp16.h>
#include <cstdint>

namespace gdn {
namespace mm {

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// c[j] (the m16n8 tiles at columns n0 + 8 j) += A[m0 : m0 + 16, 0 : K] * B[0 : K, n0 : n0 + 8 NT].
//   kAT = false: A is stored row-major as [M][K] at a (leading dimension lda);
//   kAT = true:  A is given by its transpose, stored [K][M].
//   kBT = false: B is stored [K][N];
//   kBT = true:  B is given by its transpose, stored [N][K].
// a, b are shared-space byte addresses of element (0, 0); K is a multiple of 16,
// NT of 2. kUnroll: K steps unrolled together (more fragments in flight, more registers).
template <bool kAT, bool kBT, int NT, int kUnroll = 2>
__device__ __forceinline__ void warp_mma(float (&c)[NT][4], uint32_t a, int lda, uint32_t b, int ldb, int m0, int n0,
                                         int K) {
  static_assert(NT % 2 == 0, "B operands are loaded two n8 tiles at a time");
  const int lane = threadIdx.x & 31;
  // Lanes 8i .. 8i + 7 give the row addresses of the i-th 8 x 8 matrix of an x4 load.
  // A (m16 x k16): matrices (m 0-7, k 0-7), (m 8-15, k 0-7), (m 0-7, k 8-15), (m 8-15, k 8-15).
  // B (k16 x n16): matrices (k 0-7, n 0-7), (k 8-15, n 0-7), (k 0-7, n 8-15), (k 8-15, n 8-15).
  uint32_t a_lane, b_lane;
  int a_step, b_step;  // bytes per 16 of K
  if (!kAT) {
    a_lane = a + 2u * static_cast<uint32_t>((m0 + (lane & 15)) * lda + (lane >> 4) * 8);
    a_step = 32;
  } else {
    a_lane = a + 2u * static_cast<uint32_t>(((lane & 7) + ((lane >> 4) << 3)) * lda + m0 + ((lane >> 3) & 1) * 8);
    a_step = 32 * lda;
  }
  if (kBT) {
    b_lane = b + 2u * static_cast<uint32_t>((n0 + (lane & 7) + ((lane >> 4) << 3)) * ldb + ((lane >> 3) & 1) * 8);
    b_step = 32;
  } else {
    b_lane = b + 2u * static_cast<uint32_t>((lane & 15) * ldb + n0 + (lane >> 4) * 8);
    b_step = 32 * ldb;
  }
  const uint32_t b_pair = kBT ? 32u * ldb : 32u;  // bytes to the next pair of n8 tiles
#pragma unroll kUnroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t af[4];
    if (!kAT) ldsm_x4(a_lane, af);
    else ldsm_x4_t(a_lane, af);
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) {
      uint32_t bf[4];
      if (kBT) ldsm_x4(b_lane + j * b_pair, bf);
      else ldsm_x4_t(b_lane + j * b_pair, bf);
      mma16816(c[2 * j], af, bf[0], bf[1]);
      mma16816(c[2 * j + 1], af, bf[2], bf[3]);
    }
    a_lane += a_step;
    b_lane += b_step;
  }
}

// Two m16 row tiles per warp: c[m][j] += A[m0 + 16 m : +16, 0 : K] * B[0 : K, n0 + 8 j : +8].
// Each B fragment feeds both row tiles, halving B's shared-memory traffic per MMA.
template <bool kAT, bool kBT, int NT, int kUnroll = 2>
__device__ __forceinline__ void warp_mma2(float (&c)[2][NT][4], uint32_t a, int lda, uint32_t b, int ldb, int m0,
                                          int n0, int K) {
  static_assert(NT % 2 == 0, "B operands are loaded two n8 tiles at a time");
  const int lane = threadIdx.x & 31;
  uint32_t a_lane, b_lane;
  int a_step, b_step;
  uint32_t a_next;  // bytes from row tile 0 to row tile 1
  if (!kAT) {
    a_lane = a + 2u * static_cast<uint32_t>((m0 + (lane & 15)) * lda + (lane >> 4) * 8);
    a_step = 32;
    a_next = 32u * lda;
  } else {
    a_lane = a + 2u * static_cast<uint32_t>(((lane & 7) + ((lane >> 4) << 3)) * lda + m0 + ((lane >> 3) & 1) * 8);
    a_step = 32 * lda;
    a_next = 32u;
  }
  if (kBT) {
    b_lane = b + 2u * static_cast<uint32_t>((n0 + (lane & 7) + ((lane >> 4) << 3)) * ldb + ((lane >> 3) & 1) * 8);
    b_step = 32;
  } else {
    b_lane = b + 2u * static_cast<uint32_t>((lane & 15) * ldb + n0 + (lane >> 4) * 8);
    b_step = 32 * ldb;
  }
  const uint32_t b_pair = kBT ? 32u * ldb : 32u;
#pragma unroll kUnroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t af0[4], af1[4];
    if (!kAT) {
      ldsm_x4(a_lane, af0);
      ldsm_x4(a_lane + a_next, af1);
    } else {
      ldsm_x4_t(a_lane, af0);
      ldsm_x4_t(a_lane + a_next, af1);
    }
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) {
      uint32_t bf[4];
      if (kBT) ldsm_x4(b_lane + j * b_pair, bf);
      else ldsm_x4_t(b_lane + j * b_pair, bf);
      mma16816(c[0][2 * j], af0, bf[0], bf[1]);
      mma16816(c[0][2 * j + 1], af0, bf[2], bf[3]);
      mma16816(c[1][2 * j], af1, bf[0], bf[1]);
      mma16816(c[1][2 * j + 1], af1, bf[2], bf[3]);
    }
    a_lane += a_step;
    b_lane += b_step;
  }
}

// Two products that share their B operand: c += A B and d += A2 B, where A2 is a second
// tile with A's orientation and leading dimension (shared address a2). Each B fragment
// is loaded once for both, so the pair costs three quarters of the two calls' ldmatrix.
template <bool kAT, bool kBT, int NT, int kUnroll = 2>
__device__ __forceinline__ void warp_mma_pair(float (&c)[NT][4], float (&d)[NT][4], uint32_t a, uint32_t a2, int lda,
                                              uint32_t b, int ldb, int m0, int n0, int K) {
  static_assert(NT % 2 == 0, "B operands are loaded two n8 tiles at a time");
  const int lane = threadIdx.x & 31;
  uint32_t a_lane, b_lane;
  int a_step, b_step;
  if (!kAT) {
    a_lane = a + 2u * static_cast<uint32_t>((m0 + (lane & 15)) * lda + (lane >> 4) * 8);
    a_step = 32;
  } else {
    a_lane = a + 2u * static_cast<uint32_t>(((lane & 7) + ((lane >> 4) << 3)) * lda + m0 + ((lane >> 3) & 1) * 8);
    a_step = 32 * lda;
  }
  if (kBT) {
    b_lane = b + 2u * static_cast<uint32_t>((n0 + (lane & 7) + ((lane >> 4) << 3)) * ldb + ((lane >> 3) & 1) * 8);
    b_step = 32;
  } else {
    b_lane = b + 2u * static_cast<uint32_t>((lane & 15) * ldb + n0 + (lane >> 4) * 8);
    b_step = 32 * ldb;
  }
  const uint32_t a_other = a2 - a;  // bytes from A's tile to A2's
  const uint32_t b_pair = kBT ? 32u * ldb : 32u;
#pragma unroll kUnroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t af[4], ag[4];
    if (!kAT) {
      ldsm_x4(a_lane, af);
      ldsm_x4(a_lane + a_other, ag);
    } else {
      ldsm_x4_t(a_lane, af);
      ldsm_x4_t(a_lane + a_other, ag);
    }
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) {
      uint32_t bf[4];
      if (kBT) ldsm_x4(b_lane + j * b_pair, bf);
      else ldsm_x4_t(b_lane + j * b_pair, bf);
      mma16816(c[2 * j], af, bf[0], bf[1]);
      mma16816(c[2 * j + 1], af, bf[2], bf[3]);
      mma16816(d[2 * j], ag, bf[0], bf[1]);
      mma16816(d[2 * j + 1], ag, bf[2], bf[3]);
    }
    a_lane += a_step;
    b_lane += b_step;
  }
}

// warp_mma2 for two products that share B: c += A B and d += A2 B over two m16 row tiles.
template <bool kAT, bool kBT, int NT, int kUnroll = 2>
__device__ __forceinline__ void warp_mma2_pair(float (&c)[2][NT][4], float (&d)[2][NT][4], uint32_t a, uint32_t a2,
                                               int lda, uint32_t b, int ldb, int m0, int n0, int K) {
  static_assert(NT % 2 == 0, "B operands are loaded two n8 tiles at a time");
  const int lane = threadIdx.x & 31;
  uint32_t a_lane, b_lane;
  int a_step, b_step;
  uint32_t a_next;
  if (!kAT) {
    a_lane = a + 2u * static_cast<uint32_t>((m0 + (lane & 15)) * lda + (lane >> 4) * 8);
    a_step = 32;
    a_next = 32u * lda;
  } else {
    a_lane = a + 2u * static_cast<uint32_t>(((lane & 7) + ((lane >> 4) << 3)) * lda + m0 + ((lane >> 3) & 1) * 8);
    a_step = 32 * lda;
    a_next = 32u;
  }
  if (kBT) {
    b_lane = b + 2u * static_cast<uint32_t>((n0 + (lane & 7) + ((lane >> 4) << 3)) * ldb + ((lane >> 3) & 1) * 8);
    b_step = 32;
  } else {
    b_lane = b + 2u * static_cast<uint32_t>((lane & 15) * ldb + n0 + (lane >> 4) * 8);
    b_step = 32 * ldb;
  }
  const uint32_t a_other = a2 - a;
  const uint32_t b_pair = kBT ? 32u * ldb : 32u;
#pragma unroll kUnroll
  for (int k0 = 0; k0 < K; k0 += 16) {
    uint32_t af0[4], af1[4], ag0[4], ag1[4];
    if (!kAT) {
      ldsm_x4(a_lane, af0);
      ldsm_x4(a_lane + a_next, af1);
      ldsm_x4(a_lane + a_other, ag0);
      ldsm_x4(a_lane + a_other + a_next, ag1);
    } else {
      ldsm_x4_t(a_lane, af0);
      ldsm_x4_t(a_lane + a_next, af1);
      ldsm_x4_t(a_lane + a_other, ag0);
      ldsm_x4_t(a_lane + a_other + a_next, ag1);
    }
#pragma unroll
    for (int j = 0; j < NT / 2; ++j) {
      uint32_t bf[4];
      if (kBT) ldsm_x4(b_lane + j * b_pair, bf);
      else ldsm_x4_t(b_lane + j * b_pair, bf);
      mma16816(c[0][2 * j], af0, bf[0], bf[1]);
      mma16816(c[0][2 * j + 1], af0, bf[2], bf[3]);
      mma16816(c[1][2 * j], af1, bf[0], bf[1]);
      mma16816(c[1][2 * j + 1], af1, bf[2], bf[3]);
      mma16816(d[0][2 * j], ag0, bf[0], bf[1]);
      mma16816(d[0][2 * j + 1], ag0, bf[2], bf[3]);
      mma16816(d[1][2 * j], ag1, bf[0], bf[1]);
      mma16816(d[1][2 * j + 1], ag1, bf[2], bf[3]);
    }
    a_lane += a_step;
    b_lane += b_step;
  }
}


template <int NT>
__device__ __forceinline__ void zero(float (&c)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.f;
}

template <int NT>
__device__ __forceinline__ void zero(float (&c)[2][NT][4]) {
  zero(c[0]);
  zero(c[1]);
}

// 16-byte global -> shared copy that bypasses the registers; with valid = false
// it writes 16 zero bytes and reads nothing (src must still be a mapped address).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

}  // namespace mm
}  // namespace gdn

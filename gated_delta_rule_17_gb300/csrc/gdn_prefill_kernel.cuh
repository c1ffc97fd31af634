// Fused chunked gated-delta-rule prefill kernel for sm_103a (warp-specialised).
//
// One CTA owns one (sequence, v-head) and walks its 64-token chunks in order.
// It runs the three stages of the GDN prefill op (ssm_gdn_a3.rs, doc comment
// of `gdn_prefill_fla`) on chip, split between two warp groups:
//
//   producer (8 warps), chunk c+1:  WY stage
//     gc = cumsum(g);  L_ij = beta_i e^{gc_i-gc_j} k_i.k_j (j < i);
//     T = (I + L)^{-1};  U = T diag(beta) V;  W = T diag(beta e^gc) K;
//     and the operand tiles the spine needs (e^gc Q / sqrt(dk), e^{gc_last-gc} K,
//     A_ij = e^{gc_i-gc_j} q_i.k_j / sqrt(dk) for j <= i)
//   consumer (4 warps), chunk c:    state spine and output
//     u = U - W S;  S <- e^{gc_last} S + (diag(e^{gc_last-gc}) K)^T u;
//     O = diag(e^gc) Q S / sqrt(dk) + A u          (S: state entering chunk c)
//
// The spine is computed transposed, with the value index v on the 128 tensor
// memory lanes: u^T = U^T - S^T W^T, dS^T = u^T Kd, O^T = S^T Q~^T + u^T A^T.
// Every spine product is then an M=128 tcgen05 MMA whose A operand (S^T or
// u^T, fp16) is read straight from tensor memory, and each consumer thread
// owns one v column, so the output rows are written with coalesced stores.
// The fp32 state S^T lives in tensor memory as the accumulator of dS^T.
//
// Precision: the Gram matrices use the exact bf16 inputs; U and W use bf16 hi+lo
// splits of T diag(beta) and T diag(beta e^gc) against the exact V and K tiles;
// the spine uses fp16 operands with fp32
// accumulation, and A u uses fp16 hi+lo splits of both factors (the largest
// outputs must be accurate to ~1e-4 before the final bf16 rounding).
//
// Tail rows of a chunk (past the end of the sequence) are treated as k = v =
// 0, beta = 0, g = 0 and their outputs are not stored. Every wait on an
// mbarrier is bounded; on expiry the CTA records a status bit and unwinds.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "tc.cuh"

namespace gdn {

constexpr int kDim = 128;   // dk == dv
constexpr int kChunk = 64;  // tokens per chunk
constexpr int kConsumerWarps = 4;
constexpr int kProducerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr uint32_t kBarProducer = 1;  // named barrier ids
constexpr uint32_t kBarConsumer = 2;
constexpr uint32_t kBarCrewX = 3;     // producer crew X (warps 0-3 of the producer)
constexpr int kCrewThreads = kProducerThreads / 2;

// Status bits written to the per-device status word.
constexpr unsigned kStatusBadSeqlens = 1u;
constexpr unsigned kStatusTimeout = 2u;

struct ChunkParams {
  const float* g;
  const float* beta;
  void* state;                // float[B][nv][128][128], or float*[B] when state_is_table
  __nv_bfloat16* out;
  const int32_t* cu_seqlens;  // null for dense batches
  const int32_t* order;       // varlen: sequences by decreasing length (null: identity)
  unsigned* status;
  int64_t g_stride, beta_stride, out_stride;
  int B, T, nk, nv;
  int state_is_table;
};

// Shared-memory plan (bytes from a 1024-aligned base). Operand tiles are
// row-major 16-bit tiles stored as 64-column blocks of 128-byte swizzled rows
// (the layout TMA writes); the same bytes serve as a K-major operand whose
// rows are M/N, or as an MN-major operand whose rows are K.
struct Plan {
  static constexpr int KQ0 = 0;            // raw bf16 [K;Q] (2 blocks x 128 rows), chunk parity 0
  static constexpr int KQ1 = KQ0 + 32768;  // ... chunk parity 1
  static constexpr int VR = KQ1 + 32768;   // raw bf16 V (2 blocks x 64 rows)
  static constexpr int LF = VR + 16384;    // fp32 64 x 64 L, overwritten by T
  static constexpr int LT = LF + 16384;    // fp32 2 x 32 x 32 diagonal blocks of L, transposed (8 KB),
  static constexpr int XP = LT + 4096;     //   whose upper half is reused for 32 x 32 partial products
  static constexpr int TB = XP + 4096;     // bf16 T diag(beta) hi, lo; T diag(beta e^gc) hi, lo
  static constexpr int W16 = TB + 32768;   // fp16 -W^T, rows k (128 x 64)
  static constexpr int QT = W16 + 16384;   // fp16 e^gc Q / sqrt(dk), rows t (64 x 128)
  static constexpr int KD0 = QT + 16384;   // fp16 e^{gc_last-gc} K, rows t, chunk parity 0
  static constexpr int KD1 = KD0 + 16384;  // ... chunk parity 1
  static constexpr int A16 = KD1 + 16384;  // fp16 A hi, lo (64 x 64 each)
  static constexpr int BYTES = A16 + 16384;
  static constexpr int DYN_SMEM = BYTES + 1024;  // slack for 1024-byte alignment
  static_assert(DYN_SMEM <= 227 * 1024 - 4096, "shared memory budget");
  static_assert(TB % 1024 == 0 && W16 % 1024 == 0 && KD0 % 1024 == 0 && A16 % 1024 == 0, "tile alignment");

  // Tensor-memory columns (512 x 32-bit, lanes = rows).
  static constexpr uint32_t COL_S = 0;     // fp32 S^T [v][k], 128 columns
  static constexpr uint32_t COL_U = 128;   // fp32 U^T -> u^T [v][t], 2 x 64 columns (chunk parity)
  static constexpr uint32_t COL_GW = 256;  // fp32 [K;Q] K^T [m][j], then W^T [k][t], 64 columns
  static constexpr uint32_t COL_O = 320;   // fp32 O^T [v][t], 64 columns
  static constexpr uint32_t COL_ST = 384;  // fp16 pairs S^T [v][k], 64 columns
  static constexpr uint32_t COL_UT = 448;  // fp16 pairs u^T hi [v][t] (32 columns), then lo (32)
  static constexpr uint32_t TMEM_COLS = 512;
};

// fp32 64 x 64 work matrix with 16-byte chunks XOR-swizzled by row, so that
// float4 accesses by threads on different rows hit different banks.
__device__ __forceinline__ int lf_idx(int r, int c) {
  return r * 64 + ((((c >> 2) ^ r) & 15) << 2) + (c & 3);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 raw, float (&f)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack_half8(const float (&f)[8], float s) {
  return make_uint4(pack_half2(f[0] * s, f[1] * s), pack_half2(f[2] * s, f[3] * s),
                    pack_half2(f[4] * s, f[5] * s), pack_half2(f[6] * s, f[7] * s));
}

__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// (a, b) = hi + lo with hi = fp16(x), lo = fp16(x - hi): about 22 significant bits.
__device__ __forceinline__ void split_half2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 x = __floats2half2_rn(a, b);
  const float2 xf = __half22float2(x);
  const __half2 y = __floats2half2_rn(a - xf.x, b - xf.y);
  hi = *reinterpret_cast<const uint32_t*>(&x);
  lo = *reinterpret_cast<const uint32_t*>(&y);
}

// (a, b) = hi + lo with hi = bf16(x), lo = bf16(x - hi): about 16 significant bits.
__device__ __forceinline__ void split_bf162(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 x = __floats2bfloat162_rn(a, b);
  const float2 xf = __bfloat1622float2(x);
  const __nv_bfloat162 y = __floats2bfloat162_rn(a - xf.x, b - xf.y);
  hi = *reinterpret_cast<const uint32_t*>(&x);
  lo = *reinterpret_cast<const uint32_t*>(&y);
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr float kInvSqrtD = 0.08838834764831845f;  // 1 / sqrt(128)

// Per-CTA state shared by the two warp groups.
struct Ctx {
  uint8_t* sm;       // 1024-aligned dynamic shared memory
  uint32_t sbase;    // its shared-window address
  uint32_t tmem;     // tensor-memory base address
  int64_t row0, len; // first packed row and length of the sequence
  int nchunks, h, kh;
  float* state;      // this (sequence, head)'s fp32 [128][128] state, k-major
  // producer-side per-token scales of the current chunk
  float *s_gc, *s_eg, *s_edec, *s_ebg, *s_beta;
  float *s_E, *s_F;     // e^{gc - m}, e^{m - gc} about the chunk's mid gate m
  int* s_fast;          // 1 when the chunk's gate range allows the factorised decays
  float* s_gstage;      // [2][2][64] g and beta of the next chunk, staged by cp.async
  uint16_t* s_ostage;   // [4 warps][8][32] bf16 output staging of the consumer
  float* s_elast;    // [2] e^{gc_last} by chunk parity (read by the consumer)
  volatile int* s_abort;
  uint32_t mb_kq0, mb_kq1, mb_v, mb_g, mb_uw, mb_c1, mb_c2, mb_hand, mb_cu;
};

// All threads of a group wait on one mbarrier phase; the outcome is made
// uniform across the group so that it can leave its loop together.
__device__ __forceinline__ bool group_wait(const Ctx& x, const ChunkParams& p, uint32_t mbar, uint32_t parity,
                                           uint32_t bar_id, uint32_t nthreads, bool leader) {
  bool ok = (*x.s_abort == 0) && tc::mbar_wait_timed(mbar, parity, kWaitLimitNs);
  ok = tc::barrier_all(bar_id, nthreads, ok);
  if (!ok) {
    if (leader) {
      *x.s_abort = 1;
      atomicOr(p.status, kStatusTimeout);
    }
    return false;
  }
  tc::fence_after_sync();
  return true;
}

// ---------------------------------------------------------------------------------
// Producer: the WY stage of each chunk, one chunk ahead of the consumer.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void producer_role(const Ctx& x, const ChunkParams& p, const CUtensorMap* tmap_q,
                                              const CUtensorMap* tmap_k, const CUtensorMap* tmap_v, int ptid) {
  using P = Plan;
  const int pw = ptid >> 5, lane = ptid & 31;
  const int quad = pw & 3;   // tensor-memory lane quarter of this warp
  const int half = pw >> 2;  // which half of a 64-column accumulator it reads
  const bool leader = ptid == 0;
  const bool crew_x = pw < 4;                  // crews X and Y each hold one warp per sub-partition
  const int cx = (pw & 3) * 32 + lane;         // thread index within its crew
  const int cy = cx;
  uint8_t* sm = x.sm;
  float* lf = reinterpret_cast<float*>(sm + P::LF);
  float* lt = reinterpret_cast<float*>(sm + P::LT);
  float* xp = reinterpret_cast<float*>(sm + P::XP);

  auto issue_kq = [&](int c) {
    const uint32_t dst = x.sbase + ((c & 1) ? P::KQ1 : P::KQ0);
    const uint32_t mb = (c & 1) ? x.mb_kq1 : x.mb_kq0;
    const int32_t y = static_cast<int32_t>(x.row0 + static_cast<int64_t>(c) * kChunk);
    tc::mbar_arrive_expect_tx(mb, 32768);
    tc::tma_load_2d(dst, tmap_k, x.kh * kDim, y, mb);
    tc::tma_load_2d(dst + 16384, tmap_k, x.kh * kDim + 64, y, mb);
    tc::tma_load_2d(dst + 8192, tmap_q, x.kh * kDim, y, mb);
    tc::tma_load_2d(dst + 16384 + 8192, tmap_q, x.kh * kDim + 64, y, mb);
  };
  auto issue_v = [&](int c) {
    const int32_t y = static_cast<int32_t>(x.row0 + static_cast<int64_t>(c) * kChunk);
    tc::mbar_arrive_expect_tx(x.mb_v, 16384);
    tc::tma_load_2d(x.sbase + P::VR, tmap_v, x.h * kDim, y, x.mb_v);
    tc::tma_load_2d(x.sbase + P::VR + 8192, tmap_v, x.h * kDim + 64, y, x.mb_v);
  };
  // gates of tokens 2*lane and 2*lane+1 of chunk c, copied to shared memory
  // (stage c & 1) without a register round trip (producer warp 0 only)
  auto load_gates = [&](int c) {
    float* st = x.s_gstage + (c & 1) * 128;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tt = 2 * lane + e;
      const int64_t t = static_cast<int64_t>(c) * kChunk + tt;
      if (t < x.len) {
        const int64_t r = x.row0 + t;
        tc::cp_async_4(tc::smem_u32(st + tt), p.g + r * p.g_stride + x.h);
        tc::cp_async_4(tc::smem_u32(st + 64 + tt), p.beta + r * p.beta_stride + x.h);
      } else {
        st[tt] = 0.f;
        st[64 + tt] = 0.f;
      }
    }
    tc::cp_async_commit();
  };

  if (leader) {
    issue_kq(0);
    issue_v(0);
    if (x.nchunks > 1) issue_kq(1);
  }
  if (pw == 4) {  // crew Y stages the gates; the join barrier publishes them
    load_gates(0);
    tc::cp_async_wait_all();
  }
  tc::named_barrier(kBarProducer, kProducerThreads);

  for (int c = 0; c < x.nchunks; ++c) {
    const int b = c & 1;
    const int64_t rem = x.len - static_cast<int64_t>(c) * kChunk;
    const int clen = rem < kChunk ? static_cast<int>(rem) : kChunk;
    const uint32_t kq_off = b ? P::KQ1 : P::KQ0;
    const uint32_t kd_off = b ? P::KD1 : P::KD0;

    // ---- gates: in-chunk cumulative log-gate and the per-token scales ----------------
    if (pw == 0) {
      const float* st = x.s_gstage + b * 128;
      const float g0 = st[2 * lane], g1 = st[2 * lane + 1];
      const float b0 = st[64 + 2 * lane], b1 = st[64 + 2 * lane + 1];
      const float pair = g0 + g1;
      float incl = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const float gca = incl - pair + g0, gcb = incl;
      const float glast = __shfl_sync(0xffffffffu, incl, 31);
      const float gfirst = __shfl_sync(0xffffffffu, gca, 0);
      // e^{gc_i - gc_j} = e^{gc_i - m} e^{m - gc_j} with m the middle of the chunk's
      // gate range; both factors stay within e^{+-60} when the range is <= 120.
      const float mid = 0.5f * (gfirst + glast);
      const float ea = __expf(gca), eb = __expf(gcb);
      x.s_gc[2 * lane] = gca;
      x.s_gc[2 * lane + 1] = gcb;
      x.s_eg[2 * lane] = ea;
      x.s_eg[2 * lane + 1] = eb;
      x.s_edec[2 * lane] = __expf(glast - gca);
      x.s_edec[2 * lane + 1] = __expf(glast - gcb);
      x.s_ebg[2 * lane] = b0 * ea;
      x.s_ebg[2 * lane + 1] = b1 * eb;
      x.s_beta[2 * lane] = b0;
      x.s_beta[2 * lane + 1] = b1;
      x.s_E[2 * lane] = __expf(gca - mid);
      x.s_E[2 * lane + 1] = __expf(gcb - mid);
      x.s_F[2 * lane] = __expf(mid - gca);
      x.s_F[2 * lane + 1] = __expf(mid - gcb);
      if (lane == 0) {
        x.s_elast[b] = __expf(glast);
        *x.s_fast = (gfirst - glast) <= 120.f;
      }
    }

    // ---- Gram matrices [K;Q] K^T (bf16, M=128, N=64, K=128) ----------------------------
    if (!group_wait(x, p, b ? x.mb_kq1 : x.mb_kq0, (c >> 1) & 1, kBarProducer, kProducerThreads, leader)) break;
    if (leader) {
      constexpr uint32_t idesc = tc::idesc_f16(128, 64, tc::kBF16, false, false);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const uint32_t a = x.sbase + kq_off + (st >> 2) * 16384 + (st & 3) * 32;
        tc::mma_f16(x.tmem + P::COL_GW, tc::desc_sw128(a, 16, 1024), tc::desc_sw128(a, 16, 1024), idesc, st > 0);
      }
      tc::mma_commit(x.mb_g);
    }

    // ---- L (fp32) from K K^T (lanes 0-63) and A (fp16 hi + lo) from Q K^T (lanes 64-127) --
    bool ok = (*x.s_abort == 0) && tc::mbar_wait_timed(x.mb_g, b, kWaitLimitNs);
    if (quad >= 2 && c > 0)  // A is rewritten only after the spine of chunk c-1 used it
      ok = ok && (*x.s_abort == 0) && tc::mbar_wait_timed(x.mb_c2, (c - 1) & 1, kWaitLimitNs);
    tc::fence_after_sync();
    {
      uint32_t d[32];
      tc::tmem_ld32(x.tmem + ((quad * 32u) << 16) + P::COL_GW + half * 32, d);
      tc::tmem_ld_wait();
      const bool fast = *x.s_fast != 0;
      if (quad < 2) {  // L_tj = beta_t e^{gc_t - gc_j} k_t.k_j for j < t
        const int t = quad * 32 + lane;
        const bool live = t < clen;
        float l[32];
        if (fast) {
          const float be = x.s_beta[t] * x.s_E[t];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = half * 32 + e;
            l[e] = (j < t && live) ? be * x.s_F[j] * __uint_as_float(d[e]) : 0.f;
          }
        } else {
          const float gt = x.s_gc[t], bt = x.s_beta[t];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = half * 32 + e;
            l[e] = (j < t && live) ? bt * __expf(gt - x.s_gc[j]) * __uint_as_float(d[e]) : 0.f;
          }
        }
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4)
          *reinterpret_cast<float4*>(lf + lf_idx(t, half * 32 + j4 * 4)) =
              make_float4(l[4 * j4], l[4 * j4 + 1], l[4 * j4 + 2], l[4 * j4 + 3]);
        // the diagonal 32 x 32 block of L, transposed, for the inverse's first phase
        if (quad == half) {
          float* dst = lt + quad * 1024 + lane;
#pragma unroll
          for (int m = 0; m < 32; ++m) dst[m * 32] = l[m];
        }
      } else if (ok) {  // A_ij = e^{gc_i - gc_j} q_i.k_j / sqrt(dk) for j <= i
        const int i = (quad - 2) * 32 + lane;
        float a[32];
        if (fast) {
          const float ei = x.s_E[i] * kInvSqrtD;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = half * 32 + e;
            a[e] = (j <= i) ? ei * x.s_F[j] * __uint_as_float(d[e]) : 0.f;
          }
        } else {
          const float gi = x.s_gc[i];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = half * 32 + e;
            a[e] = (j <= i) ? __expf(gi - x.s_gc[j]) * kInvSqrtD * __uint_as_float(d[e]) : 0.f;
          }
        }
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_half2(a[j8 * 8 + 2 * e], a[j8 * 8 + 2 * e + 1], hi[e], lo[e]);
          const uint32_t o = tc::sw128(i, (half * 32 + j8 * 8) * 2);
          *reinterpret_cast<uint4*>(sm + P::A16 + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(sm + P::A16 + 8192 + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    }
    tc::fence_before_sync();
    if (!tc::barrier_all(kBarProducer, kProducerThreads, ok && *x.s_abort == 0)) {
      if (leader) {
        *x.s_abort = 1;
        atomicOr(p.status, kStatusTimeout);
      }
      break;
    }

    // Crew X (producer warps 0-3, one per SM sub-partition) inverts L while crew Y
    // (warps 4-7) builds the Kd and Q~ tiles and prefetches the next chunk's gates.
    if (crew_x) {
      // ---- T = (I + L)^{-1} in fp32, in place over L -------------------------------------
      // (a) the two diagonal 32 x 32 blocks: one column per thread, right-looking
      //     substitution; column m of the block comes from the transposed copy as
      //     broadcast loads.
      if (pw < 2) {
        const int r0 = 32 * pw;
        const float* ltb = lt + pw * 1024;
        float xv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) xv[i] = (i == lane) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < 31; ++m) {
          float lc[32];
#pragma unroll
          for (int i4 = (m + 1) >> 2; i4 < 8; ++i4) {
            const float4 v4 = *reinterpret_cast<const float4*>(ltb + m * 32 + 4 * i4);
            lc[4 * i4] = v4.x;
            lc[4 * i4 + 1] = v4.y;
            lc[4 * i4 + 2] = v4.z;
            lc[4 * i4 + 3] = v4.w;
          }
          const float xm = xv[m];
#pragma unroll
          for (int i = m + 1; i < 32; ++i) xv[i] = fmaf(-lc[i], xm, xv[i]);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) lf[lf_idx(r0 + i, r0 + lane)] = xv[i];
      }
      tc::named_barrier(kBarCrewX, kCrewThreads);
      // (b) lower-left 32 x 32: X = L[32:64, 0:32] T[0:32, 0:32];
      //     T[32:64, 0:32] = -T[32:64, 32:64] X   (2 x 4 outputs per thread, 4 warps)
      {
        const int r0 = (cx >> 3) * 2, c0 = (cx & 7) * 4;
        float la[32], lb[32];
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 va = *reinterpret_cast<const float4*>(lf + lf_idx(32 + r0, 4 * i4));
          const float4 vb = *reinterpret_cast<const float4*>(lf + lf_idx(33 + r0, 4 * i4));
          la[4 * i4] = va.x; la[4 * i4 + 1] = va.y; la[4 * i4 + 2] = va.z; la[4 * i4 + 3] = va.w;
          lb[4 * i4] = vb.x; lb[4 * i4 + 1] = vb.y; lb[4 * i4 + 2] = vb.z; lb[4 * i4 + 3] = vb.w;
        }
        float4 xa = make_float4(0.f, 0.f, 0.f, 0.f), xb = xa;
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          const float4 tv = *reinterpret_cast<const float4*>(lf + lf_idx(m, c0));
          xa.x = fmaf(la[m], tv.x, xa.x); xa.y = fmaf(la[m], tv.y, xa.y);
          xa.z = fmaf(la[m], tv.z, xa.z); xa.w = fmaf(la[m], tv.w, xa.w);
          xb.x = fmaf(lb[m], tv.x, xb.x); xb.y = fmaf(lb[m], tv.y, xb.y);
          xb.z = fmaf(lb[m], tv.z, xb.z); xb.w = fmaf(lb[m], tv.w, xb.w);
        }
        *reinterpret_cast<float4*>(xp + r0 * 32 + c0) = xa;
        *reinterpret_cast<float4*>(xp + (r0 + 1) * 32 + c0) = xb;
      }
      tc::named_barrier(kBarCrewX, kCrewThreads);
      {
        const int r0 = (cx >> 3) * 2, c0 = (cx & 7) * 4;
        float ta[32], tb[32];
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 va = *reinterpret_cast<const float4*>(lf + lf_idx(32 + r0, 32 + 4 * i4));
          const float4 vb = *reinterpret_cast<const float4*>(lf + lf_idx(33 + r0, 32 + 4 * i4));
          ta[4 * i4] = va.x; ta[4 * i4 + 1] = va.y; ta[4 * i4 + 2] = va.z; ta[4 * i4 + 3] = va.w;
          tb[4 * i4] = vb.x; tb[4 * i4 + 1] = vb.y; tb[4 * i4 + 2] = vb.z; tb[4 * i4 + 3] = vb.w;
        }
        float4 ya = make_float4(0.f, 0.f, 0.f, 0.f), yb = ya;
#pragma unroll
        for (int m = 0; m < 32; ++m) {
          const float4 xv = *reinterpret_cast<const float4*>(xp + m * 32 + c0);
          ya.x = fmaf(ta[m], xv.x, ya.x); ya.y = fmaf(ta[m], xv.y, ya.y);
          ya.z = fmaf(ta[m], xv.z, ya.z); ya.w = fmaf(ta[m], xv.w, ya.w);
          yb.x = fmaf(tb[m], xv.x, yb.x); yb.y = fmaf(tb[m], xv.y, yb.y);
          yb.z = fmaf(tb[m], xv.z, yb.z); yb.w = fmaf(tb[m], xv.w, yb.w);
        }
        *reinterpret_cast<float4*>(lf + lf_idx(32 + r0, c0)) = make_float4(-ya.x, -ya.y, -ya.z, -ya.w);
        *reinterpret_cast<float4*>(lf + lf_idx(33 + r0, c0)) = make_float4(-yb.x, -yb.y, -yb.z, -yb.w);
      }
      tc::named_barrier(kBarCrewX, kCrewThreads);
    } else {
      // ---- Kd = e^{gc_last-gc} K (fp16, rows t) for the consumer's state update ------
      // KD[b] was last read by the state update of chunk c-2, which finished before
      // this group handed over chunk c-1.
      {
        uint4 raw[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int it = cy + r * kCrewThreads, t = it & 63, cc = it >> 6;
          raw[r] = *reinterpret_cast<const uint4*>(sm + kq_off + (cc >> 3) * 16384 + tc::sw128(t, (cc & 7) * 16));
        }
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int it = cy + r * kCrewThreads, t = it & 63, cc = it >> 6;
          float f[8];
          unpack_bf16x8(raw[r], f);
          *reinterpret_cast<uint4*>(sm + kd_off + (cc >> 3) * 8192 + tc::sw128(t, (cc & 7) * 16)) =
              t < clen ? pack_half8(f, x.s_edec[t]) : make_uint4(0, 0, 0, 0);
        }
      }
      if (pw == 4 && c + 1 < x.nchunks) load_gates(c + 1);
      // ---- Q~ = e^gc Q / sqrt(dk) (fp16, rows t), once the spine of chunk c-1 read Q~ --
      if (c > 0) ok = (*x.s_abort == 0) && tc::mbar_wait_timed(x.mb_c1, (c - 1) & 1, kWaitLimitNs);
      {
        uint4 raw[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int it = cy + r * kCrewThreads, t = it & 63, cc = it >> 6;
          raw[r] = *reinterpret_cast<const uint4*>(sm + kq_off + (cc >> 3) * 16384 + 8192 + tc::sw128(t, (cc & 7) * 16));
        }
        if (ok) {
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const int it = cy + r * kCrewThreads, t = it & 63, cc = it >> 6;
            float f[8];
            unpack_bf16x8(raw[r], f);
            *reinterpret_cast<uint4*>(sm + P::QT + (cc >> 3) * 8192 + tc::sw128(t, (cc & 7) * 16)) =
                t < clen ? pack_half8(f, x.s_eg[t] * kInvSqrtD) : make_uint4(0, 0, 0, 0);
          }
        }
      }
      if (pw == 4) tc::cp_async_wait_all();
    }
    if (!tc::barrier_all(kBarProducer, kProducerThreads, ok && *x.s_abort == 0)) {
      if (leader) {
        *x.s_abort = 1;
        atomicOr(p.status, kStatusTimeout);
      }
      break;
    }

    // ---- bf16 hi/lo tiles of T diag(beta) and T diag(beta e^gc) (rows t, columns j) -----
    {
      const int t = ptid >> 2, j0 = (ptid & 3) * 16;
#pragma unroll
      for (int h8 = 0; h8 < 2; ++h8) {
        const int jb = j0 + h8 * 8;
        const float4 ta = *reinterpret_cast<const float4*>(lf + lf_idx(t, jb));
        const float4 tb = *reinterpret_cast<const float4*>(lf + lf_idx(t, jb + 4));
        const float4 ba = *reinterpret_cast<const float4*>(x.s_beta + jb);
        const float4 bb4 = *reinterpret_cast<const float4*>(x.s_beta + jb + 4);
        const float4 ea = *reinterpret_cast<const float4*>(x.s_ebg + jb);
        const float4 eb4 = *reinterpret_cast<const float4*>(x.s_ebg + jb + 4);
        const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
        const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb4.x, bb4.y, bb4.z, bb4.w};
        const float ev[8] = {ea.x, ea.y, ea.z, ea.w, eb4.x, eb4.y, eb4.z, eb4.w};
        uint32_t bh[4], bl[4], wh[4], wl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          split_bf162(tv[2 * e] * bv[2 * e], tv[2 * e + 1] * bv[2 * e + 1], bh[e], bl[e]);
          split_bf162(tv[2 * e] * ev[2 * e], tv[2 * e + 1] * ev[2 * e + 1], wh[e], wl[e]);
        }
        const uint32_t o = tc::sw128(t, jb * 2);
        *reinterpret_cast<uint4*>(sm + P::TB + o) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
        *reinterpret_cast<uint4*>(sm + P::TB + 8192 + o) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
        *reinterpret_cast<uint4*>(sm + P::TB + 16384 + o) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4*>(sm + P::TB + 24576 + o) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
    }
    tc::fence_proxy_async();

    // ---- U^T = V^T (T diag beta)^T and W^T = K^T (T diag(beta e^gc))^T, hi + lo each ----
    // U^T goes to the chunk-parity half of the U columns, free once the consumer has
    // read u of chunk c-2 (it signals every chunk; waiting for chunk c-1 covers it).
    if (!group_wait(x, p, x.mb_v, b, kBarProducer, kProducerThreads, leader)) break;  // V tile of chunk c
    if (c >= 2 && !group_wait(x, p, x.mb_cu, (c - 1) & 1, kBarProducer, kProducerThreads, leader)) break;
    if (leader) {
      tc::fence_after_sync();
      constexpr uint32_t id = tc::idesc_f16(128, 64, tc::kBF16, true, false);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int st = 0; st < 4; ++st)
          tc::mma_f16(x.tmem + P::COL_U + 64 * b, tc::desc_sw128(x.sbase + P::VR + st * 2048, 8192, 1024),
                      tc::desc_sw128(x.sbase + P::TB + part * 8192 + st * 32, 16, 1024), id, part + st > 0);
      }
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int st = 0; st < 4; ++st)
          tc::mma_f16(x.tmem + P::COL_GW, tc::desc_sw128(x.sbase + kq_off + st * 2048, 16384, 1024),
                      tc::desc_sw128(x.sbase + P::TB + 16384 + part * 8192 + st * 32, 16, 1024), id, part + st > 0);
      }
      tc::mma_commit(x.mb_uw);
    }
    if (!group_wait(x, p, x.mb_uw, b, kBarProducer, kProducerThreads, leader)) break;
    if (leader) {  // this chunk's raw tiles are consumed: prefetch ahead
      if (c + 1 < x.nchunks) issue_v(c + 1);
      if (c + 2 < x.nchunks) issue_kq(c + 2);
    }

    // ---- -W^T as the spine's fp16 B operand (rows k, columns t) -----------------------
    {
      uint32_t d[32];
      tc::tmem_ld32(x.tmem + ((quad * 32u) << 16) + P::COL_GW + half * 32, d);
      tc::tmem_ld_wait();
      const int k = quad * 32 + lane;
#pragma unroll
      for (int j8 = 0; j8 < 4; ++j8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w[e] = pack_half2(-__uint_as_float(d[j8 * 8 + 2 * e]), -__uint_as_float(d[j8 * 8 + 2 * e + 1]));
        *reinterpret_cast<uint4*>(sm + P::W16 + tc::sw128(k, (half * 32 + j8 * 8) * 2)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    tc::named_barrier(kBarProducer, kProducerThreads);
    if (leader) tc::mbar_arrive(x.mb_hand);  // chunk c's operands are ready
  }
}

// ---------------------------------------------------------------------------------
// Consumer: the state spine and the output of each chunk. Thread v owns value
// column v: tensor-memory lane v holds S^T[v][:], u^T[v][:] and O^T[v][:].
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void consumer_role(const Ctx& x, const ChunkParams& p, int ctid) {
  using P = Plan;
  const int quad = ctid >> 5;
  const int v = ctid;
  const bool leader = ctid == 0;
  const uint32_t lanes = x.tmem + ((quad * 32u) << 16);

  // carried-in state: fp32 S^T into tensor memory, plus its fp16 operand copy
  {
    uint32_t s[32], st[32];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
      for (int e = 0; e < 32; ++e) s[e] = __float_as_uint(x.state[(q4 * 32 + e) * kDim + v]);
      tc::tmem_st32(lanes + P::COL_S + q4 * 32, s);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        st[(q4 & 1) * 16 + e] = pack_half2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1]));
      if (q4 & 1) tc::tmem_st32(lanes + P::COL_ST + (q4 >> 1) * 32, st);
    }
    tc::tmem_st_wait();
  }
  tc::fence_before_sync();
  tc::named_barrier(kBarConsumer, kConsumerThreads);

  for (int c = 0; c < x.nchunks; ++c) {
    const int b = c & 1;
    const int64_t rem = x.len - static_cast<int64_t>(c) * kChunk;
    const int clen = rem < kChunk ? static_cast<int>(rem) : kChunk;
    const uint32_t kd_off = b ? P::KD1 : P::KD0;
    const uint32_t col_u = P::COL_U + 64 * b;

    if (!group_wait(x, p, x.mb_hand, b, kBarConsumer, kConsumerThreads, leader)) break;
    // ---- u^T = U^T - S^T W^T (accumulated onto U^T) and O^T = S^T Q~^T -------------------
    if (leader) {
      constexpr uint32_t id_u = tc::idesc_f16(128, 64, tc::kF16, false, true);
      constexpr uint32_t id_o = tc::idesc_f16(128, 64, tc::kF16, false, false);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const uint32_t a = x.tmem + P::COL_ST + st * 8;
        tc::mma_f16_ts(x.tmem + col_u, a, tc::desc_sw128(x.sbase + P::W16 + st * 2048, 16384, 1024), id_u, 1);
        tc::mma_f16_ts(x.tmem + P::COL_O, a,
                       tc::desc_sw128(x.sbase + P::QT + (st >> 2) * 8192 + (st & 3) * 32, 16, 1024), id_o, st > 0);
      }
      tc::mma_commit(x.mb_c1);
    }
    // meanwhile: S^T <- e^{gc_last} S^T, the decay half of the state update
    {
      const float el = x.s_elast[b];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t s[32];
        tc::tmem_ld32(lanes + P::COL_S + q4 * 32, s);
        tc::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) s[e] = __float_as_uint(el * __uint_as_float(s[e]));
        tc::tmem_st32(lanes + P::COL_S + q4 * 32, s);
      }
      tc::tmem_st_wait();
    }
    if (!group_wait(x, p, x.mb_c1, b, kBarConsumer, kConsumerThreads, leader)) break;

    // ---- u^T as an fp16 hi + lo pair in tensor memory (the A operand of the next MMAs) ---
    {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t u[32], hi[16], lo[16];
        tc::tmem_ld32(lanes + col_u + h2 * 32, u);
        tc::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e)
          split_half2(__uint_as_float(u[2 * e]), __uint_as_float(u[2 * e + 1]), hi[e], lo[e]);
        tc::tmem_st16u(lanes + P::COL_UT + h2 * 16, hi);
        tc::tmem_st16u(lanes + P::COL_UT + 32 + h2 * 16, lo);
      }
      tc::tmem_st_wait();
    }
    tc::fence_before_sync();
    tc::named_barrier(kBarConsumer, kConsumerThreads);
    // ---- S^T += u^T Kd (the write half of the update) and O^T += u^T A^T (hi/lo x3) -------
    if (leader) {
      tc::fence_after_sync();
      tc::mbar_arrive(x.mb_cu);  // the U columns of this chunk parity are free again
      constexpr uint32_t id_s = tc::idesc_f16(128, 128, tc::kF16, false, true);
      constexpr uint32_t id_o = tc::idesc_f16(128, 64, tc::kF16, false, false);
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint32_t u_hi = x.tmem + P::COL_UT + st * 8, u_lo = x.tmem + P::COL_UT + 32 + st * 8;
        const uint64_t a_hi = tc::desc_sw128(x.sbase + P::A16 + st * 32, 16, 1024);
        const uint64_t a_lo = tc::desc_sw128(x.sbase + P::A16 + 8192 + st * 32, 16, 1024);
        tc::mma_f16_ts(x.tmem + P::COL_S, u_hi, tc::desc_sw128(x.sbase + kd_off + st * 2048, 8192, 1024), id_s, 1);
        tc::mma_f16_ts(x.tmem + P::COL_O, u_hi, a_hi, id_o, 1);
        tc::mma_f16_ts(x.tmem + P::COL_O, u_hi, a_lo, id_o, 1);
        tc::mma_f16_ts(x.tmem + P::COL_O, u_lo, a_hi, id_o, 1);
      }
      tc::mma_commit(x.mb_c2);
    }
    if (!group_wait(x, p, x.mb_c2, b, kBarConsumer, kConsumerThreads, leader)) break;

    // ---- next chunk's fp16 S^T operand, and this chunk's output rows -------------------
    {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t s[32], st[16];
        tc::tmem_ld32(lanes + P::COL_S + q4 * 32, s);
        tc::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) st[e] = pack_half2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1]));
        tc::tmem_st16u(lanes + P::COL_ST + q4 * 16, st);
      }
      // O^T holds one value column per thread; an 8-row x 32-column staging tile per
      // warp turns it into 16-byte row segments for coalesced global stores.
      uint16_t* stg = x.s_ostage + quad * 256;
      const int lane = ctid & 31;
      __nv_bfloat16* orow = p.out + (x.row0 + static_cast<int64_t>(c) * kChunk) * p.out_stride +
                            static_cast<int64_t>(x.h) * kDim + quad * 32 + (lane & 3) * 8;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t o[32];
        tc::tmem_ld32(lanes + P::COL_O + h2 * 32, o);
        tc::tmem_ld_wait();
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const __nv_bfloat16 bv = __float2bfloat16_rn(__uint_as_float(o[blk * 8 + r]));
            stg[r * 32 + lane] = *reinterpret_cast<const uint16_t*>(&bv);
          }
          __syncwarp();
          const uint4 w = *reinterpret_cast<const uint4*>(stg + (lane >> 2) * 32 + (lane & 3) * 8);
          const int t = h2 * 32 + blk * 8 + (lane >> 2);
          if (t < clen) *reinterpret_cast<uint4*>(orow + static_cast<int64_t>(t) * p.out_stride) = w;
          __syncwarp();
        }
      }
      tc::tmem_st_wait();
    }
    tc::fence_before_sync();
  }

  if (*x.s_abort == 0) {  // carried-out state S_T, k-major
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint32_t s[32];
      tc::tmem_ld32(lanes + P::COL_S + q4 * 32, s);
      tc::tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) x.state[(q4 * 32 + e) * kDim + v] = __uint_as_float(s[e]);
    }
  }
}

template <int kUnused = 0>
__global__ void __launch_bounds__(kThreads, 1)
gdn_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const ChunkParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(16) float s_gc[kChunk], s_eg[kChunk], s_edec[kChunk], s_ebg[kChunk], s_beta[kChunk];
  __shared__ __align__(16) float s_E[kChunk], s_F[kChunk], s_gstage[2 * 2 * kChunk];
  __shared__ float s_elast[2];
  __shared__ int s_fast;
  __shared__ __align__(16) uint16_t s_ostage[kConsumerWarps * 256];
  __shared__ __align__(8) uint64_t s_mb[9];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5;

  // ---- which (sequence, head) this CTA owns -------------------------------------------
  Ctx x;
  x.h = blockIdx.x % p.nv;
  const int slot = blockIdx.x / p.nv;
  const int s = p.order ? p.order[slot] : slot;
  x.kh = x.h / (p.nv / p.nk);
  if (p.cu_seqlens) {
    if (s < 0 || s >= p.B) {
      if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
    const int a = p.cu_seqlens[s], e = p.cu_seqlens[s + 1];
    if (a < 0 || e < a || e > p.T) {
      if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
    x.row0 = a;
    x.len = e - a;
  } else {
    x.row0 = static_cast<int64_t>(s) * p.T;
    x.len = p.T;
  }
  x.nchunks = static_cast<int>((x.len + kChunk - 1) / kChunk);
  if (x.nchunks == 0) return;  // empty sequence: the state passes through unchanged
  float* state = p.state_is_table ? reinterpret_cast<float* const*>(p.state)[s]
                                  : reinterpret_cast<float*>(p.state) + static_cast<int64_t>(s) * p.nv * kDim * kDim;
  x.state = state + static_cast<int64_t>(x.h) * kDim * kDim;
  x.sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  x.sbase = tc::smem_u32(x.sm);
  x.s_gc = s_gc;
  x.s_eg = s_eg;
  x.s_edec = s_edec;
  x.s_ebg = s_ebg;
  x.s_beta = s_beta;
  x.s_elast = s_elast;
  x.s_E = s_E;
  x.s_F = s_F;
  x.s_fast = &s_fast;
  x.s_gstage = s_gstage;
  x.s_ostage = s_ostage;
  x.s_abort = &s_abort;
  x.mb_kq0 = tc::smem_u32(&s_mb[0]);
  x.mb_kq1 = tc::smem_u32(&s_mb[1]);
  x.mb_v = tc::smem_u32(&s_mb[2]);
  x.mb_g = tc::smem_u32(&s_mb[3]);
  x.mb_uw = tc::smem_u32(&s_mb[4]);
  x.mb_c1 = tc::smem_u32(&s_mb[5]);
  x.mb_c2 = tc::smem_u32(&s_mb[6]);
  x.mb_hand = tc::smem_u32(&s_mb[7]);
  x.mb_cu = tc::smem_u32(&s_mb[8]);

  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&s_tmem), Plan::TMEM_COLS);
  if (tid == 0) {
    s_abort = 0;
#pragma unroll
    for (int i = 0; i < 9; ++i) tc::mbar_init(tc::smem_u32(&s_mb[i]), 1);
    tc::mbar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  x.tmem = s_tmem;

  if (warp < kConsumerWarps)
    consumer_role(x, p, tid);
  else
    producer_role(x, p, &tmap_q, &tmap_k, &tmap_v, tid - kConsumerThreads);

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    if (s_abort) {  // a wait expired: give any copy or MMA still in flight time to land
      const uint64_t t0 = tc::globaltimer_ns();
      while (tc::globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
    }
    tc::fence_after_sync();
    tc::tmem_dealloc(x.tmem, Plan::TMEM_COLS);
  }
}

}  // namespace gdn

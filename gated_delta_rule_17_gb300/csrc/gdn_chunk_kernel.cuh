// Fused chunked gated-delta-rule prefill kernel for sm_103a.
//
// One CTA owns one (sequence, v-head, v-column slice of NS columns) and walks
// the sequence's 64-token chunks in order, keeping its NS columns of the
// fp32 128 x 128 state in registers. Per chunk it runs the three stages of
// the GDN prefill op (ssm_gdn_a3.rs, doc comment of `gdn_prefill_fla`):
//
//   WY stage   gc = cumsum(g); L_ij = beta_i e^{gc_i-gc_j} k_i.k_j (j < i);
//              T = (I + L)^{-1}; U = T diag(beta) V; W = T diag(beta e^{gc}) K
//   spine      u = U - W S;  S <- e^{gc_last} S + (diag(e^{gc_last-gc}) K)^T u
//   output     O = diag(e^{gc}) Q S / sqrt(dk) + A u,
//              A_ij = e^{gc_i-gc_j} q_i.k_j / sqrt(dk) for j <= i
//
// where S is the state entering the chunk. Products run on the 5th-gen
// tensor cores (tcgen05.mma, accumulators in tensor memory): the Gram
// matrices [K;Q] K^T in bf16 (exact inputs), everything that touches the
// state or feeds the output with fp16 operands and fp32 accumulation. The
// triangular inverse, the gates and the state update are fp32 on the CUDA
// cores. Raw K, Q, V tiles arrive by TMA (128-byte swizzle) and the next
// chunk's tiles are fetched while the current chunk's spine runs.
//
// Tail rows of a chunk (past the end of the sequence) are treated as k = v =
// 0, beta = 0, g = 0: they contribute nothing and gc_last is the last real
// token's cumulative gate. Their output rows are not stored.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "tc.cuh"

namespace gdn {

constexpr int kDim = 128;    // dk == dv
constexpr int kChunk = 64;   // tokens per chunk
constexpr int kThreads = 256;

// Status bits written to the per-device status word.
constexpr unsigned kStatusBadSeqlens = 1u;
constexpr unsigned kStatusTimeout = 2u;

struct ChunkParams {
  const float* g;
  const float* beta;
  void* state;               // float[B][nv][128][128], or float*[B] when state_is_table
  __nv_bfloat16* out;
  const int32_t* cu_seqlens; // null for dense batches
  const int32_t* order;      // varlen: sequences by decreasing length (null: identity)
  unsigned* status;
  int64_t g_stride, beta_stride, out_stride;
  int B, T, nk, nv;
  int state_is_table;
};

// Shared-memory plan (bytes from a 1024-aligned base). Every operand tile is
// a row-major 16-bit tile stored as 64-column blocks of 128-byte swizzled rows
// (the layout TMA writes); the same bytes serve as a K-major operand whose
// rows are M/N, or an MN-major operand whose rows are K.
template <int NS>
struct Plan {
  static_assert(NS == 64 || NS == 128, "v-slice width");
  static constexpr int KQ = 0;                        // raw bf16 [K;Q]: 2 blocks x 128 rows
  static constexpr int VR = KQ + 2 * 128 * 128;       // raw bf16 V slice: NS/64 blocks x 64 rows
  static constexpr int QT = VR + NS * 128;            // fp16 e^gc Q / sqrt(dk), 64 rows
  static constexpr int KD = QT + 128 * 128;           // fp16 e^{gc_last-gc} K, 64 rows
  static constexpr int W16 = KD + 128 * 128;          // fp16 -W, 64 rows
  static constexpr int TB = W16 + 128 * 128;          // bf16 T diag(beta) hi, lo; T diag(beta e^gc) hi, lo
  static constexpr int A16 = TB + 4 * 64 * 128;       // fp16 A hi, lo (64 x 64 each)
  static constexpr int S16 = A16 + 2 * 64 * 128;      // fp16 S slice, 128 rows x NS
  static constexpr int U16 = S16 + NS * 256;          // fp16 u hi, lo (64 rows x NS each)
  static constexpr int U16_BYTES = NS * 256 > 20480 ? NS * 256 : 20480;
  static constexpr int LF = U16;                      // fp32 L / T work, 64 x 64 (dead before u is written)
  static constexpr int XB = LF + 64 * 64 * 4;         // fp32 inverse partials, 3 x 16 x 16
  static constexpr int BYTES = U16 + U16_BYTES;
  static constexpr int DYN_SMEM = BYTES + 1024;       // slack for 1024-byte alignment
  static_assert(XB + 3 * 256 * 4 <= BYTES, "inverse workspace fits in the u tiles");
  static_assert(DYN_SMEM <= 227 * 1024, "shared memory budget");
  static_assert(QT % 1024 == 0 && TB % 1024 == 0 && S16 % 1024 == 0 && U16 % 1024 == 0, "align");

  // Tensor-memory columns (fp32): Gram [K;Q]K^T (M=128, 64 cols); output
  // accumulator (M=64, NS cols); U (M=64, NS cols) then W (M=64, 128 cols).
  // The state increment (M=128, NS cols) reuses the W columns once W has
  // been read.
  static constexpr uint32_t COL_G = 0;
  static constexpr uint32_t COL_O = 64;
  static constexpr uint32_t COL_U = COL_O + NS;
  static constexpr uint32_t COL_W = COL_U + NS;
  static constexpr uint32_t COL_S = COL_W;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_W + 128 <= TMEM_COLS, "tensor memory budget");
};

// fp32 64 x 64 work matrix with 16-byte chunks XOR-swizzled by row so that a
// warp writing one chunk of 32 different rows hits distinct banks.
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

// x = hi + lo with hi = fp16(x), lo = fp16(x - hi): about 22 significant bits.
__device__ __forceinline__ void split_half8(const float (&f)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 x = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    const float2 xf = __half22float2(x);
    const __half2 y = __floats2half2_rn(f[2 * i] - xf.x, f[2 * i + 1] - xf.y);
    h[i] = *reinterpret_cast<const uint32_t*>(&x);
    l[i] = *reinterpret_cast<const uint32_t*>(&y);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi): about 16 significant bits.
__device__ __forceinline__ void split_bf16x8(const float (&f)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 x = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    const float2 xf = __bfloat1622float2(x);
    const __nv_bfloat162 y = __floats2bfloat162_rn(f[2 * i] - xf.x, f[2 * i + 1] - xf.y);
    h[i] = *reinterpret_cast<const uint32_t*>(&x);
    l[i] = *reinterpret_cast<const uint32_t*>(&y);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int NS>
__global__ void __launch_bounds__(kThreads, 1)
gdn_chunk_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, const ChunkParams p) {
  using P = Plan<NS>;
  constexpr int NSPLIT = kDim / NS;
  constexpr int HALF = NS / 2;  // state / output columns per thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(sm);
  float* lf = reinterpret_cast<float*>(sm + P::LF);
  float* xb = reinterpret_cast<float*>(sm + P::XB);

  __shared__ float s_gc[kChunk], s_eg[kChunk], s_edec[kChunk], s_ebg[kChunk], s_beta[kChunk];
  __shared__ float s_elast;
  __shared__ __align__(8) uint64_t s_mbar_tma, s_mbar_mma;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3;   // tensor-memory lane quarter this warp may access
  const int half = warp >> 2;  // which half of the columns this warp handles

  // ---- which (sequence, head, slice) this CTA owns -------------------------------
  const int vs = blockIdx.x % NSPLIT;
  const int h = (blockIdx.x / NSPLIT) % p.nv;
  const int slot = blockIdx.x / (NSPLIT * p.nv);
  const int s = p.order ? p.order[slot] : slot;
  const int kh = h / (p.nv / p.nk);
  const int v0 = vs * NS;
  int64_t row0, len;
  if (p.cu_seqlens) {
    if (s < 0 || s >= p.B) {
      if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
    const int a = p.cu_seqlens[s], b = p.cu_seqlens[s + 1];
    if (a < 0 || b < a || b > p.T) {
      if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
    row0 = a;
    len = b - a;
  } else {
    row0 = static_cast<int64_t>(s) * p.T;
    len = p.T;
  }
  const int nchunks = static_cast<int>((len + kChunk - 1) / kChunk);
  if (nchunks == 0) return;  // empty sequence: the state passes through unchanged
  float* state = p.state_is_table ? reinterpret_cast<float* const*>(p.state)[s]
                                  : reinterpret_cast<float*>(p.state) + static_cast<int64_t>(s) * p.nv * kDim * kDim;
  state += static_cast<int64_t>(h) * kDim * kDim;

  const uint32_t mbar_tma = tc::smem_u32(&s_mbar_tma);
  const uint32_t mbar_mma = tc::smem_u32(&s_mbar_mma);
  constexpr uint32_t kTmaBytes = (4 + NS / 64) * 64 * 128;
  constexpr uint32_t kMaxPolls = 1u << 24;

  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&s_tmem), P::TMEM_COLS);
  if (tid == 0) {
    s_abort = 0;
    tc::mbar_init(mbar_tma, 1);
    tc::mbar_init(mbar_mma, 1);
    tc::mbar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;

  auto issue_tma = [&](int c) {
    const int32_t y = static_cast<int32_t>(row0 + static_cast<int64_t>(c) * kChunk);
    tc::mbar_arrive_expect_tx(mbar_tma, kTmaBytes);
    tc::tma_load_2d(sbase + P::KQ, &tmap_k, kh * kDim, y, mbar_tma);
    tc::tma_load_2d(sbase + P::KQ + 16384, &tmap_k, kh * kDim + 64, y, mbar_tma);
    tc::tma_load_2d(sbase + P::KQ + 8192, &tmap_q, kh * kDim, y, mbar_tma);
    tc::tma_load_2d(sbase + P::KQ + 16384 + 8192, &tmap_q, kh * kDim + 64, y, mbar_tma);
#pragma unroll
    for (int b = 0; b < NS / 64; ++b)
      tc::tma_load_2d(sbase + P::VR + b * 8192, &tmap_v, h * kDim + v0 + 64 * b, y, mbar_tma);
  };
  // gates of tokens 2*lane and 2*lane+1 of chunk c (warp 0 only)
  float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
  auto load_gates = [&](int c) {
    const int64_t t0 = static_cast<int64_t>(c) * kChunk + 2 * lane;
    g0 = g1 = b0 = b1 = 0.f;
    if (t0 < len) {
      const int64_t r = row0 + t0;
      g0 = p.g[r * p.g_stride + h];
      b0 = p.beta[r * p.beta_stride + h];
    }
    if (t0 + 1 < len) {
      const int64_t r = row0 + t0 + 1;
      g1 = p.g[r * p.g_stride + h];
      b1 = p.beta[r * p.beta_stride + h];
    }
  };

  if (tid == 0) issue_tma(0);
  if (warp == 0) load_gates(0);

  // ---- carried-in state: registers (fp32 master) and fp16 operand tile ------------
  const int krow = quad * 32 + lane;         // state row (key index) this thread owns
  const int vcol0 = half * HALF;             // first slice column this thread owns
  float S[HALF];
  {
    const float4* src = reinterpret_cast<const float4*>(state + static_cast<int64_t>(krow) * kDim + v0 + vcol0);
#pragma unroll
    for (int j = 0; j < HALF / 4; ++j) {
      const float4 x = src[j];
      S[4 * j] = x.x; S[4 * j + 1] = x.y; S[4 * j + 2] = x.z; S[4 * j + 3] = x.w;
    }
  }
  auto store_state_tile = [&]() {
#pragma unroll
    for (int j = 0; j < HALF; j += 8) {
      const int v = vcol0 + j;
      const uint4 w = make_uint4(pack_half2(S[j], S[j + 1]), pack_half2(S[j + 2], S[j + 3]),
                                 pack_half2(S[j + 4], S[j + 5]), pack_half2(S[j + 6], S[j + 7]));
      *reinterpret_cast<uint4*>(sm + P::S16 + (v >> 6) * 16384 + tc::sw128(krow, (v & 63) * 2)) = w;
    }
  };
  store_state_tile();

  uint32_t tma_phase = 0, mma_phase = 0;
  const float inv_sqrt_d = 0.08838834764831845f;  // 1 / sqrt(128)

  // all threads wait on an mbarrier phase; any timeout aborts the whole CTA
  auto wait_all = [&](uint32_t mbar, uint32_t& phase) -> bool {
    if (!tc::mbar_wait(mbar, phase, kMaxPolls)) {
      atomicOr(&s_abort, 1);
      atomicOr(p.status, kStatusTimeout);
    }
    phase ^= 1u;
    tc::fence_after_sync();
    __syncthreads();
    return s_abort == 0;
  };
  auto commit_sync = [&]() {  // make generic smem writes and tmem reads visible, then barrier
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
  };

  bool ok = true;
  for (int c = 0; c < nchunks && ok; ++c) {
    const int64_t rem = len - static_cast<int64_t>(c) * kChunk;
    const int clen = rem < kChunk ? static_cast<int>(rem) : kChunk;
    // ---- stage 1: in-chunk cumulative gate and the per-token scales ----------------
    if (warp == 0) {
      const float pair = g0 + g1;
      float incl = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const float gca = incl - pair + g0, gcb = incl;
      const float glast = __shfl_sync(0xffffffffu, incl, 31);
      s_gc[2 * lane] = gca;
      s_gc[2 * lane + 1] = gcb;
      const float ea = __expf(gca), eb = __expf(gcb);
      s_eg[2 * lane] = ea;
      s_eg[2 * lane + 1] = eb;
      s_edec[2 * lane] = __expf(glast - gca);
      s_edec[2 * lane + 1] = __expf(glast - gcb);
      s_ebg[2 * lane] = b0 * ea;
      s_ebg[2 * lane + 1] = b1 * eb;
      s_beta[2 * lane] = b0;
      s_beta[2 * lane + 1] = b1;
      if (lane == 0) s_elast = __expf(glast);
    }
    __syncthreads();

    // ---- stage 2: Gram matrices [K;Q] K^T (bf16, M=128, N=64, K=128) ----------------
    if (!wait_all(mbar_tma, tma_phase)) break;
    if (tid == 0) {
      constexpr uint32_t idesc = tc::idesc_f16(128, 64, tc::kBF16, false, false);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const uint32_t a = sbase + P::KQ + (st >> 2) * 16384 + (st & 3) * 32;
        tc::mma_f16(tmem + P::COL_G, tc::desc_sw128(a, 16, 1024), tc::desc_sw128(a, 16, 1024), idesc,
                    st > 0);
      }
      tc::mma_commit(mbar_mma);
    }

    // ---- stage 3: fp16 operand tiles from the raw bf16 tiles -----------------------
    // 64 rows x (16 K chunks + 16 Q chunks) of 8 elements each.
    for (int it = tid; it < 64 * 32; it += kThreads) {
      const int t = it & 63;
      const int cc = it >> 6;  // 0..15 K, 16..31 Q
      const bool live = t < clen;
      float f[8];
      if (cc < 16) {
        const uint32_t o = (cc >> 3) * 8192 + tc::sw128(t, (cc & 7) * 16);
        unpack_bf16x8(*reinterpret_cast<const uint4*>(sm + P::KQ + (cc >> 3) * 16384 + tc::sw128(t, (cc & 7) * 16)), f);
        *reinterpret_cast<uint4*>(sm + P::KD + o) = live ? pack_half8(f, s_edec[t]) : make_uint4(0, 0, 0, 0);
      } else {
        const int q8 = cc - 16;
        unpack_bf16x8(*reinterpret_cast<const uint4*>(sm + P::KQ + (q8 >> 3) * 16384 + 8192 + tc::sw128(t, (q8 & 7) * 16)), f);
        *reinterpret_cast<uint4*>(sm + P::QT + (q8 >> 3) * 8192 + tc::sw128(t, (q8 & 7) * 16)) =
            live ? pack_half8(f, s_eg[t] * inv_sqrt_d) : make_uint4(0, 0, 0, 0);
      }
    }

    // ---- stage 4: L (fp32, for the inverse) and the output's intra-chunk matrix A ---
    // A is stored as an fp16 hi/lo pair: A = A_hi + A_lo to ~22 bits.
    if (!wait_all(mbar_mma, mma_phase)) break;
    {
      float d[32], d0[16], d1[16];
      tc::tmem_ld16(tmem + ((quad * 32u) << 16) + P::COL_G + half * 32, d0);
      tc::tmem_ld16(tmem + ((quad * 32u) << 16) + P::COL_G + half * 32 + 16, d1);
      tc::tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        d[e] = d0[e];
        d[16 + e] = d1[e];
      }
      if (quad < 2) {  // K K^T rows -> L_tj = beta_t e^{gc_t - gc_j} k_t.k_j for j < t
        const int t = quad * 32 + lane;
        const float gt = s_gc[t], bt = s_beta[t];
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          float4 w;
          float* wp = reinterpret_cast<float*>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = half * 32 + j4 * 4 + e;
            wp[e] = (j < t && t < clen) ? bt * __expf(gt - s_gc[j]) * d[j4 * 4 + e] : 0.f;
          }
          *reinterpret_cast<float4*>(lf + lf_idx(t, half * 32 + j4 * 4)) = w;
        }
      } else {  // Q K^T rows -> A_ij = e^{gc_i - gc_j} q_i.k_j / sqrt(dk) for j <= i
        const int i = (quad - 2) * 32 + lane;
        const float gi = s_gc[i];
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          float a[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = half * 32 + j8 * 8 + e;
            a[e] = (j <= i) ? __expf(gi - s_gc[j]) * d[j8 * 8 + e] * inv_sqrt_d : 0.f;
          }
          uint4 hi, lo;
          split_half8(a, hi, lo);
          const uint32_t o = tc::sw128(i, (half * 32 + j8 * 8) * 2);
          *reinterpret_cast<uint4*>(sm + P::A16 + o) = hi;
          *reinterpret_cast<uint4*>(sm + P::A16 + 8192 + o) = lo;
        }
      }
    }
    commit_sync();

    // ---- stage 5: T = (I + L)^{-1}, blocked over 16 x 16 blocks, fp32 ---------------
    {
      float x[16];
      const int bb = tid >> 4, col = tid & 15;
      if (tid < 64) {  // diagonal blocks: column `col` of block `bb` by forward substitution
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float val = (i == col) ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < i; ++m)
            if (m >= col) val -= lf[lf_idx(16 * bb + i, 16 * bb + m)] * x[m];
          x[i] = (i < col) ? 0.f : val;
        }
      }
      __syncthreads();
      if (tid < 64) {
#pragma unroll
        for (int i = 0; i < 16; ++i) lf[lf_idx(16 * bb + i, 16 * bb + col)] = x[i];
      }
      __syncthreads();
      // off-diagonal blocks, block row by block row:
      //   T_ij = -T_ii * sum_{k=j}^{i-1} L_ik T_kj
      for (int ib = 1; ib < 4; ++ib) {
        for (int e = tid; e < ib * 256; e += kThreads) {
          const int jb = e >> 8, r = (e >> 4) & 15, cc = e & 15;
          float acc = 0.f;
          for (int kb = jb; kb < ib; ++kb) {
#pragma unroll
            for (int m = 0; m < 16; ++m)
              acc += lf[lf_idx(16 * ib + r, 16 * kb + m)] * lf[lf_idx(16 * kb + m, 16 * jb + cc)];
          }
          xb[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < ib * 256; e += kThreads) {
          const int jb = e >> 8, r = (e >> 4) & 15, cc = e & 15;
          float acc = 0.f;
#pragma unroll
          for (int m = 0; m < 16; ++m) acc += lf[lf_idx(16 * ib + r, 16 * ib + m)] * xb[jb * 256 + m * 16 + cc];
          lf[lf_idx(16 * ib + r, 16 * jb + cc)] = -acc;
        }
        __syncthreads();
      }
      // bf16 hi/lo tiles of T diag(beta) and T diag(beta e^gc) (rows t, columns j),
      // zero above the diagonal blocks
      {
        const int t = tid >> 2, j0 = (tid & 3) * 16;
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          float fb[8], fe[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = j0 + h8 * 8 + e;
            const float tv = ((j >> 4) <= (t >> 4)) ? lf[lf_idx(t, j)] : 0.f;
            fb[e] = tv * s_beta[j];
            fe[e] = tv * s_ebg[j];
          }
          const uint32_t o = tc::sw128(t, (j0 + h8 * 8) * 2);
          uint4 hi, lo;
          split_bf16x8(fb, hi, lo);
          *reinterpret_cast<uint4*>(sm + P::TB + o) = hi;
          *reinterpret_cast<uint4*>(sm + P::TB + 8192 + o) = lo;
          split_bf16x8(fe, hi, lo);
          *reinterpret_cast<uint4*>(sm + P::TB + 16384 + o) = hi;
          *reinterpret_cast<uint4*>(sm + P::TB + 24576 + o) = lo;
        }
      }
    }
    commit_sync();

    // ---- stage 6: U = T diag(beta) V and W = T diag(beta e^gc) K, bf16 hi + lo ------
    // The raw bf16 V and K tiles are exact, so only T's side is split.
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t id_u = tc::idesc_f16(64, NS, tc::kBF16, false, true);
      constexpr uint32_t id_w = tc::idesc_f16(64, 128, tc::kBF16, false, true);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          tc::mma_f16(tmem + P::COL_U, tc::desc_sw128(sbase + P::TB + part * 8192 + st * 32, 16, 1024),
                      tc::desc_sw128(sbase + P::VR + st * 2048, 64 * 128, 1024), id_u, part + st > 0);
          tc::mma_f16(tmem + P::COL_W, tc::desc_sw128(sbase + P::TB + 16384 + part * 8192 + st * 32, 16, 1024),
                      tc::desc_sw128(sbase + P::KQ + st * 2048, 128 * 128, 1024), id_w, part + st > 0);
        }
      }
      tc::mma_commit(mbar_mma);
    }
    if (!wait_all(mbar_mma, mma_phase)) break;
    // raw tiles are free now: fetch the next chunk's tiles and gates
    if (c + 1 < nchunks) {
      if (tid == 0) issue_tma(c + 1);
      if (warp == 0) load_gates(c + 1);
    }

    // ---- stage 7: -W as an fp16 operand (rows t, 64 of its 128 columns per warp) ----
    {
      const int t = quad * 16 + lane;  // M=64 accumulator: row 16q+l lives in lane 32q+l
#pragma unroll
      for (int q16 = 0; q16 < 4; ++q16) {
        float d[16];
        tc::tmem_ld16(tmem + ((quad * 32u) << 16) + P::COL_W + half * 64 + q16 * 16, d);
        tc::tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = d[h8 * 8 + e];
            *reinterpret_cast<uint4*>(sm + P::W16 + half * 8192 + tc::sw128(t, (q16 * 16 + h8 * 8) * 2)) =
                pack_half8(f, -1.f);
          }
        }
      }
    }
    commit_sync();

    // ---- stage 8: u = U - W S (into U), and the output's inter-chunk term Q~ S -------
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t idesc = tc::idesc_f16(64, NS, tc::kF16, false, true);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const uint64_t bd = tc::desc_sw128(sbase + P::S16 + st * 2048, 128 * 128, 1024);
        tc::mma_f16(tmem + P::COL_U, tc::desc_sw128(sbase + P::W16 + (st >> 2) * 8192 + (st & 3) * 32, 16, 1024),
                    bd, idesc, 1);
        tc::mma_f16(tmem + P::COL_O, tc::desc_sw128(sbase + P::QT + (st >> 2) * 8192 + (st & 3) * 32, 16, 1024),
                    bd, idesc, st > 0);
      }
      tc::mma_commit(mbar_mma);
    }
    if (!wait_all(mbar_mma, mma_phase)) break;

    // ---- stage 9: u as an fp16 hi/lo operand pair (rows t, NS/2 columns per warp) ----
    {
      const int t = quad * 16 + lane;
#pragma unroll
      for (int q16 = 0; q16 < HALF / 16; ++q16) {
        float d[16];
        tc::tmem_ld16(tmem + ((quad * 32u) << 16) + P::COL_U + vcol0 + q16 * 16, d);
        tc::tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = d[h8 * 8 + e];
            const int v = vcol0 + q16 * 16 + h8 * 8;
            const uint32_t o = (v >> 6) * 8192 + tc::sw128(t, (v & 63) * 2);
            uint4 hi, lo;
            split_half8(f, hi, lo);
            *reinterpret_cast<uint4*>(sm + P::U16 + o) = hi;
            *reinterpret_cast<uint4*>(sm + P::U16 + NS * 128 + o) = lo;
          }
        }
      }
    }
    commit_sync();

    // ---- stage 10: state increment Kd^T u (M=128, N=NS, K=64) and output += A u ------
    // A u = A_hi u_hi + A_hi u_lo + A_lo u_hi (fp16 operands, fp32 accumulate).
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t id_s = tc::idesc_f16(128, NS, tc::kF16, true, true);
      constexpr uint32_t id_o = tc::idesc_f16(64, NS, tc::kF16, false, true);
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint64_t u_hi = tc::desc_sw128(sbase + P::U16 + st * 2048, 64 * 128, 1024);
        const uint64_t u_lo = tc::desc_sw128(sbase + P::U16 + NS * 128 + st * 2048, 64 * 128, 1024);
        const uint64_t a_hi = tc::desc_sw128(sbase + P::A16 + st * 32, 16, 1024);
        const uint64_t a_lo = tc::desc_sw128(sbase + P::A16 + 8192 + st * 32, 16, 1024);
        tc::mma_f16(tmem + P::COL_S, tc::desc_sw128(sbase + P::KD + st * 2048, 64 * 128, 1024), u_hi, id_s, st > 0);
        tc::mma_f16(tmem + P::COL_O, a_hi, u_hi, id_o, 1);
        tc::mma_f16(tmem + P::COL_O, a_hi, u_lo, id_o, 1);
        tc::mma_f16(tmem + P::COL_O, a_lo, u_hi, id_o, 1);
      }
      tc::mma_commit(mbar_mma);
    }
    if (!wait_all(mbar_mma, mma_phase)) break;

    // ---- stage 11: S <- e^{gc_last} S + Kd^T u (fp32 master), and the output rows -----
    {
      const float el = s_elast;
#pragma unroll
      for (int q16 = 0; q16 < HALF / 16; ++q16) {
        float d[16];
        tc::tmem_ld16(tmem + ((quad * 32u) << 16) + P::COL_S + vcol0 + q16 * 16, d);
        tc::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) S[q16 * 16 + e] = fmaf(el, S[q16 * 16 + e], d[e]);
      }
      store_state_tile();
      const int i = quad * 16 + lane;
      const bool live = lane < 16 && i < clen;
      __nv_bfloat16* orow = p.out + (row0 + static_cast<int64_t>(c) * kChunk + i) * p.out_stride +
                            static_cast<int64_t>(h) * kDim + v0 + vcol0;
#pragma unroll
      for (int q16 = 0; q16 < HALF / 16; ++q16) {
        float d[16];
        tc::tmem_ld16(tmem + ((quad * 32u) << 16) + P::COL_O + vcol0 + q16 * 16, d);
        tc::tmem_ld_wait();
        if (live) {
          uint4 w0 = make_uint4(pack_bf162(d[0], d[1]), pack_bf162(d[2], d[3]), pack_bf162(d[4], d[5]),
                                pack_bf162(d[6], d[7]));
          uint4 w1 = make_uint4(pack_bf162(d[8], d[9]), pack_bf162(d[10], d[11]), pack_bf162(d[12], d[13]),
                                pack_bf162(d[14], d[15]));
          reinterpret_cast<uint4*>(orow + q16 * 16)[0] = w0;
          reinterpret_cast<uint4*>(orow + q16 * 16)[1] = w1;
        }
      }
    }
    commit_sync();
  }

  if (s_abort == 0) {
    float4* dst = reinterpret_cast<float4*>(state + static_cast<int64_t>(krow) * kDim + v0 + vcol0);
#pragma unroll
    for (int j = 0; j < HALF / 4; ++j) dst[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
  } else {
    // a wait expired: let outstanding async work drain (bounded) before freeing tensor memory
    if (tid == 0) {
      tc::mbar_wait(mbar_mma, mma_phase, kMaxPolls);
      tc::mbar_wait(mbar_tma, tma_phase, kMaxPolls);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, P::TMEM_COLS);
  }
}

}  // namespace gdn

// Per-chunk gradients of the chunked backward on the 5th-generation tensor cores.
//
// With S0 and dS_end of every chunk stored by the two chains (the forward chain and
// gdn_bwd_dstates_tc.cuh), the gradients of a chunk (derived in the header of
// gdn_bwd_common.cuh) need no state from other chunks:
//
//     dQ = Gamma dO S0^T / sqrt(dk) + dA K
//     dK = E K + E^T K - Gamma beta P + dA^T Q + (gamma / Gamma) u dS_end^T
//     dbeta, d b and dg from the per-token sums of those products
//
// with P = du' S0^T, dA = lower(dO u^T) . M / sqrt(dk), F = -strict_lower(du' u^T) . M,
// E = beta F. One CTA takes a (chunk, key head) and walks the value heads of its GQA
// group; every product is a tcgen05 MMA of M = 128 issued by thread 0, with the rows of
// two 64-row operands stacked so that one MMA serves both:
//
//     Gram  [Q;K] K^T                 (M=128, N=64):  lanes 0-63 Q K^T, 64-127 K K^T
//     X1    [dO; du'] S0^T            (M=128, N=128): lanes 0-63 dO S0^T, 64-127 P
//     X2    [dO; du'] u^T             (M=128, N=64):  lanes 0-63 dO u^T, 64-127 du' u^T
//     UD    [0; u] dS_end^T           (M=128, N=128): lanes 64-127 u dS_end^T
//     Y    += [dA; E] K + [0; E^T] K + [0; dA^T] Q    (M=128, N=128, over the group)
//
// Lanes 0-63 of Y accumulate dQ and lanes 64-127 dK. The transposed operands E^T and dA^T
// are the dA and E tiles themselves, read as MN-major A operands next to a zero tile. The
// row-scaled terms (Gamma dO S0^T / sqrt(dk), -Gamma beta P, (gamma / Gamma) u dS_end^T)
// are added to Y in tensor memory by the epilogue, which also forms the per-token sums.
// Operands are fp16 with fp32 accumulation, as in the chains: q, k (bf16 rows), dO (fp32
// rows), u, du', S0 and dS_end (the chains' fp16 stores). Every wait is bounded; on
// expiry the CTA sets the status bit and stops.
#pragma once
#include "gdn_bwd_common.cuh"

namespace gdn {

struct GtPlan {
  // byte offsets from a 1024-aligned base: 16-bit tiles of 128-byte swizzled rows,
  // 64 columns per 16 KB block of 128 rows
  static constexpr int QK = 0;        // fp16 [Q;K] (rows 0-63 Q, 64-127 K) x k, two k-blocks
  static constexpr int AX = 32768;    // fp16 [dO; du'] x v, two v-blocks
  static constexpr int AU = 65536;    // fp16 [0; u] x v, two v-blocks (rows 0-63 stay zero)
  static constexpr int S0 = 98304;    // fp16 S0 [k][v], two v-blocks of 128 rows
  static constexpr int DSE = 131072;  // fp16 dS_end [k][v], likewise
  static constexpr int ZDE = 163840;  // fp16 64 x 64 tiles: zeros, then dA [t][t'], then E [t][t']
  static constexpr int BYTES = 188416;
  static constexpr int DYN_SMEM = BYTES + 1024;  // slack for 1024-byte alignment
  // tensor-memory columns
  static constexpr uint32_t COL_G = 0;     // Gram (64)
  static constexpr uint32_t COL_X2 = 64;   // X2 (64)
  static constexpr uint32_t COL_X1 = 128;  // X1 (128)
  static constexpr uint32_t COL_UD = 256;  // UD (128)
  static constexpr uint32_t COL_Y = 384;   // [dQ; dK] (128)
  static constexpr uint32_t TMEM_COLS = 512;
};

constexpr int kGtThreads = 512;

// Column sums of a 32-row x 16-column block held one row per lane: returns, in lanes l
// and l ^ 1, the sum over the 32 lanes of column gt_col(l) (halving exchanges).
__device__ __forceinline__ int gt_col(int l) {
  return ((l >> 4) & 1) * 8 + ((l >> 3) & 1) * 4 + ((l >> 2) & 1) * 2 + ((l >> 1) & 1);
}
__device__ __forceinline__ float gt_colsum16(const float (&v)[16], int lane) {
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const bool hi = lane & 16;
    const float send = hi ? v[k] : v[k + 8], keep = hi ? v[k + 8] : v[k];
    a[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
  float b[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const bool hi = lane & 8;
    const float send = hi ? a[k] : a[k + 4], keep = hi ? a[k + 4] : a[k];
    b[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float c[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const bool hi = lane & 4;
    const float send = hi ? b[k] : b[k + 2], keep = hi ? b[k + 2] : b[k];
    c[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const bool hi = lane & 2;
  float d = (hi ? c[1] : c[0]) + __shfl_xor_sync(0xffffffffu, hi ? c[0] : c[1], 2);
  return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

// Sum of the products of 8 fp16 pairs
__device__ __forceinline__ float gt_dot_h8(const uint4 a, const float (&b)[8]) {
  const __half2* a2 = reinterpret_cast<const __half2*>(&a);
  float s = 0.f;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const float2 f = __half22float2(a2[x]);
    s = fmaf(f.x, b[2 * x], fmaf(f.y, b[2 * x + 1], s));
  }
  return s;
}

__global__ void __launch_bounds__(kGtThreads, 1) gdn_bwd_grads_tc_kernel(const BwdChunkParams p) {
  using P = GtPlan;
  extern __shared__ uint8_t smem_raw[];
  // per token of the current value head: log-decay prefix b and beta; the per-token sums
  // q.(dO S0^T), k.P, rows / columns of dA . QK^T, rows / columns of E . G, rows of F . G,
  // w, du'.v; and <dS_end, S0>
  __shared__ float s_b[kChunk], s_beta[kChunk];
  __shared__ float s_sum[9][kChunk];
  __shared__ float s_dot;
  __shared__ __align__(8) uint64_t s_mb[3];
  __shared__ uint32_t s_tmem;
  float* const s_rq = s_sum[0];
  float* const s_rkp = s_sum[1];
  float* const s_r1 = s_sum[2];
  float* const s_c1 = s_sum[3];
  float* const s_r2 = s_sum[4];
  float* const s_c2 = s_sum[5];
  float* const s_rf = s_sum[6];
  float* const s_rw = s_sum[7];
  float* const s_rdv = s_sum[8];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, part = warp >> 2;  // lane quarter; column quarter
  const int r = quarter * 32 + lane;              // this thread's accumulator row (lane)

  const int ci = blockIdx.x / p.nk, kh = blockIdx.x % p.nk;
  int group = p.nv / p.nk;
  int s;
  int64_t c;
  if (p.cu_seqlens) {
    if (ci >= p.cu_chunks[p.B]) return;
    int lo = 0, hi = p.B - 1;  // the sequence with cu_chunks[s] <= ci < cu_chunks[s + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.cu_chunks[mid] <= ci) lo = mid;
      else hi = mid - 1;
    }
    s = lo;
    c = ci - p.cu_chunks[s];
  } else {
    const int nch = (p.T + kChunk - 1) / kChunk;
    s = ci / nch;
    c = ci % nch;
    if (s >= p.B) return;
  }
  int64_t row0, len;
  if (!bc_sequence(p, s, row0, len)) return;
  const int64_t r0 = row0 + c * kChunk;
  if (c * kChunk >= len) return;
  const int n = static_cast<int>(len - c * kChunk < kChunk ? len - c * kChunk : kChunk);
  const int64_t hrow = static_cast<int64_t>(p.nv) * kDim, krow = static_cast<int64_t>(p.nk) * kDim;

  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = tc::smem_u32(sm);
  const uint32_t mb_g = tc::smem_u32(&s_mb[0]), mb_x = tc::smem_u32(&s_mb[1]), mb_y = tc::smem_u32(&s_mb[2]);

  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&s_tmem), P::TMEM_COLS);
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 3; ++i) tc::mbar_init(tc::smem_u32(&s_mb[i]), 1);
    tc::mbar_fence_init();
  }
  // zero tiles: rows 0-63 of both [0; u] blocks and the tile before dA
  {
    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < 3; ++i) {  // 3 x 8 KB = 1536 pieces of 16 bytes
      const int idx = tid + kGtThreads * i, blk = idx >> 9, o = (idx & 511) * 16;
      const int base = blk < 2 ? P::AU + blk * 16384 : P::ZDE;
      *reinterpret_cast<uint4*>(sm + base + o) = z;
    }
  }
  // q and k rows of the key head as fp16 (rows past the chunk's end zero): Q rows 0-63
  // and K rows 64-127 of each 64-column block
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int idx = tid + kGtThreads * i, t = idx & 63, c8 = (idx >> 6) & 15, isk = idx >> 10;
    const __nv_bfloat16* src = (isk ? p.k + (r0 + t) * p.k_stride : p.q + (r0 + t) * p.q_stride) + kh * kDim + 8 * c8;
    const uint4 raw = t < n ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
    float f[8];
    unpack_bf16x8(raw, f);
    *reinterpret_cast<uint4*>(sm + P::QK + (c8 >> 3) * 16384 + tc::sw128(isk * 64 + t, (c8 & 7) * 16)) =
        pack_half8(f, 1.f);
  }
  tc::fence_proxy_async();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t lanes = tmem + ((static_cast<uint32_t>(quarter) * 32u) << 16);

  bool ok = true;
  auto wait_mb = [&](uint32_t mb, uint32_t parity) {
    bool w = ok && tc::mbar_wait_timed(mb, parity, kWaitLimitNs);
    w = __syncthreads_and(w) != 0;
    if (!w && ok && tid == 0) atomicOr(p.status, kStatusTimeout);
    ok = w;
    tc::fence_after_sync();
    return w;
  };

  // Gram [Q;K] K^T, and [dQ; dK] = 0
  if (tid == 0) {
    constexpr uint32_t id_g = tc::idesc_f16(128, 64, tc::kF16, false, false);
    const uint64_t dqk = tc::desc_sw128(sb + P::QK, 16, 1024);
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      const uint64_t a = dqk + (((st >> 2) * 16384 + (st & 3) * 32) >> 4);
      tc::mma_f16(tmem + P::COL_G, a, a + (8192 >> 4), id_g, st > 0);
    }
    tc::mma_commit(mb_g);
  }
  {
    uint32_t z[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) z[e] = 0u;
    tc::tmem_st32(lanes + P::COL_Y + part * 32, z);
    tc::tmem_st_wait();
  }
  if (!wait_mb(mb_g, 0)) group = 0;

  for (int j = 0; j < group; ++j) {
    const int h = kh * group + j;
    const uint32_t ph = static_cast<uint32_t>(j) & 1u;
    const int64_t state_off = (bc_slot(row0, s, c) * p.nv + h) * kDim * kDim;

    // ---- this value head's operands --------------------------------------------------------
    {
      const __half* dug = p.dubuf + r0 * hrow + h * kDim;
      const __half* ug = p.ubuf + r0 * hrow + h * kDim;
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // du' into rows 64-127 of [dO; du'], u into rows 64-127 of [0; u]
        const int idx = tid + kGtThreads * i, t = idx & 63, c8 = idx >> 6;
        const int64_t srow = t < n ? t : 0;
        const uint32_t o = (c8 >> 3) * 16384 + tc::sw128(64 + t, (c8 & 7) * 16);
        cp_async16(sb + P::AX + o, dug + srow * hrow + 8 * c8, t < n);
        cp_async16(sb + P::AU + o, ug + srow * hrow + 8 * c8, t < n);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // S0 and dS_end, [k][v]
        const int idx = tid + kGtThreads * i, k = idx & 127, c8 = idx >> 7;
        const uint32_t o = (c8 >> 3) * 16384 + tc::sw128(k, (c8 & 7) * 16);
        cp_async16(sb + P::S0 + o, p.s0buf + state_off + k * kDim + 8 * c8, true);
        cp_async16(sb + P::DSE + o, p.dsbuf + state_off + k * kDim + 8 * c8, true);
      }
      tc::cp_async_commit();
      const float* dog = p.dout + r0 * hrow + h * kDim;
#pragma unroll
      for (int i = 0; i < 2; ++i) {  // dO as fp16 into rows 0-63 of [dO; du']
        const int idx = tid + kGtThreads * i, t = idx & 63, c8 = idx >> 6;
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (t < n) {
          const float4 a = __ldg(reinterpret_cast<const float4*>(dog + t * hrow + 8 * c8));
          const float4 b = __ldg(reinterpret_cast<const float4*>(dog + t * hrow + 8 * c8 + 4));
          f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        }
        *reinterpret_cast<uint4*>(sm + P::AX + (c8 >> 3) * 16384 + tc::sw128(t, (c8 & 7) * 16)) = pack_half8(f, 1.f);
      }
      if (warp == 0) {
        BcGates fg;
        bc_fetch_gates(fg, p, r0, n, h);
        bc_put_gates(fg, s_b, s_beta);
      }
      if (tid < kChunk) {
#pragma unroll
        for (int q = 0; q < 9; ++q) s_sum[q][tid] = 0.f;
        if (tid == 0) s_dot = 0.f;
      }
      tc::cp_async_wait_all();
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- X1, X2, UD -------------------------------------------------------------------------
    if (tid == 0) {
      constexpr uint32_t id_n128 = tc::idesc_f16(128, 128, tc::kF16, false, false);
      constexpr uint32_t id_n64 = tc::idesc_f16(128, 64, tc::kF16, false, false);
      const uint64_t dax = tc::desc_sw128(sb + P::AX, 16, 1024), dau = tc::desc_sw128(sb + P::AU, 16, 1024);
      const uint64_t ds0 = tc::desc_sw128(sb + P::S0, 16, 1024), dse = tc::desc_sw128(sb + P::DSE, 16, 1024);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const uint64_t off = ((st >> 2) * 16384 + (st & 3) * 32) >> 4;
        tc::mma_f16(tmem + P::COL_X1, dax + off, ds0 + off, id_n128, st > 0);
        tc::mma_f16(tmem + P::COL_X2, dax + off, dau + (8192 >> 4) + off, id_n64, st > 0);
        tc::mma_f16(tmem + P::COL_UD, dau + off, dse + off, id_n128, st > 0);
      }
      tc::mma_commit(mb_x);
    }
    // (the X commit also covers the previous value head's Y MMAs: Y, dA and E are free)
    if (!wait_mb(mb_x, ph)) break;

    // ---- dA and E from X2 and the Gram, with their row and column sums -----------------------
    {
      const int i0 = 16 * part;
      float x[16], gm[16];
      tc::tmem_ld16(lanes + P::COL_X2 + i0, x);
      tc::tmem_ld16(lanes + P::COL_G + i0, gm);
      tc::tmem_ld_wait();
      const int t = r & 63;
      const float bt = s_b[t];
      float rs = 0.f, rfs = 0.f, v[16];
      if (r < 64) {  // dA = lower(dO u^T) . M / sqrt(dk); sums of dA . (Q K^T)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int i = i0 + e;
          const float m = i <= t ? __expf(bt - s_b[i]) : 0.f;
          x[e] = x[e] * (m * kInvSqrtD);
          v[e] = x[e] * gm[e];
          rs += v[e];
        }
      } else {  // E = beta F, F = -strict_lower(du' u^T) . M; sums of F . G and E . G
        const float be = s_beta[t];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int i = i0 + e;
          const float m = i < t ? __expf(bt - s_b[i]) : 0.f;
          const float f = -x[e] * m;
          rfs = fmaf(f, gm[e], rfs);
          x[e] = be * f;
          v[e] = x[e] * gm[e];
          rs += v[e];
        }
      }
      uint32_t hx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) hx[e] = pack_half2(x[2 * e], x[2 * e + 1]);
      const uint32_t tile = P::ZDE + (r < 64 ? 8192 : 16384);
      *reinterpret_cast<uint4*>(sm + tile + tc::sw128(t, i0 * 2)) = make_uint4(hx[0], hx[1], hx[2], hx[3]);
      *reinterpret_cast<uint4*>(sm + tile + tc::sw128(t, i0 * 2 + 16)) = make_uint4(hx[4], hx[5], hx[6], hx[7]);
      const float cs = gt_colsum16(v, lane);
      if (r < 64) {
        atomicAdd(&s_r1[t], rs);
        if (!(lane & 1)) atomicAdd(&s_c1[i0 + gt_col(lane)], cs);
      } else {
        atomicAdd(&s_r2[t], rs);
        atomicAdd(&s_rf[t], rfs);
        if (!(lane & 1)) atomicAdd(&s_c2[i0 + gt_col(lane)], cs);
      }
    }

    // ---- Y += Gamma dO S0^T / sqrt(dk) (rows 0-63); Y += -Gamma beta P + (gamma / Gamma)
    //      u dS_end^T (rows 64-127); the row sums q.(dO S0^T), k.P and w -------------------------
    {
      const int t = r & 63;
      const float G = __expf(s_b[t]);
      const float gl = s_b[kChunk - 1];
      const float f1 = r < 64 ? G * kInvSqrtD : -G * s_beta[t];
      const float fu = __expf(gl - s_b[t]);
      float d1 = 0.f, dw = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int k0 = 32 * part + 16 * hh;
        float x1[16], ud[16], y[16];
        tc::tmem_ld16(lanes + P::COL_X1 + k0, x1);
        tc::tmem_ld16(lanes + P::COL_UD + k0, ud);
        tc::tmem_ld16(lanes + P::COL_Y + k0, y);
        tc::tmem_ld_wait();
        // row r of [Q;K] (q_t for rows 0-63, k_t for 64-127), columns k0 .. k0 + 15
        const uint32_t rowoff = P::QK + (k0 >> 6) * 16384;
        const uint4 qa = *reinterpret_cast<const uint4*>(sm + rowoff + tc::sw128(r, (k0 & 63) * 2));
        const uint4 qb = *reinterpret_cast<const uint4*>(sm + rowoff + tc::sw128(r, (k0 & 63) * 2 + 16));
        const float xa[8] = {x1[0], x1[1], x1[2], x1[3], x1[4], x1[5], x1[6], x1[7]};
        const float xb[8] = {x1[8], x1[9], x1[10], x1[11], x1[12], x1[13], x1[14], x1[15]};
        d1 += gt_dot_h8(qa, xa) + gt_dot_h8(qb, xb);
        if (r >= 64) {
#pragma unroll
          for (int e = 0; e < 16; ++e) ud[e] *= fu;
          const float ua[8] = {ud[0], ud[1], ud[2], ud[3], ud[4], ud[5], ud[6], ud[7]};
          const float ub[8] = {ud[8], ud[9], ud[10], ud[11], ud[12], ud[13], ud[14], ud[15]};
          dw += gt_dot_h8(qa, ua) + gt_dot_h8(qb, ub);
#pragma unroll
          for (int e = 0; e < 16; ++e) y[e] = fmaf(f1, x1[e], y[e] + ud[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) y[e] = fmaf(f1, x1[e], y[e]);
        }
        tc::tmem_st16(lanes + P::COL_Y + k0, y);
      }
      tc::tmem_st_wait();
      if (r < 64) {
        atomicAdd(&s_rq[t], d1);
      } else {
        atomicAdd(&s_rkp[t], d1);
        atomicAdd(&s_rw[t], dw);
      }
    }

    // ---- du'_t . v_t (rows 64-127: du' rows of [dO; du']) and <dS_end, S0> (the others) ----
    if (r >= 64) {
      const int t = r - 64;
      float d = 0.f;
      if (t < n) {
        const __nv_bfloat16* vg = p.v + (r0 + t) * p.v_stride + h * kDim + 32 * part;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int col = 32 * part + 8 * q;
          const uint4 du = *reinterpret_cast<const uint4*>(sm + P::AX + (col >> 6) * 16384 + tc::sw128(r, (col & 63) * 2));
          float vf[8];
          unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(vg + 8 * q)), vf);
          d += gt_dot_h8(du, vf);
        }
      }
      atomicAdd(&s_rdv[t], d);
    } else {
      float d = 0.f;
      const int u256 = part * 64 + r;  // this thread among the 256 of rows 0-63
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // 2048 pieces of 16 bytes over 256 threads
        const int idx = u256 + 256 * i;
        const uint4 a = *reinterpret_cast<const uint4*>(sm + P::S0 + idx * 16);
        const uint4 b = *reinterpret_cast<const uint4*>(sm + P::DSE + idx * 16);
        const __half2* b2 = reinterpret_cast<const __half2*>(&b);
        float bf[8];
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const float2 f = __half22float2(b2[x]);
          bf[2 * x] = f.x;
          bf[2 * x + 1] = f.y;
        }
        d += gt_dot_h8(a, bf);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (lane == 0) atomicAdd(&s_dot, d);
    }
    tc::fence_proxy_async();  // dA and E, for the Y MMAs
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---- Y += [dA; E] K + [0; E^T] K + [0; dA^T] Q ------------------------------------------
    if (tid == 0) {
      constexpr uint32_t id_kk = tc::idesc_f16(128, 128, tc::kF16, false, true);
      constexpr uint32_t id_mk = tc::idesc_f16(128, 128, tc::kF16, true, true);
      const uint64_t dade = tc::desc_sw128(sb + P::ZDE + 8192, 16, 1024);   // [dA; E], K-major
      const uint64_t det = tc::desc_sw128(sb + P::ZDE, 16384, 1024);        // [0; E^T], MN-major
      const uint64_t ddat = tc::desc_sw128(sb + P::ZDE, 8192, 1024);        // [0; dA^T], MN-major
      const uint64_t bk = tc::desc_sw128(sb + P::QK + 8192, 16384, 1024);   // K, MN-major
      const uint64_t bq = tc::desc_sw128(sb + P::QK, 16384, 1024);          // Q, MN-major
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        tc::mma_f16(tmem + P::COL_Y, dade + st * 2, bk + st * 128, id_kk, 1);
        tc::mma_f16(tmem + P::COL_Y, det + st * 128, bk + st * 128, id_mk, 1);
        tc::mma_f16(tmem + P::COL_Y, ddat + st * 128, bq + st * 128, id_mk, 1);
      }
      tc::mma_commit(mb_y);
    }

    // ---- per-token dbeta and d b of this value head, then dg = suffix sums of d b (warp 0) -----
    if (warp == 0) {
      const float gam = __expf(s_b[kChunk - 1]);
      float wsum = s_rw[2 * lane] + s_rw[2 * lane + 1];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
      float db[2], dbe[2];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int t = 2 * lane + x;
        const float G = __expf(s_b[t]);
        db[x] = G * kInvSqrtD * s_rq[t] - G * s_beta[t] * s_rkp[t] + (s_r2[t] - s_c2[t]) + (s_r1[t] - s_c1[t]) -
                s_rw[t];
        dbe[x] = s_rdv[t] - G * s_rkp[t] + s_rf[t];
      }
      if (lane == 31) db[1] += gam * s_dot + wsum;
      const float pair = db[0] + db[1];
      float incl = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      const float dg0 = incl, dg1 = incl - db[0];
      const int t0 = 2 * lane, t1 = t0 + 1;
      if (t0 < n) {
        p.dg[(r0 + t0) * p.nv + h] = dg0;
        p.dbeta[(r0 + t0) * p.nv + h] = dbe[0];
      }
      if (t1 < n) {
        p.dg[(r0 + t1) * p.nv + h] = dg1;
        p.dbeta[(r0 + t1) * p.nv + h] = dbe[1];
      }
    }
    __syncthreads();  // the per-token sums are read before the next value head clears them
  }

  // ---- dQ (rows 0-63) and dK (rows 64-127) ------------------------------------------------
  if (group > 0 && wait_mb(mb_y, static_cast<uint32_t>(group - 1) & 1u)) {
    const int t = r & 63;
    float* dst = (r < 64 ? p.dq : p.dk) + (r0 + t) * krow + kh * kDim + 32 * part;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float y[16];
      // (every lane: tensor-memory loads are warp-collective; only the stores are per row)
      tc::tmem_ld16(lanes + P::COL_Y + 32 * part + 16 * hh, y);
      tc::tmem_ld_wait();
      if (t < n) {
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4)
          *reinterpret_cast<float4*>(dst + 16 * hh + 4 * e4) =
              make_float4(y[4 * e4], y[4 * e4 + 1], y[4 * e4 + 2], y[4 * e4 + 3]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    if (!ok) {  // a wait expired: give any copy or MMA still in flight time to land
      const uint64_t t0 = tc::globaltimer_ns();
      while (tc::globaltimer_ns() - t0 < 2000000ull) __nanosleep(1000);
    }
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, P::TMEM_COLS);
  }
}

}  // namespace gdn

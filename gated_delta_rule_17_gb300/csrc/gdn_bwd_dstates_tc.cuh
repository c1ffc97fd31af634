// Reverse chain of the chunked backward on the 5th-generation tensor cores.
//
// The reverse chain of the chunk-level derivative (derived in the header of
// gdn_bwd_common.cuh), per chunk c from the last:
//
//     du  = (Q K^T . M)^T dO / sqrt(dk) + (gamma / Gamma) K dS_end
//     du' = T^T du,  dV = beta du'
//     dS0 = gamma dS_end + Q^T (Gamma dO) / sqrt(dk) - K^T (Gamma beta du')
//
// computed transposed, with the value index on the 128 tensor-memory lanes: dS^T [v][k]
// stays in tensor memory as the fp32 accumulator, and every product is one tcgen05 MMA
// group issued by thread 0:
//
//     Gram    [K;Q] K^T              (bf16, M = 128, N = 64; lanes 64-127 are Q K^T)
//     P2      dS^T K^T               (A = dS^T as bf16 hi + lo from tensor memory)
//     P1      dO^T A~                (fp16; A~ = (Q K^T . M) / sqrt(dk), lower triangle)
//     P3      du^T T                 (fp16 hi + lo of both)
//     P4      dS^T += (Gamma dO / sqrt(dk))^T Q + (-Gamma beta du')^T K   (bf16 hi + lo)
//
// Between them 16 warps move accumulators through registers (warp w reaches lanes
// 32 (w % 4) .. + 31 and takes the column quarter w / 4 of each accumulator): du^T = P1 +
// (gamma / Gamma_t) P2 (zero past the chunk's end), the du' and dV rows, the scaled
// operand of P4, the decay dS^T <- gamma dS^T, and the bf16 copy of dS^T for the next
// chunk's P2. Operand tiles use the 128-byte swizzle (tc.cuh). K and Q arrive by TMA
// (two buffers, one chunk ahead); dO and T by cp.async one chunk ahead. Every wait is
// bounded; on expiry the CTA sets the status bit and stops.
#pragma once
#include "gdn_bwd_common.cuh"

namespace gdn {

struct DsPlan {
  static constexpr int KQ0 = 0;            // [K;Q] bf16: 2 k-blocks of 128 rows x 128 B
  static constexpr int KQ1 = 32768;
  static constexpr int DO16 = 65536;       // dO fp16 [t][v]: 2 v-blocks of 64 rows x 128 B
  static constexpr int DOS0 = 81920;       // Gamma dO / sqrt(dk), bf16 hi, then lo at +16384;
  static constexpr int DOS1 = 114688;      //   two buffers by chunk parity
  static constexpr int AT = 147456;        // A~ fp16 [t'][t]: 64 rows x 128 B
  static constexpr int TB0 = 155648;       // T fp16 [i][t]: hi, then lo at +8192
  static constexpr int TB1 = 172032;
  static constexpr int DOST = 188416;      // dO fp32 staging, row-major 64 x 512 B
  static constexpr int BYTES = 221184;
  static constexpr int DYN_SMEM = BYTES + 1024;  // slack for 1024-byte alignment
  // tensor-memory columns
  static constexpr uint32_t COL_DS = 0;    // dS^T fp32 (128)
  static constexpr uint32_t COL_DSH = 128; // dS^T bf16 hi (64: two values per column)
  static constexpr uint32_t COL_DSL = 192; // ... lo
  static constexpr uint32_t COL_G = 256;   // Gram (64), then P1
  static constexpr uint32_t COL_A2 = 320;  // P2 (64)
  static constexpr uint32_t COL_DU = 384;  // du^T fp16 hi (32) + lo (32), then (-Gamma beta du')^T bf16
  static constexpr uint32_t COL_DUP = 448; // P3 (64)
  static constexpr uint32_t TMEM_COLS = 512;
};

constexpr int kDsThreads = 512;

__device__ __forceinline__ void ds_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

__global__ void __launch_bounds__(kDsThreads, 1)
gdn_bwd_dstates_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                          const BwdChunkParams p) {
  using P = DsPlan;
  extern __shared__ uint8_t smem_raw[];
  // per token: log-decay prefix b, beta, Gamma / sqrt(dk), gamma / Gamma, -Gamma beta
  __shared__ float s_b[kChunk], s_beta[kChunk], s_sc[kChunk], s_gd[kChunk], s_ngb[kChunk];
  __shared__ float s_gam;
  __shared__ __align__(8) uint64_t s_mb[7];
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, part = warp >> 2;  // lane quarter; column quarter
  const int v = quarter * 32 + lane;              // this thread's tensor-memory lane (value index)

  const int si = blockIdx.x / p.nv, h = blockIdx.x % p.nv, kh = h / (p.nv / p.nk);
  const int s = p.order ? p.order[si] : si;
  int64_t row0, len;
  if (!bc_sequence(p, s, row0, len)) return;
  const int nch = static_cast<int>((len + kChunk - 1) / kChunk);
  const int64_t hrow = static_cast<int64_t>(p.nv) * kDim;

  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = tc::smem_u32(sm);
  const uint32_t mb_kq0 = tc::smem_u32(&s_mb[0]), mb_kq1 = tc::smem_u32(&s_mb[1]);
  const uint32_t mb_a = tc::smem_u32(&s_mb[2]), mb_b = tc::smem_u32(&s_mb[3]), mb_c = tc::smem_u32(&s_mb[4]),
                 mb_d = tc::smem_u32(&s_mb[5]), mb_g = tc::smem_u32(&s_mb[6]);

  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&s_tmem), P::TMEM_COLS);
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 7; ++i) tc::mbar_init(tc::smem_u32(&s_mb[i]), 1);
    tc::mbar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t lanes = tmem + ((static_cast<uint32_t>(quarter) * 32u) << 16);

  // ---- copies one chunk ahead -----------------------------------------------------------
  auto issue_kq = [&](int c) {  // thread 0
    const uint32_t dst = sb + ((c & 1) ? P::KQ1 : P::KQ0);
    const uint32_t mb = (c & 1) ? mb_kq1 : mb_kq0;
    const int32_t y = static_cast<int32_t>(row0 + static_cast<int64_t>(c) * kChunk);
    tc::mbar_arrive_expect_tx(mb, 32768);
    tc::tma_load_2d(dst, &tmap_k, kh * kDim, y, mb);
    tc::tma_load_2d(dst + 16384, &tmap_k, kh * kDim + 64, y, mb);
    tc::tma_load_2d(dst + 8192, &tmap_q, kh * kDim, y, mb);
    tc::tma_load_2d(dst + 16384 + 8192, &tmap_q, kh * kDim + 64, y, mb);
  };
  auto chunk_len = [&](int c) {
    const int64_t rem = len - static_cast<int64_t>(c) * kChunk;
    return static_cast<int>(rem < kChunk ? rem : kChunk);
  };
  auto issue_copies = [&](int c) {  // every thread: T rows (swizzled) and dO rows (staging)
    const int n = chunk_len(c);
    const int64_t r0 = row0 + static_cast<int64_t>(c) * kChunk;
    const uint32_t tb = sb + ((c & 1) ? P::TB1 : P::TB0);
    const uint16_t* tsrc = p.tm + r0 * hrow + h * kDim;
#pragma unroll
    for (int i = 0; i < 1024 / kDsThreads; ++i) {
      const int idx = tid + kDsThreads * i, row = idx >> 4, c8 = idx & 15;
      const int srow = row < n ? row : 0;
      cp_async16(tb + (c8 >> 3) * 8192 + tc::sw128(row, (c8 & 7) * 16), tsrc + srow * hrow + 8 * c8, row < n);
    }
    const float* dsrc = p.dout + r0 * hrow + h * kDim;
#pragma unroll
    for (int i = 0; i < 2048 / kDsThreads; ++i) {
      const int idx = tid + kDsThreads * i, row = idx >> 5, c4 = idx & 31;
      const int srow = row < n ? row : 0;
      cp_async16(sb + P::DOST + row * 512 + c4 * 16, dsrc + srow * hrow + 4 * c4, row < n);
    }
    tc::cp_async_commit();
  };

  bool ok = true;
  uint32_t kq_phase = 0;  // thread 0: parity of the next wait on each K/Q buffer
  auto wait_mb = [&](uint32_t mb, uint32_t parity) {
    bool w = ok && tc::mbar_wait_timed(mb, parity, kWaitLimitNs);
    w = __syncthreads_and(w) != 0;
    if (!w && ok && tid == 0) atomicOr(p.status, kStatusTimeout);
    ok = w;
    tc::fence_after_sync();
    return w;
  };
  auto sync_tmem = [&]() {
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  };

  // Gates of chunk c into registers (warp 0), fetched with the chunk's other copies
  float fg0 = 0.f, fg1 = 0.f, fb0 = 0.f, fb1 = 0.f;
  auto fetch_gates = [&](int c) {
    const int n = chunk_len(c);
    const int64_t r0 = row0 + static_cast<int64_t>(c) * kChunk;
    const int t0 = 2 * lane, t1 = t0 + 1;
    fg0 = t0 < n ? p.g[(r0 + t0) * p.g_stride + h] : 0.f;
    fg1 = t1 < n ? p.g[(r0 + t1) * p.g_stride + h] : 0.f;
    fb0 = t0 < n ? p.beta[(r0 + t0) * p.beta_stride + h] : 0.f;
    fb1 = t1 < n ? p.beta[(r0 + t1) * p.beta_stride + h] : 0.f;
  };
  // Per-token factors of the fetched chunk (warp 0) and its dO operands from the staged rows.
  auto gates = [&]() {
    const int t0 = 2 * lane, t1 = t0 + 1;
    const float be0 = fb0, be1 = fb1;
    const GatePrefix gp = gate_prefix(fg0, fg1);
    const float e0 = __expf(gp.gca), e1 = __expf(gp.gcb);
    s_b[t0] = gp.gca;
    s_b[t1] = gp.gcb;
    s_beta[t0] = be0;
    s_beta[t1] = be1;
    s_sc[t0] = e0 * kInvSqrtD;
    s_sc[t1] = e1 * kInvSqrtD;
    s_gd[t0] = __expf(gp.last - gp.gca);
    s_gd[t1] = __expf(gp.last - gp.gcb);
    s_ngb[t0] = -e0 * be0;
    s_ngb[t1] = -e1 * be1;
    if (lane == 0) s_gam = __expf(gp.last);
  };
  auto convert_do = [&](int c) {  // dO as fp16 and (Gamma / sqrt(dk)) dO as bf16 hi + lo
    uint8_t* dos = sm + ((c & 1) ? P::DOS1 : P::DOS0);
#pragma unroll
    for (int i = 0; i < 1024 / kDsThreads; ++i) {
      const int idx = tid + kDsThreads * i, row = idx >> 4, c8 = idx & 15;
      const float4 a = *reinterpret_cast<const float4*>(sm + P::DOST + row * 512 + c8 * 32);
      const float4 b = *reinterpret_cast<const float4*>(sm + P::DOST + row * 512 + c8 * 32 + 16);
      const float f[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      const float sc = s_sc[row];
      uint32_t h16[4], bh[4], bl[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h16[e] = pack_half2(f[2 * e], f[2 * e + 1]);
        split_bf162(sc * f[2 * e], sc * f[2 * e + 1], bh[e], bl[e]);
      }
      const uint32_t o = (c8 >> 3) * 8192 + tc::sw128(row, (c8 & 7) * 16);
      *reinterpret_cast<uint4*>(sm + P::DO16 + o) = make_uint4(h16[0], h16[1], h16[2], h16[3]);
      *reinterpret_cast<uint4*>(dos + o) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
      *reinterpret_cast<uint4*>(dos + 16384 + o) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
    }
  };
  // The state gradient in COL_DS is dS_end of chunk c: stage it (fp16, [k][v], in the
  // dO staging buffer, which is free until the next chunk's copies), make its bf16 hi + lo
  // copy (chunk c's P2 operand) and decay it by chunk c's gamma (for P4).
  auto state_pass = [&](const uint32_t (&x)[32]) {
    const float gam = s_gam;
    __half* stage = reinterpret_cast<__half*>(sm + P::DOST) + v;
    uint32_t hi[16], lo[16], y[32];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float f0 = __uint_as_float(x[2 * e]), f1 = __uint_as_float(x[2 * e + 1]);
      stage[(part * 32 + 2 * e) * kDim] = __float2half_rn(f0);
      stage[(part * 32 + 2 * e + 1) * kDim] = __float2half_rn(f1);
      split_bf162(f0, f1, hi[e], lo[e]);
      y[2 * e] = __float_as_uint(gam * f0);
      y[2 * e + 1] = __float_as_uint(gam * f1);
    }
    tc::tmem_st16u(lanes + P::COL_DSH + part * 16, hi);
    tc::tmem_st16u(lanes + P::COL_DSL + part * 16, lo);
    tc::tmem_st32(lanes + P::COL_DS + part * 32, y);
    tc::tmem_st_wait();
  };

  // Gram of chunk c (thread 0), once its K/Q tile has landed; false on expiry
  auto issue_gram = [&](int c) {
    const int b = c & 1;
    const bool w = tc::mbar_wait_timed(b ? mb_kq1 : mb_kq0, (kq_phase >> b) & 1u, kWaitLimitNs);
    kq_phase ^= 1u << b;
    if (!w) return false;
    tc::fence_after_sync();
    // descriptors step by adding (byte offset >> 4) to the start-address field
    const uint64_t dkq = tc::desc_sw128(sb + (b ? P::KQ1 : P::KQ0), 16, 1024);
    constexpr uint32_t id_g = tc::idesc_f16(128, 64, tc::kBF16, false, false);
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      const uint64_t a = dkq + (((st >> 2) * 16384 + (st & 3) * 32) >> 4);
      tc::mma_f16(tmem + P::COL_G, a, a, id_g, st > 0);
    }
    tc::mma_commit(mb_g);
    return true;
  };
  // A~ of chunk c from the Gram (lanes 64-127, rows t'), 16 columns per warp
  auto a_tilde = [&](int c) {
    if (quarter < 2) return;
    const int n = chunk_len(c);
    const int tp = v - 64;
    const float bt = s_b[tp];
    float d[16];
    tc::tmem_ld16(lanes + P::COL_G + part * 16, d);
    tc::tmem_ld_wait();
    uint32_t pk[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j0 = part * 16 + 2 * e, j1 = j0 + 1;
      const float a0 = (j0 <= tp && tp < n) ? d[2 * e] * __expf(bt - s_b[j0]) * kInvSqrtD : 0.f;
      const float a1 = (j1 <= tp && tp < n) ? d[2 * e + 1] * __expf(bt - s_b[j1]) * kInvSqrtD : 0.f;
      pk[e] = pack_half2(a0, a1);
    }
    *reinterpret_cast<uint4*>(sm + P::AT + tc::sw128(tp, part * 32)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    *reinterpret_cast<uint4*>(sm + P::AT + tc::sw128(tp, part * 32 + 16)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  };
  auto issue_p1 = [&]() {  // P1 = dO^T A~ onto the Gram columns (thread 0)
    constexpr uint32_t id_1 = tc::idesc_f16(128, 64, tc::kF16, true, true);
    const uint64_t ddo = tc::desc_sw128(sb + P::DO16, 8192, 1024), dat = tc::desc_sw128(sb + P::AT, 8192, 1024);
#pragma unroll
    for (int st = 0; st < 4; ++st) tc::mma_f16(tmem + P::COL_G, ddo + st * 128, dat + st * 128, id_1, st > 0);
    tc::mma_commit(mb_b);
  };
  uint32_t g_count = 0;  // completions of mb_g waited so far

  // ---- the last chunk: operands, dS_end = dL/dS_T (or zero), its Gram, A~ and P1 --------------
  if (nch > 0) {
    if (tid == 0) {
      issue_kq(nch - 1);
      if (nch > 1) issue_kq(nch - 2);
    }
    issue_copies(nch - 1);
    if (warp == 0) {
      fetch_gates(nch - 1);
      gates();
    }
    tc::cp_async_wait_all();
    __syncthreads();
    convert_do(nch - 1);
    const float* d0 = p.dst ? p.dst + (static_cast<int64_t>(s) * p.nv + h) * kDim * kDim : nullptr;
    uint32_t x[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) x[e] = __float_as_uint(d0 ? d0[(part * 32 + e) * kDim + v] : 0.f);
    __syncthreads();  // the staging buffer's dO rows are converted
    state_pass(x);
    tc::fence_proxy_async();
    sync_tmem();
    if (tid == 0 && !issue_gram(nch - 1)) {
      atomicOr(p.status, kStatusTimeout);
      ok = false;
    }
    if (wait_mb(mb_g, g_count++ & 1u)) {
      a_tilde(nch - 1);
      tc::fence_proxy_async();
      sync_tmem();
      if (tid == 0) issue_p1();
    }
  } else {
    const float* d0 = p.dst ? p.dst + (static_cast<int64_t>(s) * p.nv + h) * kDim * kDim : nullptr;
    uint32_t x[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) x[e] = __float_as_uint(d0 ? d0[(part * 32 + e) * kDim + v] : 0.f);
    tc::tmem_st32(lanes + P::COL_DS + part * 32, x);
    tc::tmem_st_wait();
    sync_tmem();
  }

  for (int it = 0; it < nch && ok; ++it) {
    const int c = nch - 1 - it;
    const int n = chunk_len(c);
    const int64_t r0 = row0 + static_cast<int64_t>(c) * kChunk;
    const uint32_t ph = static_cast<uint32_t>(it) & 1u;

    // ---- P2 = dS^T K^T; the previous chunk's copies ----------------------------------------
    if (tid == 0) {
      constexpr uint32_t id_2 = tc::idesc_f16(128, 64, tc::kBF16, false, false);
      const uint64_t dkq = tc::desc_sw128(sb + ((c & 1) ? P::KQ1 : P::KQ0), 16, 1024);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        const uint64_t bk = dkq + (((st >> 2) * 16384 + (st & 3) * 32) >> 4);
        tc::mma_f16_ts(tmem + P::COL_A2, tmem + P::COL_DSH + st * 8, bk, id_2, st > 0);
        tc::mma_f16_ts(tmem + P::COL_A2, tmem + P::COL_DSL + st * 8, bk, id_2, 1);
      }
      tc::mma_commit(mb_a);
    }
    {  // this chunk's dS_end, staged by the state pass, out to global memory
      __half* dst = p.dsbuf + (bc_slot(row0, s, c) * p.nv + h) * kDim * kDim;
#pragma unroll
      for (int i = 0; i < 2048 / kDsThreads; ++i) {
        const int idx = tid + kDsThreads * i;
        reinterpret_cast<uint4*>(dst)[idx] = *reinterpret_cast<const uint4*>(sm + P::DOST + idx * 16);
      }
    }
    __syncthreads();
    if (c > 0) {
      issue_copies(c - 1);  // the staging and T buffer c - 1 uses are free
      if (warp == 0) fetch_gates(c - 1);
    }
    // P1 of this chunk was issued one step earlier
    if (!wait_mb(mb_b, ph) || !wait_mb(mb_a, ph)) break;

    // ---- du^T = P1 + (gamma / Gamma_t) P2, zero past the chunk's end, as fp16 hi + lo ---------
    {
      float a1[16], a2[16];
      tc::tmem_ld16(lanes + P::COL_G + part * 16, a1);
      tc::tmem_ld16(lanes + P::COL_A2 + part * 16, a2);
      tc::tmem_ld_wait();
      uint32_t hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t0 = part * 16 + 2 * e, t1 = t0 + 1;
        const float x0 = t0 < n ? fmaf(s_gd[t0], a2[2 * e], a1[2 * e]) : 0.f;
        const float x1 = t1 < n ? fmaf(s_gd[t1], a2[2 * e + 1], a1[2 * e + 1]) : 0.f;
        split_half2(x0, x1, hi[e], lo[e]);
      }
      ds_st8(lanes + P::COL_DU + part * 8, hi);
      ds_st8(lanes + P::COL_DU + 32 + part * 8, lo);
      tc::tmem_st_wait();
    }
    sync_tmem();

    // ---- P3 = du^T T; the previous chunk's Gram onto the columns P1 has left ------------------
    bool gram_ok = true;
    if (tid == 0) {
      constexpr uint32_t id_3 = tc::idesc_f16(128, 64, tc::kF16, false, true);
      const uint64_t dtb = tc::desc_sw128(sb + ((c & 1) ? P::TB1 : P::TB0), 8192, 1024);
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint64_t th = dtb + st * 128, tl = dtb + 512 + st * 128;
        tc::mma_f16_ts(tmem + P::COL_DUP, tmem + P::COL_DU + st * 8, th, id_3, st > 0);
        tc::mma_f16_ts(tmem + P::COL_DUP, tmem + P::COL_DU + st * 8, tl, id_3, 1);
        tc::mma_f16_ts(tmem + P::COL_DUP, tmem + P::COL_DU + 32 + st * 8, th, id_3, 1);
      }
      tc::mma_commit(mb_c);
      if (c > 0) gram_ok = issue_gram(c - 1);
      if (!gram_ok) atomicOr(p.status, kStatusTimeout);
    }
    if (!gram_ok) ok = false;
    if (!wait_mb(mb_c, ph)) break;

    // ---- du' and dV rows out; (-Gamma beta du')^T as bf16 hi + lo over du^T's columns --------
    {
      float d[16];
      tc::tmem_ld16(lanes + P::COL_DUP + part * 16, d);
      tc::tmem_ld_wait();
      __half* dup = p.dubuf + r0 * hrow + h * kDim + v;
      float* dvp = p.dv + r0 * hrow + h * kDim + v;
      uint32_t hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t0 = part * 16 + 2 * e, t1 = t0 + 1;
        const float x0 = d[2 * e], x1 = d[2 * e + 1];
        if (t0 < n) {
          dup[t0 * hrow] = __float2half_rn(x0);
          dvp[t0 * hrow] = s_beta[t0] * x0;
        }
        if (t1 < n) {
          dup[t1 * hrow] = __float2half_rn(x1);
          dvp[t1 * hrow] = s_beta[t1] * x1;
        }
        split_bf162(s_ngb[t0] * x0, s_ngb[t1] * x1, hi[e], lo[e]);
      }
      ds_st8(lanes + P::COL_DU + part * 8, hi);
      ds_st8(lanes + P::COL_DU + 32 + part * 8, lo);
      tc::tmem_st_wait();
    }
    sync_tmem();

    // ---- P4: dS^T += (Gamma dO / sqrt(dk))^T Q + (-Gamma beta du')^T K ----------------------
    if (tid == 0) {
      constexpr uint32_t id_s = tc::idesc_f16(128, 128, tc::kBF16, true, true);
      constexpr uint32_t id_t = tc::idesc_f16(128, 128, tc::kBF16, false, true);
      const uint64_t dkq = tc::desc_sw128(sb + ((c & 1) ? P::KQ1 : P::KQ0), 16384, 1024);
      const uint64_t dds = tc::desc_sw128(sb + ((c & 1) ? P::DOS1 : P::DOS0), 8192, 1024);
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const uint64_t bq = dkq + 512 + st * 128, bk = dkq + st * 128;
        tc::mma_f16(tmem + P::COL_DS, dds + st * 128, bq, id_s, 1);
        tc::mma_f16(tmem + P::COL_DS, dds + 1024 + st * 128, bq, id_s, 1);
        tc::mma_f16_ts(tmem + P::COL_DS, tmem + P::COL_DU + st * 8, bk, id_t, 1);
        tc::mma_f16_ts(tmem + P::COL_DS, tmem + P::COL_DU + 32 + st * 8, bk, id_t, 1);
      }
      tc::mma_commit(mb_d);
    }
    // meanwhile, the previous chunk's chain-free work: factors, dO operands (its own scaled
    // buffer; the fp16 dO tile's last reader, this chunk's P1, is done), A~ and P1
    if (c > 0) {
      tc::cp_async_wait_all();
      if (warp == 0) gates();
      __syncthreads();
      convert_do(c - 1);
      if (!wait_mb(mb_g, g_count++ & 1u)) break;
      a_tilde(c - 1);
      tc::fence_proxy_async();
      sync_tmem();
      if (tid == 0) issue_p1();
    }
    if (!wait_mb(mb_d, ph)) break;

    // ---- dS_end of the previous chunk: stored, copied for its P2, decayed for its P4; the
    //      K/Q of the chunk after it into this chunk's buffer ----------------------------------
    if (c > 0) {
      if (tid == 0 && c > 1) issue_kq(c - 2);
      uint32_t x[32];
      tc::tmem_ld32(lanes + P::COL_DS + part * 32, x);
      tc::tmem_ld_wait();
      state_pass(x);
    }
    sync_tmem();
  }

  if (ok && p.dh0) {  // dL/dS_0, [k][v]
    float* d = p.dh0 + (static_cast<int64_t>(s) * p.nv + h) * kDim * kDim + v;
    uint32_t x[32];
    tc::tmem_ld32(lanes + P::COL_DS + part * 32, x);
    tc::tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 32; ++e) d[(part * 32 + e) * kDim] = __uint_as_float(x[e]);
  }
  tc::cp_async_wait_all();
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

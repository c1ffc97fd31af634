// Fused chunked gated-delta-rule prefill spine kernel for sm_103a
// (warp-specialised).
//
// One CTA owns one (sequence, v-head) and walks its 64-token chunks in order.
// With T diag(beta) of every chunk already solved by the chunk-parallel WY
// kernel, it runs the rest of the GDN prefill op (ssm_gdn_a3.rs, doc comment of
// `gdn_prefill_fla`) on chip, split between three roles:
//
//   producer (8 warps), chunk c+1:  WY products and operand tiles
//     U = (T diag beta) V;  W = (T diag beta) diag(e^gc) K;
//     e^gc Q / sqrt(dk), e^{gc_last-gc} K, and
//     A_ij = e^{gc_i-gc_j} q_i.k_j / sqrt(dk) for j <= i
//   consumer (4 warps), chunk c:    state spine and output
//     u = U - W S;  S <- e^{gc_last} S + (diag(e^{gc_last-gc}) K)^T u;
//     O = diag(e^gc) Q S / sqrt(dk) + A u          (S: state entering chunk c)
//   two issuer warps (one thread each), driven by readiness barriers the other
//     warps arrive on: the producer's MMAs and all TMA copies, and the spine's
//     MMAs (tcgen05.mma issue costs tens of cycles per instruction, so two
//     streams keep the tensor pipe fed better than one)
//
// The spine is computed transposed, with the value index v on the 128 tensor
// memory lanes: u^T = U^T - S^T W^T, dS^T = u^T Kd, O^T = S^T Q~^T + u^T A^T.
// Every spine product is then an M=128 tcgen05 MMA whose A operand (S^T or
// u^T, fp16) is read straight from tensor memory, and each consumer thread
// owns one v column, so the output rows are written with coalesced stores.
// The fp32 state S^T lives in tensor memory as the accumulator of dS^T.
//
// Precision: T diag(beta) arrives as an fp16 hi + lo pair; U and W multiply
// both halves with fp16 copies of V (exact for |v| < 65504) and of e^gc K.
// The spine uses fp16 operands with fp32 accumulation, and A u uses fp16
// hi + lo splits of both factors (the largest outputs must be accurate to
// ~1e-4 before the final bf16 rounding).
//
// The WY kernel leaves each chunk's T diag(beta) rows in the output rows of
// the same tokens and head; this kernel reads them (by TMA) before it writes
// the outputs there. Tail rows of a chunk (past the end of the sequence) are
// treated as k = v = 0, g = 0: their T diag(beta) rows, which belong to other
// tokens, only reach columns of u^T that are zeroed before use, and their
// outputs are not stored. Every wait on an mbarrier is bounded; on expiry the
// CTA records a status bit and unwinds. A non-finite output or final state
// (an operand outside the fp16 range) sets another status bit.
//
// Ordering. Every barrier is waited on by parity, so no barrier may complete
// twice before each of its waiters has seen the earlier phase. A barrier that
// completes once per chunk is either single (when its next completion is
// caused, through some chain of waits, by each of its waiters having passed
// the wait for the current chunk) or doubled by chunk parity (when only its
// completion two chunks later is caused that way). The per-barrier argument
// sits next to each barrier's declaration in Ctx.
#pragma once
#include "gdn_common.cuh"

namespace gdn {

constexpr int kConsumerWarps = 4;
constexpr int kProducerWarps = 8;
constexpr int kIssuerWarps = 2;
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps + kIssuerWarps);
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr uint32_t kBarProducer = 1;  // named barrier ids
constexpr uint32_t kBarConsumer = 2;
constexpr uint32_t kBarNorm = 3;      // producer, fused prologue: row norms published

struct ChunkParams {
  const float* g;
  void* state;                // float[B][nv][128][128], or float*[B] when state_is_table
  __nv_bfloat16* out;
  const int32_t* cu_seqlens;  // null for dense batches
  const int32_t* order;       // varlen: sequences by decreasing length (null: identity)
  unsigned* status;
  int64_t g_stride, out_stride;
  int B, T, nk, nv;
  int state_is_table;
  int qk_l2norm;              // fused prologue: normalise every q and k row first
  // Segment table (null: none). Entry s = {first row, length, mode, 0} of the row range
  // CTA slot s runs, for the segment-parallel schedule of long sequences; mode bit 0
  // skips the output rows (the range's T diag(beta) rows stay in place for a later run),
  // bit 1 runs it with v = 0 (the state map's linear part).
  const int32_t* seg;
  // Dense batches without a segment table: the chunk range [chunk_begin, chunk_begin +
  // chunk_count) of every sequence (chunk_count 0: to the sequence's end). The state is
  // read at the range's start and written at its end, so consecutive ranges run one
  // after the other carry it in place.
  int chunk_begin, chunk_count;
  // Test hooks, read only by the test instantiation (kTest = true): a wait limit in
  // nanoseconds in place of kWaitLimitNs, a consumer delay in nanoseconds before the
  // hand-off wait of every odd chunk (so the producer runs ahead), and a chunk whose
  // hand-off arrival the producer skips (-1: none), so that bounded waits expire.
  int64_t test_wait_ns, test_delay_ns;
  int test_skip_chunk;
  // The backward's forward chain (kBwd = true): the WY kernel hands over T itself (not
  // T diag(beta)), so the producer scales the tile's columns by beta in place; each
  // chunk's entry state S0 and u are stored as fp16 for the gradient kernels; the
  // carried-in state is only read.
  const float* beta;
  int64_t beta_stride;
  __half* s0buf;  // [slots][nv][128][128]: S0 of chunk c in slot row0 / 64 + s + c, [k][v]
  __half* ubuf;   // [rows][nv][128]: u
};
constexpr int kSegNoOutput = 1;
constexpr int kSegZeroValues = 2;

// Shared-memory plan (bytes from a 1024-aligned base). Operand tiles are
// row-major 16-bit tiles stored as 64-column blocks of 128-byte swizzled rows
// (the layout TMA writes); the same bytes serve as a K-major operand whose
// rows are M/N, or as an MN-major operand whose rows are K.
struct Plan {
  static constexpr int KQ0 = 0;            // raw bf16 [K;Q] (2 blocks x 128 rows), chunk parity 0; K becomes
  static constexpr int KQ1 = KQ0 + 32768;  //   fp16 e^gc K in place; ... parity 1
  static constexpr int V0 = KQ1 + 32768;   // raw bf16 V (2 blocks x 64 rows), made fp16 in place
  static constexpr int V1 = V0 + 16384;
  static constexpr int TB = V1 + 16384;    // fp16 T diag(beta) hi, lo (64 x 64 each, rows t)
  static constexpr int W16 = TB + 16384;   // fp16 -W^T, rows k (128 x 64)
  static constexpr int QT = W16 + 16384;   // fp16 e^gc Q / sqrt(dk), rows t (64 x 128)
  static constexpr int KD0 = QT + 16384;   // fp16 e^{gc_last-gc} K, rows t, chunk parity 0
  static constexpr int KD1 = KD0 + 16384;  // ... chunk parity 1
  static constexpr int A0 = KD1 + 16384;   // fp16 A hi, lo (64 x 64 each), chunk parity 0
  static constexpr int A1 = A0 + 16384;    // ... chunk parity 1
  static constexpr int BYTES = A1 + 16384;
  static constexpr int DYN_SMEM = BYTES + 1024;  // slack for 1024-byte alignment
  static_assert(DYN_SMEM <= 227 * 1024 - 8192, "shared memory budget");

  // Tensor-memory columns (512 x 32-bit, lanes = rows).
  static constexpr uint32_t COL_S = 0;     // fp32 S^T [v][k], 128 columns
  static constexpr uint32_t COL_U = 128;   // fp32 U^T -> u^T [v][t], 2 x 64 columns (chunk parity)
  static constexpr uint32_t COL_GW = 256;  // fp32 [K;Q] K^T [m][j], then W^T [k][t], 64 columns
  static constexpr uint32_t COL_O = 320;   // fp32 O^T [v][t], 64 columns
  static constexpr uint32_t COL_ST = 384;  // fp16 pairs S^T [v][k], 64 columns
  static constexpr uint32_t COL_UT = 448;  // fp16 pairs u^T hi [v][t] (32 columns), then lo (32)
  static constexpr uint32_t TMEM_COLS = 512;
};

// Per-CTA state shared by the two warp groups.
struct Ctx {
  uint8_t* sm;       // 1024-aligned dynamic shared memory
  uint32_t sbase;    // its shared-window address
  uint32_t tmem;     // tensor-memory base address
  int64_t row0, len; // first packed row and length of the sequence
  int nchunks, h, kh;
  int store_out, zero_v;  // segment modes (1, 0 outside segment runs)
  float* state;      // this (sequence, head)'s fp32 [128][128] state, k-major
  // producer-side per-token scales, two gate sets by chunk parity ([2][64] each)
  float *s_gc, *s_eg, *s_egq, *s_edec;  // gc, e^gc, e^gc / sqrt(dk), e^{gc_last - gc}
  float *s_E, *s_F;     // e^{gc - m}, e^{m - gc} about the chunk's mid gate m
  float *s_rq, *s_rk;   // fused prologue: 1 / |q_t|, 1 / |k_t| of the current chunk
  float* s_qpart;       // fused prologue with outputs: [4][64] partial sums of q_t^2
  // ... and 1 / |q_t|, 1 / |k_t| by chunk index mod 3 ([3][64] each), read by the
  // consumer's store and u split of that chunk. The producer writes chunk c+3's slot after
  // its wait on c2(c+1) at the top of chunk c+3; spine2(c+1) is issued after the
  // consumer's usp(c+1), which follows its store and u split of chunk c.
  float* s_rq3;
  float* s_rk3;
  int* s_fast;          // [2] 1 when the chunk's gate range allows the factorised decays
  float* s_gstage;      // [2][64] g of a chunk, staged by cp.async
  float *s_bstage, *s_bv;  // backward's forward chain: beta staged, and beta of a gate set
  float* s_elast;       // [3] e^{gc_last} by chunk index mod 3 (read by the consumer)
  volatile int* s_abort;
  // Barriers and why none can complete twice ahead of a waiter (chunk c; "->" is
  // "happens before, through waits"):
  //   kq[b], v[b]  copies of chunk c+2 are issued after qrdy[b](c), which every
  //                waiting producer warp signals after its own wait.
  //   t            waited on by the producer-side issuer only, in program order.
  //   g            Gram(c+1) is issued after wrd(c), signalled after both producer waits.
  //   uw           U/W(c+1) need krdy(c+1), signalled after the producer's uw(c) wait.
  //   c1           spine1(c+1) needs hand(c+1) (producer, after its c1(c) wait) and
  //                strdy(c+1) (consumer, after its c1(c) wait).
  //   c2[b]        spine2(c+2) needs usp(c+2) (consumer, after its c2(c) wait) and
  //                hand(c+2) (producer, after its c2[b](c) wait at the top of c+2).
  //   hand[b]      doubled: hand(c+1) may arrive while the consumer still finishes
  //                chunk c-1 (it needs only c1(c) and c2(c-1)); hand(c+2) needs
  //                c2[b](c), which needs the consumer's usp(c) and the spine
  //                issuer's spine2(c), both after their hand(c) waits.
  //   cu[b]        consumer cu(c) -> needs spine1(c) -> hand(c) -> uw(c) -> U(c) MMAs,
  //                issued after the issuer's cu[b](c-2) wait.
  //   vrdy, krdy   the producer's chunk c+1 starts after uw(c), committed after the
  //                issuer's vrdy(c) and krdy(c) waits.
  //   qrdy[b]      doubled: without outputs nothing orders qrdy(c+1) after the
  //                issuer's qrdy(c) wait; qrdy(c+2) follows the producer's uw(c+1)
  //                wait, and uw(c+1) is committed after the issuer's qrdy(c) wait.
  //   wrd          wrd(c+1) follows uw(c+1) -> W(c+1) MMAs, issued after wrd(c).
  //   strdy        strdy(c+1) follows the consumer's c2(c) wait -> spine2(c), issued
  //                after the spine issuer's strdy(c) wait.
  //   usp          usp(c+1) follows c1(c+1) -> spine1(c+1), issued after usp(c).
  uint32_t mb_kq0, mb_kq1, mb_v0, mb_v1, mb_t, mb_g, mb_uw, mb_c1, mb_c20, mb_c21, mb_hand0, mb_hand1, mb_cu0, mb_cu1;
  // readiness for the issuer (one arrival per warp): V is fp16 (4), e^gc K is done and
  // Q K^T read (8), Q~ is done (8, by chunk parity), W read (8), S^T ready and O^T
  // read (4), u split (4)
  uint32_t mb_vrdy, mb_krdy, mb_qrdy0, mb_qrdy1, mb_wrd, mb_strdy, mb_usp;
};

// All threads of a group wait on one mbarrier phase; the outcome is made
// uniform across the group so that it can leave its loop together.
__device__ __forceinline__ bool group_wait(const Ctx& x, const ChunkParams& p, uint32_t mbar, uint32_t parity,
                                           uint32_t bar_id, uint32_t nthreads, bool leader, uint64_t lim) {
  bool ok = (*x.s_abort == 0) && tc::mbar_wait_timed(mbar, parity, lim);
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

// Wait limit: the 2 s default, or the test instantiation's own.
template <bool kTest>
__device__ __forceinline__ uint64_t wait_limit(const ChunkParams& p) {
  if constexpr (kTest) return static_cast<uint64_t>(p.test_wait_ns);
  else return kWaitLimitNs;
}

// ---------------------------------------------------------------------------------
// Producer: the operand tiles of each chunk, one chunk ahead of the consumer
// (the issuer runs its MMAs). Warp 4 also scans the gates of the chunk after,
// so every chunk starts with its gate set ready.
// ---------------------------------------------------------------------------------
template <bool kOut, bool kNorm, bool kTest, bool kBwd>
__device__ __forceinline__ void producer_role(const Ctx& x, const ChunkParams& p, int ptid) {
  using P = Plan;
  const uint64_t lim = wait_limit<kTest>(p);
  const int pw = ptid >> 5, lane = ptid & 31;
  const int quad = pw & 3;   // tensor-memory lane quarter of this warp
  const int half = pw >> 2;  // which half of a 64-column accumulator it reads
  const bool leader = ptid == 0;
  const int hq = half * 64 + (quad & 1) * 32 + lane;  // index among the 4 warps of its lane-quarter pair
  uint8_t* sm = x.sm;

  // gates of chunk c (one warp, producer warp 4): the log-gates of tokens 2*lane and
  // 2*lane+1 are copied to stage c & 1 by cp.async two chunks ahead, then scanned
  // into gate set c & 1 one chunk ahead
  auto load_gates = [&](int c) {
    float* st = x.s_gstage + (c & 1) * kChunk;
    float* sb = x.s_bstage + (c & 1) * kChunk;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tt = 2 * lane + e;
      const int64_t t = static_cast<int64_t>(c) * kChunk + tt;
      if (t < x.len) {
        tc::cp_async_4(tc::smem_u32(st + tt), p.g + (x.row0 + t) * p.g_stride + x.h);
        if constexpr (kBwd) tc::cp_async_4(tc::smem_u32(sb + tt), p.beta + (x.row0 + t) * p.beta_stride + x.h);
      } else {
        st[tt] = 0.f;
        if constexpr (kBwd) sb[tt] = 0.f;
      }
    }
    tc::cp_async_commit();
  };
  auto scan_gates = [&](int c) {  // after the copy of chunk c's gates has completed
    const int gs = (c & 1) * kChunk;
    __syncwarp();
    const float* st = x.s_gstage + gs;
    const GatePrefix gp = gate_prefix(st[2 * lane], st[2 * lane + 1]);
    // e^{gc_i - gc_j} = E_i F_j with E = e^{gc - m}, F = e^{m - gc} and m the
    // middle of the chunk's gate range
    const float mid = 0.5f * (gp.first + gp.last);
    x.s_gc[gs + 2 * lane] = gp.gca;
    x.s_gc[gs + 2 * lane + 1] = gp.gcb;
    x.s_eg[gs + 2 * lane] = __expf(gp.gca);
    x.s_eg[gs + 2 * lane + 1] = __expf(gp.gcb);
    x.s_egq[gs + 2 * lane] = __expf(gp.gca) * kInvSqrtD;
    x.s_egq[gs + 2 * lane + 1] = __expf(gp.gcb) * kInvSqrtD;
    x.s_edec[gs + 2 * lane] = __expf(gp.last - gp.gca);
    x.s_edec[gs + 2 * lane + 1] = __expf(gp.last - gp.gcb);
    x.s_E[gs + 2 * lane] = __expf(gp.gca - mid);
    x.s_E[gs + 2 * lane + 1] = __expf(gp.gcb - mid);
    x.s_F[gs + 2 * lane] = __expf(mid - gp.gca);
    x.s_F[gs + 2 * lane + 1] = __expf(mid - gp.gcb);
    if constexpr (kBwd) {  // beta of the gate set, for the T diag(beta) pass
      x.s_bv[gs + 2 * lane] = x.s_bstage[gs + 2 * lane];
      x.s_bv[gs + 2 * lane + 1] = x.s_bstage[gs + 2 * lane + 1];
    }
    if (lane == 0) {
      x.s_elast[c % 3] = __expf(gp.last);
      x.s_fast[c & 1] = (gp.first - gp.last) <= kFactorisedRange;
    }
  };
  auto fail = [&]() {
    *x.s_abort = 1;
    atomicOr(p.status, kStatusTimeout);
  };
  // one arrival per warp on a readiness barrier of the issuer, after this warp's
  // shared-memory writes and tensor-memory reads
  auto signal = [&](uint32_t mbar) {
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(mbar);
  };

  if (pw == 4) {
    load_gates(0);
    tc::cp_async_wait_all();
    scan_gates(0);
    if (x.nchunks > 1) load_gates(1);
  }
  tc::named_barrier(kBarProducer, kProducerThreads);
  bool ok = true;

  for (int c = 0; c < x.nchunks; ++c) {
    const int b = c & 1;
    const int gs = b * kChunk;  // this chunk's gate set
    const uint32_t use = (c >> 1) & 1;  // phase parity of this chunk's double-buffered tiles
    const int64_t rem = x.len - static_cast<int64_t>(c) * kChunk;
    const int clen = rem < kChunk ? static_cast<int>(rem) : kChunk;
    const uint32_t kq_off = b ? P::KQ1 : P::KQ0;
    const uint32_t kd_off = b ? P::KD1 : P::KD0;
    const uint32_t v_off = b ? P::V1 : P::V0;
    const uint32_t a_off = b ? P::A1 : P::A0;

    // ---- the Gram MMA of this chunk is issued by the issuer once its tile lands ------
    // this chunk's Kd and A buffers were last read by the spine of chunk c-2
    ok = true;
    float rk_own = 1.f;  // fused prologue with outputs: 1 / |k_t| of row t = ptid % 64
    if (c >= 2) ok = (*x.s_abort == 0) && tc::mbar_wait_timed(b ? x.mb_c21 : x.mb_c20, ((c - 2) >> 1) & 1, lim);

    if (quad < 2) {
      // ---- V -> fp16 in place (rows t; tail rows zeroed), lane quarters 0, 1 -----------
      ok = ok && (*x.s_abort == 0) && tc::mbar_wait_timed(b ? x.mb_v1 : x.mb_v0, use, lim);
      if (ok) {
#pragma unroll 1
        for (int r0 = 0; r0 < 8; r0 += 4) {
          uint4 raw[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int it = hq + (r0 + r) * 128, t = it & 63, cc = it >> 6;
            raw[r] = *reinterpret_cast<const uint4*>(sm + v_off + (cc >> 3) * 8192 + tc::sw128(t, (cc & 7) * 16));
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int it = hq + (r0 + r) * 128, t = it & 63, cc = it >> 6;
            float f[8];
            unpack_bf16x8(raw[r], f);
            *reinterpret_cast<uint4*>(sm + v_off + (cc >> 3) * 8192 + tc::sw128(t, (cc & 7) * 16)) =
                t < clen && !x.zero_v ? pack_half8(f, 1.f) : make_uint4(0, 0, 0, 0);
          }
        }
      }
      signal(x.mb_vrdy);  // V is fp16: the U MMAs may go
      if constexpr (kNorm && kOut) {
        // fused prologue: |k_t|^2 is the diagonal of the Gram's K K^T half (tensor-memory
        // lanes 0-63). Every warp of lane quarters 0 and 1 reads the 32 rows t = quad * 32 +
        // lane, which are the rows its threads convert below (t = ptid % 64), and keeps
        // 1 / |k_t| in a register; the first warp of each quarter also publishes it for
        // lane quarters 2-3 and the consumer, then all arrive without waiting. Only e^gc K
        // (the W operand) takes 1 / |k_t| here; A and Kd are formed from the raw keys, and
        // the consumer scales column t of u by 1 / |k_t| instead (S^T += u^T Kd and
        // O^T += u^T A^T each have exactly one factor indexed by t)
        ok = ok && (*x.s_abort == 0) && tc::mbar_wait_timed(x.mb_g, b, lim);
        tc::fence_after_sync();
        if (ok) {
          uint32_t d[32];
          tc::tmem_ld32(x.tmem + ((quad * 32u) << 16) + P::COL_GW + quad * 32, d);
          tc::tmem_ld_wait();
          float ss = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) ss = (e == lane) ? __uint_as_float(d[e]) : ss;
          rk_own = 1.f / sqrtf(ss + kL2Eps);
          if (half == 0) x.s_rk3[(c % 3) * kChunk + quad * 32 + lane] = rk_own;
        }
        tc::named_barrier_arrive(kBarNorm, kProducerThreads);
      } else if constexpr (kNorm) {
        tc::named_barrier(kBarNorm, kProducerThreads);
      }
    } else {
      if constexpr (kBwd) {
        // lane quarters 2-3 (no A epilogue without outputs): T -> T diag(beta) in place
        // (fp16 hi + lo, 22 significant bits), once the tile has landed: column j scaled
        // by beta_j; columns past the chunk's end get 0. Then the U MMAs may go.
        ok = ok && (*x.s_abort == 0) && tc::mbar_wait_timed(x.mb_t, c & 1, lim);
        tc::fence_after_sync();
        if (ok) {
#pragma unroll 1
          for (int r = 0; r < 8; ++r) {  // 4 columns (8 bytes of hi, 8 of lo) per step
            const int it = hq + r * 128, t = it >> 4, j4 = (it & 15) * 4;
            const uint32_t o = P::TB + tc::sw128(t, j4 * 2);
            const uint2 h = *reinterpret_cast<const uint2*>(sm + o);
            const uint2 l = *reinterpret_cast<const uint2*>(sm + o + 8192);
            const float2 h0 = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
            const float2 h1 = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
            const float2 l0 = __half22float2(*reinterpret_cast<const __half2*>(&l.x));
            const float2 l1 = __half22float2(*reinterpret_cast<const __half2*>(&l.y));
            const float4 bj = *reinterpret_cast<const float4*>(x.s_bv + gs + j4);
            uint2 nh, nl;
            split_half2((h0.x + l0.x) * bj.x, (h0.y + l0.y) * bj.y, nh.x, nl.x);
            split_half2((h1.x + l1.x) * bj.z, (h1.y + l1.y) * bj.w, nh.y, nl.y);
            *reinterpret_cast<uint2*>(sm + o) = nh;
            *reinterpret_cast<uint2*>(sm + o + 8192) = nl;
          }
        }
        signal(x.mb_vrdy);
      }
      // ---- A (fp16 hi + lo) from Q K^T, lanes 64-127 ------------------------------------
      if constexpr (kNorm && !kOut) {
        // fused prologue without outputs (no Gram to take |k|^2 from): one raw row per
        // thread, K rows 0-63 then Q rows 0-63, read once the tile has landed and before
        // any thread converts it in place. The inverse norms are folded into this chunk's
        // per-token factors (K: e^gc, e^{gc_last-gc}, F; Q: e^gc/sqrt(dk), E)
        ok = ok && (*x.s_abort == 0) && tc::mbar_wait_timed(b ? x.mb_kq1 : x.mb_kq0, use, lim);
        tc::fence_after_sync();
        const int row = half * 64 + (quad - 2) * 32 + lane, t = row & 63;
        const uint32_t base = kq_off + (row >> 6) * 8192;
        float ss = 0.f;
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            ss += sumsq_bf16x8(*reinterpret_cast<const uint4*>(sm + base + kb * 16384 + tc::sw128(t, j * 16)));
        const float r = 1.f / sqrtf(ss + kL2Eps);
        if (row < 64) {
          x.s_rk[t] = r;
          x.s_eg[gs + t] *= r;
          x.s_edec[gs + t] *= r;
          x.s_F[gs + t] *= r;
        } else {
          x.s_rq[t] = r;
          x.s_egq[gs + t] *= r;
          x.s_E[gs + t] *= r;
        }
        tc::named_barrier(kBarNorm, kProducerThreads);
      }
      if constexpr (kOut) ok = ok && (*x.s_abort == 0) && tc::mbar_wait_timed(x.mb_g, b, lim);
      tc::fence_after_sync();
      if (kOut && ok) {
        const int i = (quad - 2) * 32 + lane;  // A_ij = e^{gc_i - gc_j} q_i.k_j / sqrt(dk), j <= i
        const bool fast = x.s_fast[b] != 0;
        const float ei = x.s_E[gs + i] * kInvSqrtD;
#pragma unroll 1
        for (int j8 = 0; j8 < 4; ++j8) {  // 8 columns at a time
          const int j0 = half * 32 + j8 * 8;
          uint32_t d[8];
          tc::tmem_ld8(x.tmem + ((quad * 32u) << 16) + P::COL_GW + j0, d);
          tc::tmem_ld_wait();
          float a[8];
          if (fast) {
            const float4 f0 = *reinterpret_cast<const float4*>(x.s_F + gs + j0);
            const float4 f1 = *reinterpret_cast<const float4*>(x.s_F + gs + j0 + 4);
            const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) a[e] = (j0 + e <= i) ? ei * f[e] * __uint_as_float(d[e]) : 0.f;
          } else {
            // (raw q and k: 1 / |q_i| is applied to the output row, 1 / |k_j| to u)
            const float ri = kInvSqrtD;
            const float gi = x.s_gc[gs + i];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int j = j0 + e;
              a[e] = (j <= i) ? __expf(gi - x.s_gc[gs + j]) * ri * __uint_as_float(d[e]) : 0.f;
            }
          }
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_half2(a[2 * e], a[2 * e + 1], hi[e], lo[e]);
          const uint32_t o = tc::sw128(i, j0 * 2);
          *reinterpret_cast<uint4*>(sm + a_off + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(sm + a_off + 8192 + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      if constexpr (kNorm && kOut) {
        tc::named_barrier(kBarNorm, kProducerThreads);  // lane quarters 0-1 have published 1 / |k_t|
        rk_own = x.s_rk3[(c % 3) * kChunk + (ptid & 63)];
      }
    }

    // ---- once the Gram MMA has read K: K -> e^gc K (fp16, in place, rows t) and --------
    //      Kd = e^{gc_last-gc} K (KD[b]); tail rows zeroed
    // (without outputs there is no Gram MMA: the tile only has to have landed)
    if constexpr (kOut)
      ok = ok && (*x.s_abort == 0) && tc::mbar_wait_timed(x.mb_g, b, lim);
    else
      ok = ok && (*x.s_abort == 0) && tc::mbar_wait_timed(b ? x.mb_kq1 : x.mb_kq0, use, lim);
    tc::fence_after_sync();
    if (ok) {
#pragma unroll
      for (int r0 = 0; r0 < 4; r0 += 2) {
      uint4 rk[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int it = ptid + (r0 + r) * kProducerThreads, t = it & 63, cc = it >> 6;
        rk[r] = *reinterpret_cast<const uint4*>(sm + kq_off + (cc >> 3) * 16384 + tc::sw128(t, (cc & 7) * 16));
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int it = ptid + (r0 + r) * kProducerThreads, t = it & 63, cc = it >> 6;
        const bool live = t < clen;
        float f[8];
        unpack_bf16x8(rk[r], f);
        // (with the fused prologue t = ptid % 64, the row whose 1 / |k_t| this thread holds)
        *reinterpret_cast<uint4*>(sm + kq_off + (cc >> 3) * 16384 + tc::sw128(t, (cc & 7) * 16)) =
            live ? pack_half8(f, kNorm && kOut ? x.s_eg[gs + t] * rk_own : x.s_eg[gs + t]) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(sm + kd_off + (cc >> 3) * 8192 + tc::sw128(t, (cc & 7) * 16)) =
            live ? pack_half8(f, x.s_edec[gs + t]) : make_uint4(0, 0, 0, 0);
      }
      }
    }
    signal(x.mb_krdy);  // e^gc K is converted and Q K^T has been read: the W MMAs may go

    // ---- meanwhile: Q -> Q~ = e^gc Q / sqrt(dk) (fp16, rows t, tail rows zeroed), once
    //      the spine of chunk c-1 has read Q~ (and -W^T) ------------------------------------
    if (kOut && c > 0) ok = ok && (*x.s_abort == 0) && tc::mbar_wait_timed(x.mb_c1, (c - 1) & 1, lim);
    if (kOut && ok) {
      float qss = 0.f;  // fused prologue: this thread's part of |q_t|^2 (row t = ptid % 64)
#pragma unroll 1
      for (int r0 = 0; r0 < 4; r0 += 2) {
        uint4 rq[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int it = ptid + (r0 + r) * kProducerThreads, t = it & 63, cc = it >> 6;
          rq[r] = *reinterpret_cast<const uint4*>(sm + kq_off + (cc >> 3) * 16384 + 8192 + tc::sw128(t, (cc & 7) * 16));
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int it = ptid + (r0 + r) * kProducerThreads, t = it & 63, cc = it >> 6;
          float f[8];
          unpack_bf16x8(rq[r], f);
          if constexpr (kNorm) {
#pragma unroll
            for (int e = 0; e < 8; ++e) qss = fmaf(f[e], f[e], qss);
          }
          *reinterpret_cast<uint4*>(sm + P::QT + (cc >> 3) * 8192 + tc::sw128(t, (cc & 7) * 16)) =
              t < clen ? pack_half8(f, x.s_egq[gs + t]) : make_uint4(0, 0, 0, 0);
        }
      }
      if constexpr (kNorm) x.s_qpart[(ptid >> 6) * kChunk + (ptid & 63)] = qss;
    }
    signal(b ? x.mb_qrdy1 : x.mb_qrdy0);  // the raw K/Q tile is consumed: it may be refilled
    // ---- and the gates of the next chunk, into the other gate set (their copy was
    //      started a chunk ago), and the copy of the gates of the chunk after -----------
    if (pw == 4 && c + 1 < x.nchunks) {
      tc::cp_async_wait_all();
      scan_gates(c + 1);
      if (c + 2 < x.nchunks) load_gates(c + 2);
    }
    tc::fence_proxy_async();
    if (!tc::barrier_all(kBarProducer, kProducerThreads, ok && *x.s_abort == 0)) {
      if (leader) fail();
      break;
    }
    if constexpr (kNorm && kOut) {
      // 1 / |q_t| of this chunk, for the consumer's output rows (the A and Q~ operands
      // carry the raw q: both output terms are linear in q_t); published by the hand-off
      if (pw == 2) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int t = h2 * 32 + lane;
          const float ss = x.s_qpart[t] + x.s_qpart[kChunk + t] + x.s_qpart[2 * kChunk + t] + x.s_qpart[3 * kChunk + t];
          x.s_rq3[(c % 3) * kChunk + t] = 1.f / sqrtf(ss + kL2Eps);
        }
      }
    }
    if (!group_wait(x, p, x.mb_uw, b, kBarProducer, kProducerThreads, leader, lim)) break;

    // ---- -W^T as the spine's fp16 B operand (rows k, columns t) -----------------------
    {
      uint32_t d[32];
      tc::tmem_ld32(x.tmem + ((quad * 32u) << 16) + P::COL_GW + half * 32, d);
      tc::tmem_ld_wait();
      tc::fence_before_sync();  // the W columns are read (tensor memory only): the next Gram MMA may go
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(x.mb_wrd);
      if constexpr (!kOut) {
        // The single -W^T tile was last read by the spine MMAs of chunk c - 1; runs with
        // outputs waited for them before converting Q~
        if (c > 0 && !group_wait(x, p, x.mb_c1, (c - 1) & 1, kBarProducer, kProducerThreads, leader, lim)) break;
      }
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
    bool arrive = leader;
    if constexpr (kTest) arrive = arrive && c != p.test_skip_chunk;
    if (arrive) tc::mbar_arrive(b ? x.mb_hand1 : x.mb_hand0);  // chunk c's operands are ready
  }
}

// ---------------------------------------------------------------------------------
// Consumer: the state spine and the output of each chunk. Thread v owns value
// column v: tensor-memory lane v holds S^T[v][:], u^T[v][:] and O^T[v][:].
// ---------------------------------------------------------------------------------
template <bool kOut, bool kNorm, bool kTest, bool kBwd>
__device__ __forceinline__ void consumer_role(const Ctx& x, const ChunkParams& p, int ctid, int seq) {
  using P = Plan;
  const uint64_t lim = wait_limit<kTest>(p);
  const int quad = ctid >> 5;
  const int v = ctid;
  const bool leader = ctid == 0;
  const int lane = ctid & 31;
  const uint32_t lanes = x.tmem + ((quad * 32u) << 16);
  // one arrival per warp on a readiness barrier of the issuer, after this warp's
  // tensor-memory accesses
  auto signal = [&](uint32_t mbar) {
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(mbar);
  };

  // backward's forward chain: this thread's value column of a chunk's entry state, as
  // fp16 into its slot ([k][v]: the 32 lanes of a warp write 64 consecutive bytes)
  auto store_s0 = [&](int c, int q4, const uint32_t (&s)[32]) {
    __half* dst = p.s0buf + ((x.row0 / kChunk + seq + c) * p.nv + x.h) * kDim * kDim + (q4 * 32) * kDim + v;
#pragma unroll
    for (int e = 0; e < 32; ++e) dst[e * kDim] = __float2half_rn(__uint_as_float(s[e]));
  };

  // carried-in state: fp32 S^T into tensor memory, plus its fp16 operand copy
  {
    uint32_t s[32], st[32];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
      for (int e = 0; e < 32; ++e) s[e] = __float_as_uint(x.state[(q4 * 32 + e) * kDim + v]);
      if constexpr (kBwd) store_s0(0, q4, s);
      tc::tmem_st32(lanes + P::COL_S + q4 * 32, s);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        st[(q4 & 1) * 16 + e] = pack_half2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1]));
      if (q4 & 1) tc::tmem_st32(lanes + P::COL_ST + (q4 >> 1) * 32, st);
    }
    tc::tmem_st_wait();
  }
  signal(x.mb_strdy);  // S^T of the first chunk is ready
  // output rows overwrite the WY kernel's T diag(beta) rows: no store before that
  // kernel has completed (see the issuer)
  tc::grid_dependency_wait();

  // S^T <- e^{gc_last} S^T, the decay half of the state update of chunk `cn` (its fp16
  // copy, which the MMAs read, is separate): two 64-column halves, both loads in flight
  auto decay_state = [&](int cn) {
    const float el = x.s_elast[cn % 3];
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint32_t s0[32], s1[32];
      tc::tmem_ld32(lanes + P::COL_S + h * 64, s0);
      tc::tmem_ld32(lanes + P::COL_S + h * 64 + 32, s1);
      tc::tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        s0[e] = __float_as_uint(el * __uint_as_float(s0[e]));
        s1[e] = __float_as_uint(el * __uint_as_float(s1[e]));
      }
      tc::tmem_st32(lanes + P::COL_S + h * 64, s0);
      tc::tmem_st32(lanes + P::COL_S + h * 64 + 32, s1);
    }
    tc::tmem_st_wait();
  };

  // sum of every output and final-state value this thread writes: non-finite exactly
  // when one of them is (an operand outside the fp16 range turns into inf or NaN)
  float chk = 0.f;
  for (int c = 0; c < x.nchunks; ++c) {
    const int b = c & 1;
    const int64_t rem = x.len - static_cast<int64_t>(c) * kChunk;
    const int clen = rem < kChunk ? static_cast<int>(rem) : kChunk;
    const uint32_t col_u = P::COL_U + 64 * b;

    if constexpr (kTest) {
      // test hook: fall behind the producer before the hand-off wait of odd chunks
      if ((c & 1) && p.test_delay_ns > 0) {
        const uint64_t t0 = tc::globaltimer_ns();
        while (tc::globaltimer_ns() - t0 < static_cast<uint64_t>(p.test_delay_ns)) __nanosleep(500);
      }
    }
    if (!group_wait(x, p, b ? x.mb_hand1 : x.mb_hand0, (c >> 1) & 1, kBarConsumer, kConsumerThreads, leader, lim))
      break;
    // (the issuer runs u^T = U^T - S^T W^T onto U^T and O^T = S^T Q~^T.) The decay of
    // chunk c > 0 was applied at the end of the previous iteration, while these ran.
    if (c == 0) decay_state(0);
    if (!group_wait(x, p, x.mb_c1, b, kBarConsumer, kConsumerThreads, leader, lim)) break;

    // ---- u^T as an fp16 hi + lo pair in tensor memory (the A operand of the next MMAs) ---
    {
#pragma unroll 1
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t u[32], hi[16], lo[16];
        tc::tmem_ld32(lanes + col_u + h2 * 32, u);
        tc::tmem_ld_wait();
        if constexpr (kBwd) {  // u rows for the gradient kernels (rows of the chunk only)
          __half* dst = p.ubuf + (x.row0 + static_cast<int64_t>(c) * kChunk + h2 * 32) * (p.nv * kDim) + x.h * kDim + v;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (h2 * 32 + e < clen) dst[static_cast<int64_t>(e) * p.nv * kDim] = __float2half_rn(__uint_as_float(u[e]));
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          // columns past the end of the sequence are zeroed: their U and W rows came
          // from other tokens' T diag(beta) rows
          const int t = h2 * 32 + 2 * e;
          float u0 = t < clen ? __uint_as_float(u[2 * e]) : 0.f, u1 = t + 1 < clen ? __uint_as_float(u[2 * e + 1]) : 0.f;
          if constexpr (kNorm && kOut) {  // fused prologue: A and Kd carry the raw keys
            u0 *= x.s_rk3[(c % 3) * kChunk + t];
            u1 *= x.s_rk3[(c % 3) * kChunk + t + 1];
          }
          split_half2(u0, u1, hi[e], lo[e]);
        }
        tc::tmem_st16u(lanes + P::COL_UT + h2 * 16, hi);
        tc::tmem_st16u(lanes + P::COL_UT + 32 + h2 * 16, lo);
      }
      tc::tmem_st_wait();
    }
    signal(x.mb_usp);                    // the issuer runs S^T += u^T Kd, O^T += u^T A^T
    signal(b ? x.mb_cu1 : x.mb_cu0);     // the U columns of this chunk parity are free again
    if (!group_wait(x, p, b ? x.mb_c21 : x.mb_c20, (c >> 1) & 1, kBarConsumer, kConsumerThreads, leader, lim))
      break;

    // ---- next chunk's fp16 S^T operand; this chunk's O^T into registers ---------------
    uint32_t o[64];
    {
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t s[32], st[16];
        tc::tmem_ld32(lanes + P::COL_S + q4 * 32, s);
        tc::tmem_ld_wait();
        if constexpr (kBwd) {
          if (c + 1 < x.nchunks) store_s0(c + 1, q4, s);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) st[e] = pack_half2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1]));
        tc::tmem_st16u(lanes + P::COL_ST + q4 * 16, st);
      }
      if constexpr (kOut) {
        uint32_t (&o0)[32] = *reinterpret_cast<uint32_t(*)[32]>(o);
        uint32_t (&o1)[32] = *reinterpret_cast<uint32_t(*)[32]>(o + 32);
        tc::tmem_ld32(lanes + P::COL_O, o0);
        tc::tmem_ld32(lanes + P::COL_O + 32, o1);
        tc::tmem_ld_wait();
      }
      tc::tmem_st_wait();
    }
    signal(x.mb_strdy);  // S^T of the next chunk is ready and O^T has been read

    // ---- meanwhile (the next chunk's first MMAs run): this chunk's output rows, then
    //      the decay of the next chunk --------------------------------------------------
    if (kOut && x.store_out) {
      // O^T holds one value column per thread: for each row t, the 32 lanes of a warp
      // store 32 consecutive bf16 values, one 64-byte segment (no shared-memory staging)
      __nv_bfloat16* optr = p.out + (x.row0 + static_cast<int64_t>(c) * kChunk) * p.out_stride +
                            static_cast<int64_t>(x.h) * kDim + v;
      const int64_t ostride = p.out_stride;
#pragma unroll
      for (int e = 0; e < 64; ++e) {
        if (e < clen) {
          float y = __uint_as_float(o[e]);
          if constexpr (kNorm) y *= x.s_rq3[(c % 3) * kChunk + e];  // fused prologue: 1 / |q_t|
          *optr = __float2bfloat16_rn(y);
          chk += y;
        }
        optr += ostride;
      }
    }
    if (c + 1 < x.nchunks) decay_state(c + 1);
  }

  if (!kBwd && *x.s_abort == 0) {  // carried-out state S_T, k-major
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint32_t s[32];
      tc::tmem_ld32(lanes + P::COL_S + q4 * 32, s);
      tc::tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        x.state[(q4 * 32 + e) * kDim + v] = __uint_as_float(s[e]);
        chk += __uint_as_float(s[e]);
      }
    }
    if (!isfinite(chk)) atomicOr(p.status, kStatusRange);
  }
}

// ---------------------------------------------------------------------------------
// Issuers: one thread each. The producer-side issuer runs, per chunk c, the Gram
// MMA, the U and W MMAs and the copies that refill the buffers c has consumed; the
// spine issuer runs the spine's two MMA groups of each chunk. The producer and
// consumer warps only convert operands and signal readiness, so no warp that
// converts waits for an instruction queue.
// ---------------------------------------------------------------------------------
template <bool kOut, bool kTest>
__device__ __forceinline__ void issuer_role(const Ctx& x, const ChunkParams& p, const CUtensorMap* tmap_q,
                                            const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                            const CUtensorMap* tmap_t, bool spine_side) {
  using P = Plan;
  const uint64_t lim = wait_limit<kTest>(p);
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
  auto issue_v = [&](int c) {  // V tile of chunk c, into buffer c & 1
    const uint32_t vd = x.sbase + ((c & 1) ? P::V1 : P::V0);
    const uint32_t mb = (c & 1) ? x.mb_v1 : x.mb_v0;
    const int32_t y = static_cast<int32_t>(x.row0 + static_cast<int64_t>(c) * kChunk);
    tc::mbar_arrive_expect_tx(mb, 16384);
    tc::tma_load_2d(vd, tmap_v, x.h * kDim, y, mb);
    tc::tma_load_2d(vd + 8192, tmap_v, x.h * kDim + 64, y, mb);
  };
  auto issue_t = [&](int c) {  // T diag(beta) hi/lo tiles of chunk c (single buffer)
    const int32_t y = static_cast<int32_t>(x.row0 + static_cast<int64_t>(c) * kChunk);
    tc::mbar_arrive_expect_tx(x.mb_t, 16384);
    tc::tma_load_2d(x.sbase + P::TB, tmap_t, x.h * kDim, y, x.mb_t);
    tc::tma_load_2d(x.sbase + P::TB + 8192, tmap_t, x.h * kDim + 64, y, x.mb_t);
  };
  auto wait = [&](uint32_t mbar, uint32_t parity) -> bool {
    if (*x.s_abort != 0) return false;
    if (!tc::mbar_wait_timed(mbar, parity, lim)) {
      *x.s_abort = 1;
      atomicOr(p.status, kStatusTimeout);
      return false;
    }
    tc::fence_after_sync();
    return true;
  };
  // Gram matrix [K;Q] K^T (bf16, M=128, N=64, K=128); lanes 64-127 hold Q K^T
  auto gram = [&](int c) {
    constexpr uint32_t idesc = tc::idesc_f16(128, 64, tc::kBF16, false, false);
    const uint32_t kq = x.sbase + ((c & 1) ? P::KQ1 : P::KQ0);
#pragma unroll
    for (int st = 0; st < 8; ++st) {
      const uint32_t a = kq + (st >> 2) * 16384 + (st & 3) * 32;
      tc::mma_f16(x.tmem + P::COL_GW, tc::desc_sw128(a, 16, 1024), tc::desc_sw128(a, 16, 1024), idesc, st > 0);
    }
    tc::mma_commit(x.mb_g);
  };
  // U^T = V^T (T diag beta)^T (hi + lo) into the chunk-parity U columns; W^T likewise
  // from (e^gc K)^T into the Gram columns
  auto wy = [&](int c, bool is_u) {
    constexpr uint32_t id = tc::idesc_f16(128, 64, tc::kF16, true, false);
    const int b = c & 1;
    const uint32_t d_col = is_u ? P::COL_U + 64 * b : P::COL_GW;
    const uint32_t a_base = x.sbase + (is_u ? (b ? P::V1 : P::V0) : (b ? P::KQ1 : P::KQ0));
    const uint32_t a_lbo = is_u ? 8192 : 16384;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
#pragma unroll
      for (int st = 0; st < 4; ++st)
        tc::mma_f16(x.tmem + d_col, tc::desc_sw128(a_base + st * 2048, a_lbo, 1024),
                    tc::desc_sw128(x.sbase + P::TB + part * 8192 + st * 32, 16, 1024), id, part + st > 0);
    }
  };
  // spine, first half: u^T = U^T - S^T W^T (onto U^T) and O^T = S^T Q~^T
  auto spine1 = [&](int c) {
    constexpr uint32_t id_u = tc::idesc_f16(128, 64, tc::kF16, false, true);
    constexpr uint32_t id_o = tc::idesc_f16(128, 64, tc::kF16, false, false);
    const uint32_t col_u = P::COL_U + 64 * (c & 1);
#pragma unroll 1
    for (int st = 0; st < 8; ++st) {
      const uint32_t a = x.tmem + P::COL_ST + st * 8;
      tc::mma_f16_ts(x.tmem + col_u, a, tc::desc_sw128(x.sbase + P::W16 + st * 2048, 16384, 1024), id_u, 1);
      if constexpr (kOut)
        tc::mma_f16_ts(x.tmem + P::COL_O, a,
                       tc::desc_sw128(x.sbase + P::QT + (st >> 2) * 8192 + (st & 3) * 32, 16, 1024), id_o, st > 0);
    }
    tc::mma_commit(x.mb_c1);
  };
  // spine, second half: S^T += u^T Kd and O^T += u^T A^T (hi/lo x3)
  auto spine2 = [&](int c) {
    constexpr uint32_t id_s = tc::idesc_f16(128, 128, tc::kF16, false, true);
    constexpr uint32_t id_o = tc::idesc_f16(128, 64, tc::kF16, false, false);
    const int b = c & 1;
    const uint32_t kd_off = b ? P::KD1 : P::KD0, a_off = b ? P::A1 : P::A0;
#pragma unroll 1
    for (int st = 0; st < 4; ++st) {
      const uint32_t u_hi = x.tmem + P::COL_UT + st * 8, u_lo = x.tmem + P::COL_UT + 32 + st * 8;
      const uint64_t a_hi = tc::desc_sw128(x.sbase + a_off + st * 32, 16, 1024);
      const uint64_t a_lo = tc::desc_sw128(x.sbase + a_off + 8192 + st * 32, 16, 1024);
      tc::mma_f16_ts(x.tmem + P::COL_S, u_hi, tc::desc_sw128(x.sbase + kd_off + st * 2048, 8192, 1024), id_s, 1);
      if constexpr (kOut) {
        tc::mma_f16_ts(x.tmem + P::COL_O, u_hi, a_hi, id_o, 1);
        tc::mma_f16_ts(x.tmem + P::COL_O, u_hi, a_lo, id_o, 1);
        tc::mma_f16_ts(x.tmem + P::COL_O, u_lo, a_hi, id_o, 1);
      }
    }
    tc::mma_commit(b ? x.mb_c21 : x.mb_c20);
  };

  const int n = x.nchunks;
  if (spine_side) {
    for (int c = 0; c < n; ++c) {
      // first half once the operands are handed over and S^T is ready (and O^T read)
      if (!wait((c & 1) ? x.mb_hand1 : x.mb_hand0, (c >> 1) & 1) || !wait(x.mb_strdy, c & 1)) break;
      spine1(c);
      // second half once u is split
      if (!wait(x.mb_usp, c & 1)) break;
      spine2(c);
    }
    return;
  }
  issue_kq(0);
  issue_v(0);
  if (n > 1) {
    issue_kq(1);
    issue_v(1);
  }
  for (int c = 0; c < n; ++c) {
    const int b = c & 1;
    // Gram of c: its K/Q tile has landed and the W MMAs of c-1 have been read out
    // (runs without outputs need no Gram)
    if constexpr (kOut) {
      if ((c > 0 && !wait(x.mb_wrd, (c - 1) & 1)) || !wait(b ? x.mb_kq1 : x.mb_kq0, (c >> 1) & 1)) break;
      gram(c);
    }
    // the T diag(beta) rows are the WY kernel's output: under a dependent launch this
    // CTA may have started while that kernel still runs, so the first copy of them
    // waits for its completion (the loads and the Gram above need only the inputs)
    if (c == 0) {
      tc::grid_dependency_wait();
      issue_t(0);
    }
    // U of c: V is fp16, T diag(beta) has landed, and u of c-2 has been read
    if (!wait(x.mb_vrdy, c & 1) || !wait(x.mb_t, c & 1) ||
        (c >= 2 && !wait(b ? x.mb_cu1 : x.mb_cu0, ((c - 2) >> 1) & 1)))
      break;
    wy(c, true);
    // W of c: e^gc K is converted and the Gram columns have been read
    if (!wait(x.mb_krdy, c & 1)) break;
    if constexpr (!kOut) {  // no Gram ordered this after the W epilogue of c-1
      if (c > 0 && !wait(x.mb_wrd, (c - 1) & 1)) break;
    }
    wy(c, false);
    tc::mma_commit(x.mb_uw);
    // refill what chunk c has consumed
    if (!wait(x.mb_uw, c & 1) || !wait(b ? x.mb_qrdy1 : x.mb_qrdy0, (c >> 1) & 1)) break;
    if (c + 2 < n) {
      issue_kq(c + 2);
      issue_v(c + 2);
    }
    if (c + 1 < n) issue_t(c + 1);
  }
}

// kOut = false: runs that only carry the state (the segment schedule's state maps):
// no Gram, A, Q~, output MMAs or output rows. kNorm: the fused q/k normalisation
// (ChunkParams::qk_l2norm), a separate instantiation so that the common path carries
// none of its code. kTest: the test hooks of ChunkParams (wait limit, consumer delay,
// skipped hand-off), likewise an instantiation of its own.
constexpr int kNumMbar = 21;
template <bool kOut = true, bool kNorm = false, bool kTest = false, bool kBwd = false>
__global__ void __launch_bounds__(kThreads, 1)
gdn_prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_t,
                   const ChunkParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(16) float s_gc[2 * kChunk], s_eg[2 * kChunk], s_egq[2 * kChunk], s_edec[2 * kChunk];
  __shared__ __align__(16) float s_E[2 * kChunk], s_F[2 * kChunk], s_gstage[2 * kChunk];
  __shared__ __align__(16) float s_bstage[kBwd ? 2 * kChunk : 1], s_bv[kBwd ? 2 * kChunk : 1];
  __shared__ __align__(16) float s_rq[kChunk], s_rk[kChunk];
  __shared__ __align__(16) float s_qpart[kNorm && kOut ? 4 * kChunk : 1], s_rq3[kNorm && kOut ? 3 * kChunk : 1];
  __shared__ __align__(16) float s_rk3[kNorm && kOut ? 3 * kChunk : 1];
  __shared__ float s_elast[3];
  __shared__ int s_fast[2];
  __shared__ __align__(8) uint64_t s_mb[kNumMbar];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5;

  // ---- which (sequence, head) this CTA owns -------------------------------------------
  Ctx x;
  x.h = blockIdx.x % p.nv;
  const int slot = blockIdx.x / p.nv;
  const int s = p.order ? p.order[slot] : slot;
  x.kh = x.h / (p.nv / p.nk);
  x.store_out = 1;
  x.zero_v = 0;
  if (p.seg) {  // host-built segment table: trusted ranges inside the packed rows
    x.row0 = p.seg[4 * s];
    x.len = p.seg[4 * s + 1];
    x.store_out = (p.seg[4 * s + 2] & kSegNoOutput) == 0;
    x.zero_v = (p.seg[4 * s + 2] & kSegZeroValues) != 0;
  } else if (p.cu_seqlens) {
    if (s < 0 || s >= p.B) {
      tc::grid_dependency_wait();
      if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
    const int a = p.cu_seqlens[s], e = p.cu_seqlens[s + 1];
    if (a < 0 || e < a || e > p.T) {
      tc::grid_dependency_wait();
      if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
      return;
    }
    x.row0 = a;
    x.len = e - a;
  } else {
    const int64_t skip = static_cast<int64_t>(p.chunk_begin) * kChunk < p.T ? static_cast<int64_t>(p.chunk_begin) * kChunk : p.T;
    x.row0 = static_cast<int64_t>(s) * p.T + skip;
    x.len = p.T - skip;
    if (p.chunk_count > 0 && x.len > static_cast<int64_t>(p.chunk_count) * kChunk)
      x.len = static_cast<int64_t>(p.chunk_count) * kChunk;
  }
  x.nchunks = static_cast<int>((x.len + kChunk - 1) / kChunk);
  if (x.nchunks == 0) {  // empty sequence: the state passes through unchanged
    tc::grid_dependency_wait();
    return;
  }
  float* state = p.state_is_table ? reinterpret_cast<float* const*>(p.state)[s]
                                  : reinterpret_cast<float*>(p.state) + static_cast<int64_t>(s) * p.nv * kDim * kDim;
  x.state = state + static_cast<int64_t>(x.h) * kDim * kDim;
  // 1024-byte aligned, by pointer arithmetic on the shared array so that accesses
  // through it stay shared-space (not generic) loads and stores
  x.sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  x.sbase = tc::smem_u32(x.sm);
  x.s_gc = s_gc;
  x.s_eg = s_eg;
  x.s_egq = s_egq;
  x.s_edec = s_edec;
  x.s_elast = s_elast;
  x.s_E = s_E;
  x.s_F = s_F;
  x.s_rq = s_rq;
  x.s_rk = s_rk;
  x.s_qpart = s_qpart;
  x.s_rq3 = s_rq3;
  x.s_rk3 = s_rk3;
  x.s_fast = s_fast;
  x.s_gstage = s_gstage;
  x.s_bstage = s_bstage;
  x.s_bv = s_bv;
  x.s_abort = &s_abort;
  x.mb_kq0 = tc::smem_u32(&s_mb[0]);
  x.mb_kq1 = tc::smem_u32(&s_mb[1]);
  x.mb_v0 = tc::smem_u32(&s_mb[2]);
  x.mb_v1 = tc::smem_u32(&s_mb[3]);
  x.mb_t = tc::smem_u32(&s_mb[4]);
  x.mb_g = tc::smem_u32(&s_mb[5]);
  x.mb_uw = tc::smem_u32(&s_mb[6]);
  x.mb_c1 = tc::smem_u32(&s_mb[7]);
  x.mb_c20 = tc::smem_u32(&s_mb[8]);
  x.mb_c21 = tc::smem_u32(&s_mb[9]);
  x.mb_hand0 = tc::smem_u32(&s_mb[10]);
  x.mb_cu0 = tc::smem_u32(&s_mb[11]);
  x.mb_cu1 = tc::smem_u32(&s_mb[12]);
  x.mb_vrdy = tc::smem_u32(&s_mb[13]);
  x.mb_krdy = tc::smem_u32(&s_mb[14]);
  x.mb_qrdy0 = tc::smem_u32(&s_mb[15]);
  x.mb_wrd = tc::smem_u32(&s_mb[16]);
  x.mb_strdy = tc::smem_u32(&s_mb[17]);
  x.mb_usp = tc::smem_u32(&s_mb[18]);
  x.mb_hand1 = tc::smem_u32(&s_mb[19]);
  x.mb_qrdy1 = tc::smem_u32(&s_mb[20]);

  if (warp == 0) tc::tmem_alloc(tc::smem_u32(&s_tmem), Plan::TMEM_COLS);
  if (tid == 0) {
    s_abort = 0;
    // arrival counts: copies and MMA commits 1, per-warp readiness 4 or 8
    // (V ready: 4 arrivals, or 8 when lane quarters 2-3 also scale T by beta)
    constexpr uint32_t kCount[kNumMbar] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 4, 4, kBwd ? 8u : 4u, 8, 8, 8, 4, 4, 1, 8};
#pragma unroll
    for (int i = 0; i < kNumMbar; ++i) tc::mbar_init(tc::smem_u32(&s_mb[i]), kCount[i]);
    tc::mbar_fence_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  x.tmem = s_tmem;

  if (warp < kConsumerWarps)
    consumer_role<kOut, kNorm, kTest, kBwd>(x, p, tid, s);
  else if (warp < kConsumerWarps + kProducerWarps)
    producer_role<kOut, kNorm, kTest, kBwd>(x, p, tid - kConsumerThreads);
  else if ((tid & 31) == 0)
    issuer_role<kOut, kTest>(x, p, &tmap_q, &tmap_k, &tmap_v, &tmap_t, warp == kConsumerWarps + kProducerWarps + 1);

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

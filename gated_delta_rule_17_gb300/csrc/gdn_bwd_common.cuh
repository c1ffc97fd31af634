// Chunked backward of the gated delta rule (the training pass) for sm_103a.
//
// The forward (ssm_gdn_a3.rs, `gdn_prefill_fla` doc comment: the chunked WY form
// of S_t = e^{g_t}(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
// o_t = S_t^T q_t / sqrt(dk)) is, per chunk of 64 tokens with entry state S0,
// in-chunk log-decay prefix b (Gamma = e^b, gamma = Gamma_last) and
// M_tj = e^{b_t - b_j} (j <= t):
//
//     L = strict_lower(beta_t M_tj k_t.k_j),  T = (I + L)^{-1}
//     X = V - Gamma K S0,                     u = T diag(beta) X
//     O = Gamma Q S0 / sqrt(dk) + (Q K^T . M) u / sqrt(dk)
//     S_end = gamma S0 + (gamma / Gamma) K^T u
//
// Its derivative, with dS_end the gradient of the chunk's end state (the pages
// describe only the forward; this is the chain rule through the lines above):
//
//     du  = (Q K^T . M)^T dO / sqrt(dk) + (gamma / Gamma) K dS_end
//     du' = T^T du,   r = beta du',   dV = r
//     dS0 = gamma dS_end + Q^T (Gamma dO) / sqrt(dk) - K^T (Gamma r)
//
// and, per chunk and independent of the other chunks once S0 and dS_end are known,
// with dA = lower(dO u^T) . M / sqrt(dk), F = -strict_lower(du' u^T) . M, E = beta F,
// P = du' S0^T, G = K K^T:
//
//     dQ = Gamma dO S0^T / sqrt(dk) + dA K
//     dK = E K + E^T K - Gamma beta P + dA^T Q + (gamma / Gamma) u dS_end^T
//     dbeta_t = du'_t.v_t - Gamma_t k_t.P_t + sum_j F_tj G_tj
//     d b_t   = Gamma_t q_t.(dO S0^T)_t / sqrt(dk) - Gamma_t beta_t k_t.P_t
//               + rows - columns of (E . G) and of (dA . Q K^T)
//               - w_t, w_t = (gamma / Gamma_t) k_t.(u dS_end^T)_t,
//               plus gamma <dS_end, S0> + sum_t w_t on the last token
//     dg_t = sum of d b over the chunk's tokens t .. 63
//
// Three chain and gradient kernels, all on tcgen05: the forward chain is the output-free
// spine of gdn_prefill_kernel.cuh (state in tensor memory; its backward instantiation
// scales the WY kernel's T by beta and stores every chunk's entry state S0 and u);
// gdn_bwd_dstates_tc_kernel (gdn_bwd_dstates_tc.cuh) runs the reverse chain, storing
// every chunk's dS_end and du' and writing dV; gdn_bwd_grads_tc_kernel
// (gdn_bwd_grads_tc.cuh) takes one (chunk, key head) each and writes dQ, dK (summed over
// the key head's GQA group of value heads), and dbeta and dg of every value head. T
// comes from the forward's WY kernel (unscaled by beta). This file holds what they share.
//
// Padding tokens of a ragged last chunk are loaded as q = k = v = dO = 0,
// g = beta = 0, and T's rows past the chunk's end as 0: every product then
// reduces to the chunk's real tokens, and gamma = Gamma_63.
#pragma once
#include "gdn_common.cuh"

namespace gdn {

// 16-byte asynchronous copy to shared memory; zero-fills the destination when !valid
// (the source address must still be a valid one)
__device__ __forceinline__ void cp_async16(uint32_t dst_saddr, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst_saddr), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}

struct BwdChunkParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  const void* h0;      // float[B][nv][128][128], or float*[B] when state_is_table
  const float* dout;   // [rows][nv][128]
  const float* dst;    // [B][nv][128][128] or null (zero)
  const uint16_t* tm;  // [rows][nv][128]: row t of the chunk's T, 64 fp16 hi then 64 lo
  __half* ubuf;        // [rows][nv][128]: u
  __half* dubuf;       // [rows][nv][128]: du' = T^T du
  __half* s0buf;       // [slots][nv][128][128]: each chunk's entry state S0 ([k][v])
  __half* dsbuf;       // [slots][nv][128][128]: each chunk's dS_end ([k][v])
  float* dq;           // [rows][nk][128]
  float* dk;           // [rows][nk][128]
  float* dv;           // [rows][nv][128]
  float* dg;           // [rows][nv]
  float* dbeta;        // [rows][nv]
  float* dh0;          // [B][nv][128][128] or null
  const int32_t* cu_seqlens;
  const int32_t* order;      // varlen: sequences by decreasing length
  const int32_t* cu_chunks;  // varlen: chunk prefix over the sequences
  unsigned* status;
  int64_t q_stride, k_stride, v_stride, g_stride, beta_stride;
  int B, T, nk, nv;
  int state_is_table;
};

// Rows of sequence s; false (and the status bit) for an invalid cu_seqlens entry.
__device__ __forceinline__ bool bc_sequence(const BwdChunkParams& p, int s, int64_t& row0, int64_t& len) {
  if (p.cu_seqlens) {
    const int a = p.cu_seqlens[s], e = p.cu_seqlens[s + 1];
    if (a < 0 || e < a || e > p.T) {
      if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeqlens);
      return false;
    }
    row0 = a;
    len = e - a;
  } else {
    row0 = static_cast<int64_t>(s) * p.T;
    len = p.T;
  }
  return true;
}

// Slot of chunk c of the sequence starting at row0 (unique over the batch: the
// chunks of sequence s occupy row0 / 64 + s + [0, chunks)).
__device__ __forceinline__ int64_t bc_slot(int64_t row0, int s, int64_t c) { return row0 / kChunk + s + c; }

struct BcGates {
  float g0, g1, b0, b1;  // g and beta of tokens 2 lane and 2 lane + 1
};

__device__ __forceinline__ void bc_fetch_gates(BcGates& x, const BwdChunkParams& p, int64_t r0, int n, int h) {
  const int t0 = 2 * (threadIdx.x & 31), t1 = t0 + 1;
  x.g0 = t0 < n ? p.g[(r0 + t0) * p.g_stride + h] : 0.f;
  x.g1 = t1 < n ? p.g[(r0 + t1) * p.g_stride + h] : 0.f;
  x.b0 = t0 < n ? p.beta[(r0 + t0) * p.beta_stride + h] : 0.f;
  x.b1 = t1 < n ? p.beta[(r0 + t1) * p.beta_stride + h] : 0.f;
}

// In-chunk log-decay prefix b of the fetched gates (every warp computes it); warp 0
// also writes b and beta per token to shared memory.
__device__ __forceinline__ GatePrefix bc_put_gates(const BcGates& x, float* s_b, float* s_beta) {
  const GatePrefix gp = gate_prefix(x.g0, x.g1);
  if ((threadIdx.x >> 5) == 0) {
    const int t0 = 2 * (threadIdx.x & 31);
    s_b[t0] = gp.gca;
    s_b[t0 + 1] = gp.gcb;
    s_beta[t0] = x.b0;
    s_beta[t0 + 1] = x.b1;
  }
  return gp;
}

}  // namespace gdn

// Backward of the gated delta rule (the training pass) for sm_103a.
//
// The recurrence of the GDN prefill op (ssm_gdn_a3.rs, `gdn_prefill_fla`: the
// chunked form of S_t = e^{g_t}(I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
// o_t = S_t^T q_t / sqrt(dk)) differentiated token by token in reverse, in fp32
// on the CUDA cores. Per token, with P = S_{t-1}, D = e^{g} P, p = D^T k,
// w = v - p, S = D + beta k w^T and G = dL/dS (the future's gradient plus the
// token's read-out term q do^T / sqrt(dk)):
//
//     dq = S do / sqrt(dk)          dv = beta G^T k          dp = -dv
//     dbeta = (G^T k) . w           dD = G + k dp^T
//     dk = beta G w + D dp          dg = <dD, D>             dL/dS_{t-1} = e^{g} dD
//
// A persistent CTA walks (sequence, v-head) items. For each it runs the
// sequence forward once, storing the state at every 64-token boundary, then
// walks the blocks backwards: it recomputes the block's 64 entry states into
// its own scratch slot and steps back through them. Thread (kg, vg) of 256
// owns rows 16 kg .. 16 kg + 15 and columns 4 vg .. 4 vg + 3 of P and of G;
// sums over k go through shared memory, sums over v through warp shuffles.
// q and k gradients are written per v-head and summed over each GQA group by
// gdn_backward_reduce_kernel.
#pragma once
#include "gdn_common.cuh"

namespace gdn {

constexpr int kBwdThreads = 256;
constexpr int kBwdBlock = 64;  // tokens between stored states

struct BwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  const void* h0;  // float[B][nv][128][128], or float*[B] when state_is_table
  const float* dout;  // [rows][nv][128]
  const float* dst;   // [B][nv][128][128] or null (zero)
  float* dq_part;     // [rows][nv][128]: dq of each v-head, summed per key head afterwards
  float* dk_part;     // [rows][nv][128]
  float* dv;          // [rows][nv][128]
  float* dg;          // [rows][nv]
  float* dbeta;       // [rows][nv]
  float* dh0;         // [B][nv][128][128] or null
  float* ckpt;        // [rows/64 + B + 1][nv][128][128]: states at block boundaries
  float* blocks;      // [gridDim.x][65][128][128]: a CTA's recomputed block states
  const int32_t* cu_seqlens;
  unsigned* status;
  int64_t q_stride, k_stride, v_stride, g_stride, beta_stride;
  int B, T, nk, nv;
  int state_is_table;
};

// Sum over the 32 lanes of each of the 16 per-row partials; lane i (< 16) ends
// with the total of row i.
__device__ __forceinline__ float warp_rows16(float (&r)[16]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] += __shfl_xor_sync(0xffffffffu, r[i], o);
  const int lane = threadIdx.x & 31;
  float mine = r[0];
#pragma unroll
  for (int i = 1; i < 16; ++i) mine = (lane == i) ? r[i] : mine;
  return mine;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__global__ void __launch_bounds__(kBwdThreads, 1) gdn_backward_kernel(const BwdParams p) {
  __shared__ float s_k[kDim], s_q[kDim], s_v[kDim], s_do[kDim];
  __shared__ __align__(16) float s_part[kBwdThreads / 32][kDim];
  __shared__ float s_red[kBwdThreads / 32];
  __shared__ float s_ab[2];
  const int tid = threadIdx.x;
  const int vg = tid & 31, kg = tid >> 5;
  const int items = p.B * p.nv;
  float* slot = p.blocks + static_cast<int64_t>(blockIdx.x) * (kBwdBlock + 1) * kDim * kDim;
  const int64_t my = static_cast<int64_t>(16 * kg) * kDim + 4 * vg;  // this thread's first element

  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int s = item / p.nv, h = item % p.nv, kh = h / (p.nv / p.nk);
    int64_t row0, len;
    if (p.cu_seqlens) {
      const int a = p.cu_seqlens[s], e = p.cu_seqlens[s + 1];
      if (a < 0 || e < a || e > p.T) {
        if (tid == 0) atomicOr(p.status, kStatusBadSeqlens);
        continue;
      }
      row0 = a;
      len = e - a;
    } else {
      row0 = static_cast<int64_t>(s) * p.T;
      len = p.T;
    }
    const int64_t nblk = (len + kBwdBlock - 1) / kBwdBlock;
    const int64_t cbase = row0 / kBwdBlock + s;  // this sequence's first checkpoint index
    auto ck = [&](int64_t j) { return p.ckpt + ((cbase + j) * p.nv + h) * kDim * kDim; };
    const float* h0 = p.state_is_table ? reinterpret_cast<const float* const*>(p.h0)[s]
                                       : reinterpret_cast<const float*>(p.h0) + static_cast<int64_t>(s) * p.nv * kDim * kDim;
    h0 += static_cast<int64_t>(h) * kDim * kDim;

    float4 S[16];
    // one forward step of token r from S (the entry state) in place; needs s_k, s_v, s_ab
    auto forward_step = [&]() {
      const float a = s_ab[0], b = s_ab[1];
      float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float kk = s_k[16 * kg + i];
        r.x = fmaf(kk, S[i].x, r.x); r.y = fmaf(kk, S[i].y, r.y);
        r.z = fmaf(kk, S[i].z, r.z); r.w = fmaf(kk, S[i].w, r.w);
      }
      *reinterpret_cast<float4*>(&s_part[kg][4 * vg]) = r;
      __syncthreads();
      float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < kBwdThreads / 32; ++j) {
        const float4 t = *reinterpret_cast<const float4*>(&s_part[j][4 * vg]);
        pv.x += t.x; pv.y += t.y; pv.z += t.z; pv.w += t.w;
      }
      const float4 w = make_float4(s_v[4 * vg] - a * pv.x, s_v[4 * vg + 1] - a * pv.y,
                                   s_v[4 * vg + 2] - a * pv.z, s_v[4 * vg + 3] - a * pv.w);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float bk = b * s_k[16 * kg + i];
        S[i].x = fmaf(a, S[i].x, bk * w.x); S[i].y = fmaf(a, S[i].y, bk * w.y);
        S[i].z = fmaf(a, S[i].z, bk * w.z); S[i].w = fmaf(a, S[i].w, bk * w.w);
      }
    };
    auto load_token = [&](int64_t r, bool with_q) {
      __syncthreads();  // the previous step is done with the token buffers
      if (tid < kDim) {
        s_k[tid] = __bfloat162float(p.k[r * p.k_stride + kh * kDim + tid]);
        s_v[tid] = __bfloat162float(p.v[r * p.v_stride + h * kDim + tid]);
        if (with_q) {
          s_q[tid] = __bfloat162float(p.q[r * p.q_stride + kh * kDim + tid]);
          s_do[tid] = p.dout[(r * p.nv + h) * kDim + tid];
        }
      }
      if (tid == 0) {
        s_ab[0] = __expf(p.g[r * p.g_stride + h]);
        s_ab[1] = p.beta[r * p.beta_stride + h];
      }
      __syncthreads();
    };

    // ---- forward over the sequence, keeping the state at every block boundary -----
#pragma unroll
    for (int i = 0; i < 16; ++i) S[i] = *reinterpret_cast<const float4*>(h0 + my + i * kDim);
    for (int64_t t = 0; t < len; ++t) {
      if (t % kBwdBlock == 0) {
        float* c = ck(t / kBwdBlock);
#pragma unroll
        for (int i = 0; i < 16; ++i) *reinterpret_cast<float4*>(c + my + i * kDim) = S[i];
      }
      load_token(row0 + t, false);
      forward_step();
    }

    // ---- backward, block by block from the end ----------------------------------------
    float4 G[16];
    if (p.dst) {
      const float* d = p.dst + (static_cast<int64_t>(s) * p.nv + h) * kDim * kDim;
#pragma unroll
      for (int i = 0; i < 16; ++i) G[i] = *reinterpret_cast<const float4*>(d + my + i * kDim);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) G[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int64_t bi = nblk - 1; bi >= 0; --bi) {
      const int64_t t0 = bi * kBwdBlock, t1 = t0 + kBwdBlock < len ? t0 + kBwdBlock : len;
      const float* c = ck(bi);
#pragma unroll
      for (int i = 0; i < 16; ++i) S[i] = *reinterpret_cast<const float4*>(c + my + i * kDim);
      for (int64_t t = t0; t < t1; ++t) {  // slot[j] = the state entering token t0 + j
        float* d = slot + (t - t0) * kDim * kDim;
#pragma unroll
        for (int i = 0; i < 16; ++i) *reinterpret_cast<float4*>(d + my + i * kDim) = S[i];
        load_token(row0 + t, false);
        forward_step();
      }
      for (int64_t t = t1 - 1; t >= t0; --t) {
        const int64_t r = row0 + t;
        const float* d = slot + (t - t0) * kDim * kDim;
#pragma unroll
        for (int i = 0; i < 16; ++i) S[i] = *reinterpret_cast<const float4*>(d + my + i * kDim);  // P
        load_token(r, true);
        const float a = s_ab[0], b = s_ab[1];
        // p = a P^T k, w = v - p
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float kk = s_k[16 * kg + i];
          acc.x = fmaf(kk, S[i].x, acc.x); acc.y = fmaf(kk, S[i].y, acc.y);
          acc.z = fmaf(kk, S[i].z, acc.z); acc.w = fmaf(kk, S[i].w, acc.w);
        }
        *reinterpret_cast<float4*>(&s_part[kg][4 * vg]) = acc;
        __syncthreads();
        float4 pv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kBwdThreads / 32; ++j) {
          const float4 tt = *reinterpret_cast<const float4*>(&s_part[j][4 * vg]);
          pv.x += tt.x; pv.y += tt.y; pv.z += tt.z; pv.w += tt.w;
        }
        const float4 w = make_float4(s_v[4 * vg] - a * pv.x, s_v[4 * vg + 1] - a * pv.y,
                                     s_v[4 * vg + 2] - a * pv.z, s_v[4 * vg + 3] - a * pv.w);
        const float4 dov = *reinterpret_cast<const float4*>(&s_do[4 * vg]);
        // dq rows (S_t do), G += q do^T / sqrt(dk), and this thread's part of G^T k
        float rq[16];
        float4 gk = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float kk = s_k[16 * kg + i], bk = b * kk, qq = s_q[16 * kg + i] * kInvSqrtD;
          const float4 sn = make_float4(fmaf(a, S[i].x, bk * w.x), fmaf(a, S[i].y, bk * w.y),
                                        fmaf(a, S[i].z, bk * w.z), fmaf(a, S[i].w, bk * w.w));
          rq[i] = sn.x * dov.x + sn.y * dov.y + sn.z * dov.z + sn.w * dov.w;
          G[i].x = fmaf(qq, dov.x, G[i].x); G[i].y = fmaf(qq, dov.y, G[i].y);
          G[i].z = fmaf(qq, dov.z, G[i].z); G[i].w = fmaf(qq, dov.w, G[i].w);
          gk.x = fmaf(kk, G[i].x, gk.x); gk.y = fmaf(kk, G[i].y, gk.y);
          gk.z = fmaf(kk, G[i].z, gk.z); gk.w = fmaf(kk, G[i].w, gk.w);
        }
        {
          const float dqi = warp_rows16(rq) * kInvSqrtD;
          if (vg < 16) p.dq_part[(r * p.nv + h) * kDim + 16 * kg + vg] = dqi;
        }
        __syncthreads();  // every thread has read s_part (p)
        *reinterpret_cast<float4*>(&s_part[kg][4 * vg]) = gk;
        __syncthreads();
        gk = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kBwdThreads / 32; ++j) {
          const float4 tt = *reinterpret_cast<const float4*>(&s_part[j][4 * vg]);
          gk.x += tt.x; gk.y += tt.y; gk.z += tt.z; gk.w += tt.w;
        }
        // dv = b G^T k, dp = -dv, dbeta = (G^T k) . w
        const float4 dp = make_float4(-b * gk.x, -b * gk.y, -b * gk.z, -b * gk.w);
        if (kg == 0) {
          *reinterpret_cast<float4*>(p.dv + (r * p.nv + h) * kDim + 4 * vg) =
              make_float4(b * gk.x, b * gk.y, b * gk.z, b * gk.w);
          const float db = warp_sum(gk.x * w.x + gk.y * w.y + gk.z * w.z + gk.w * w.w);
          if (vg == 0) p.dbeta[r * p.nv + h] = db;
        }
        // dD = G + k dp^T; dk = b G w + D dp; dg = <dD, D>; G <- a dD
        float rk[16];
        float dgp = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float kk = s_k[16 * kg + i];
          const float4 D = make_float4(a * S[i].x, a * S[i].y, a * S[i].z, a * S[i].w);
          rk[i] = b * (G[i].x * w.x + G[i].y * w.y + G[i].z * w.z + G[i].w * w.w) +
                  (D.x * dp.x + D.y * dp.y + D.z * dp.z + D.w * dp.w);
          const float4 dD = make_float4(fmaf(kk, dp.x, G[i].x), fmaf(kk, dp.y, G[i].y),
                                        fmaf(kk, dp.z, G[i].z), fmaf(kk, dp.w, G[i].w));
          dgp += dD.x * D.x + dD.y * D.y + dD.z * D.z + dD.w * D.w;
          G[i] = make_float4(a * dD.x, a * dD.y, a * dD.z, a * dD.w);
        }
        {
          const float dki = warp_rows16(rk);
          if (vg < 16) p.dk_part[(r * p.nv + h) * kDim + 16 * kg + vg] = dki;
        }
        dgp = warp_sum(dgp);
        if (vg == 0) s_red[kg] = dgp;
        __syncthreads();
        if (tid == 0) {
          float tot = 0.f;
#pragma unroll
          for (int j = 0; j < kBwdThreads / 32; ++j) tot += s_red[j];
          p.dg[r * p.nv + h] = tot;
        }
      }
    }
    if (p.dh0) {
      float* d = p.dh0 + (static_cast<int64_t>(s) * p.nv + h) * kDim * kDim;
#pragma unroll
      for (int i = 0; i < 16; ++i) *reinterpret_cast<float4*>(d + my + i * kDim) = G[i];
    }
    __syncthreads();
  }
}

// dq[r][kh] = sum of dq_part[r][h] over the v-heads h of key head kh (and dk).
__global__ void gdn_backward_reduce_kernel(const float* dq_part, const float* dk_part, float* dq, float* dk,
                                           int64_t rows, int nk, int nv) {
  const int64_t n = rows * nk * kDim;
  const int group = nv / nk;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / (static_cast<int64_t>(nk) * kDim);
    const int kh = static_cast<int>((i / kDim) % nk), e = static_cast<int>(i % kDim);
    float sq = 0.f, sk = 0.f;
    for (int j = 0; j < group; ++j) {
      const int64_t o = (r * nv + kh * group + j) * kDim + e;
      sq += dq_part[o];
      sk += dk_part[o];
    }
    dq[i] = sq;
    dk[i] = sk;
  }
}

}  // namespace gdn

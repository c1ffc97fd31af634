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
// Every column of S and of G evolves on its own (p, w, dp and the updates are
// per column), so a (sequence, v-head) item is split over 1, 2 or 4 CTAs of
// 128, 64 or 32 columns (kC = 4, 2, 1 columns per thread, as many as the SMs
// can hold at once); only dq, dk, dg and dbeta sum over columns, and each CTA
// writes its part of them. A persistent CTA runs its columns of the sequence
// forward once, storing them every 64 tokens, then walks the blocks backwards:
// it recomputes the block's 64 entry states into its own scratch slot and steps
// back through them. Thread (kg, lane) of 256 owns rows 16 kg .. 16 kg + 15 of
// kC adjacent columns; sums over k go through shared memory, sums over the
// columns through warp shuffles. gdn_backward_reduce_kernel adds the parts
// (and the value heads of each GQA group, for dq and dk).
#pragma once
#include "gdn_common.cuh"

namespace gdn {

constexpr int kBwdThreads = 256;
constexpr int kBwdBlock = 64;     // tokens between stored states
constexpr int kBwdMaxSplit = 4;   // at most 4 CTAs of 32 columns per (sequence, v-head)

// CTAs per SM for kC columns per thread (the registers of S and G grow with kC)
__host__ __device__ constexpr int bwd_ctas_per_sm(int kC) { return kC == 1 ? 3 : (kC == 2 ? 2 : 1); }

struct BwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  const void* h0;  // float[B][nv][128][128], or float*[B] when state_is_table
  const float* dout;  // [rows][nv][128]
  const float* dst;   // [B][nv][128][128] or null (zero)
  float* dq_part;     // [rows][nv][nsplit][128]: per v-head and column split
  float* dk_part;     // [rows][nv][nsplit][128]
  float* dg_part;     // [rows][nv][nsplit]
  float* dbeta_part;  // [rows][nv][nsplit]
  float* dv;          // [rows][nv][128]
  float* dg_out;      // [rows][nv]
  float* dbeta_out;   // [rows][nv]
  float* dh0;         // [B][nv][128][128] or null
  float* ckpt;        // [rows/64 + B + 1][nv][128][128]: states at block boundaries (by split)
  float* blocks;      // [gridDim.x][65][128 x 128/nsplit]: a CTA's recomputed block states
  const int32_t* cu_seqlens;
  unsigned* status;
  int64_t q_stride, k_stride, v_stride, g_stride, beta_stride;
  int B, T, nk, nv;
  int nsplit;  // CTAs per (sequence, v-head): 128 / nsplit columns each
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

// kC columns per thread: a CTA covers 32 kC columns, nsplit = 4 / kC CTAs per item.
template <int kC>
__global__ void __launch_bounds__(kBwdThreads, bwd_ctas_per_sm(kC)) gdn_backward_kernel(const BwdParams p) {
  constexpr int kCols = 32 * kC;                                    // columns per CTA
  constexpr int64_t kPart = static_cast<int64_t>(kDim) * kCols;     // floats of a CTA's state block
  constexpr int kSplit = kDim / kCols;
  __shared__ float s_k[kDim], s_q[kDim], s_v[kCols], s_do[kCols];
  __shared__ float s_part[kBwdThreads / 32][kCols];
  __shared__ float s_red[kBwdThreads / 32];
  __shared__ float s_ab[2];
  const int tid = threadIdx.x;
  const int lane = tid & 31, kg = tid >> 5;
  const int items = p.B * p.nv * kSplit;
  float* slot = p.blocks + static_cast<int64_t>(blockIdx.x) * (kBwdBlock + 1) * kPart;
  const int64_t mine = static_cast<int64_t>(16 * kg) * kCols + kC * lane;  // in a [128][kCols] block

  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int split = item % kSplit, sh = item / kSplit;
    const int s = sh / p.nv, h = sh % p.nv, kh = h / (p.nv / p.nk);
    const int col = split * kCols + kC * lane;  // this thread's first column of S
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
    auto ck = [&](int64_t j) { return p.ckpt + (((cbase + j) * p.nv + h) * kSplit + split) * kPart; };
    const float* h0 = p.state_is_table ? reinterpret_cast<const float* const*>(p.h0)[s]
                                       : reinterpret_cast<const float*>(p.h0) + static_cast<int64_t>(s) * p.nv * kDim * kDim;
    h0 += static_cast<int64_t>(h) * kDim * kDim;

    float S[16][kC];
    auto load_token = [&](int64_t r, bool with_q) {
      __syncthreads();  // the previous step is done with the token buffers
      if (tid < kDim) {
        s_k[tid] = __bfloat162float(p.k[r * p.k_stride + kh * kDim + tid]);
        if (with_q) s_q[tid] = __bfloat162float(p.q[r * p.q_stride + kh * kDim + tid]);
      } else if (tid < kDim + kCols) {
        const int c = tid - kDim;
        s_v[c] = __bfloat162float(p.v[r * p.v_stride + h * kDim + split * kCols + c]);
        if (with_q) s_do[c] = p.dout[(r * p.nv + h) * kDim + split * kCols + c];
      }
      if (tid == kBwdThreads - 1) {
        s_ab[0] = __expf(p.g[r * p.g_stride + h]);
        s_ab[1] = p.beta[r * p.beta_stride + h];
      }
      __syncthreads();
    };
    // w = v - a S^T k for this thread's columns (S the entry state); one barrier
    auto columns_w = [&](float a, float (&w)[kC]) {
      float acc[kC];
#pragma unroll
      for (int c = 0; c < kC; ++c) acc[c] = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int c = 0; c < kC; ++c) acc[c] = fmaf(s_k[16 * kg + i], S[i][c], acc[c]);
#pragma unroll
      for (int c = 0; c < kC; ++c) s_part[kg][kC * lane + c] = acc[c];
      __syncthreads();
#pragma unroll
      for (int c = 0; c < kC; ++c) {
        float pv = 0.f;
#pragma unroll
        for (int j = 0; j < kBwdThreads / 32; ++j) pv += s_part[j][kC * lane + c];
        w[c] = s_v[kC * lane + c] - a * pv;
      }
    };
    auto forward_step = [&]() {
      const float a = s_ab[0], b = s_ab[1];
      float w[kC];
      columns_w(a, w);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float bk = b * s_k[16 * kg + i];
#pragma unroll
        for (int c = 0; c < kC; ++c) S[i][c] = fmaf(a, S[i][c], bk * w[c]);
      }
    };
    auto load_block = [&](const float* src, int64_t ld) {  // rows of S at row stride ld
#pragma unroll
      for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int c = 0; c < kC; ++c) S[i][c] = src[i * ld + c];
    };
    auto store_block = [&](float* dst) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int c = 0; c < kC; ++c) dst[i * kCols + c] = S[i][c];
    };

    // ---- forward over the sequence, keeping the state at every block boundary -----
    load_block(h0 + (16 * kg) * kDim + col, kDim);
    for (int64_t t = 0; t < len; ++t) {
      if (t % kBwdBlock == 0) store_block(ck(t / kBwdBlock) + mine);
      load_token(row0 + t, false);
      forward_step();
    }

    // ---- backward, block by block from the end ----------------------------------------
    float G[16][kC];
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int c = 0; c < kC; ++c)
        G[i][c] = p.dst ? p.dst[(static_cast<int64_t>(s) * p.nv + h) * kDim * kDim + (16 * kg + i) * kDim + col + c] : 0.f;
    for (int64_t bi = nblk - 1; bi >= 0; --bi) {
      const int64_t t0 = bi * kBwdBlock, t1 = t0 + kBwdBlock < len ? t0 + kBwdBlock : len;
      load_block(ck(bi) + mine, kCols);
      for (int64_t t = t0; t < t1; ++t) {  // slot[j] = the state entering token t0 + j
        store_block(slot + (t - t0) * kPart + mine);
        load_token(row0 + t, false);
        forward_step();
      }
      for (int64_t t = t1 - 1; t >= t0; --t) {
        const int64_t r = row0 + t;
        load_block(slot + (t - t0) * kPart + mine, kCols);  // P
        load_token(r, true);
        const float a = s_ab[0], b = s_ab[1];
        float w[kC], dov[kC];
        columns_w(a, w);
#pragma unroll
        for (int c = 0; c < kC; ++c) dov[c] = s_do[kC * lane + c];
        // dq rows (S_t do), G += q do^T / sqrt(dk), and this thread's part of G^T k
        float rq[16];
        float gk[kC];
#pragma unroll
        for (int c = 0; c < kC; ++c) gk[c] = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float kk = s_k[16 * kg + i], bk = b * kk, qq = s_q[16 * kg + i] * kInvSqrtD;
          rq[i] = 0.f;
#pragma unroll
          for (int c = 0; c < kC; ++c) {
            rq[i] = fmaf(fmaf(a, S[i][c], bk * w[c]), dov[c], rq[i]);
            G[i][c] = fmaf(qq, dov[c], G[i][c]);
            gk[c] = fmaf(kk, G[i][c], gk[c]);
          }
        }
        const int64_t part = (r * p.nv + h) * kSplit + split;
        {
          const float dqi = warp_rows16(rq) * kInvSqrtD;
          if (lane < 16) p.dq_part[part * kDim + 16 * kg + lane] = dqi;
        }
        __syncthreads();  // every thread has read s_part (w)
#pragma unroll
        for (int c = 0; c < kC; ++c) s_part[kg][kC * lane + c] = gk[c];
        __syncthreads();
        float dp[kC], dbp = 0.f;
#pragma unroll
        for (int c = 0; c < kC; ++c) {
          float sum = 0.f;
#pragma unroll
          for (int j = 0; j < kBwdThreads / 32; ++j) sum += s_part[j][kC * lane + c];
          // dv = b G^T k, dp = -dv, dbeta = (G^T k) . w over these columns
          dp[c] = -b * sum;
          dbp = fmaf(sum, w[c], dbp);
          if (kg == 0) p.dv[(r * p.nv + h) * kDim + col + c] = b * sum;
        }
        if (kg == 0) {
          dbp = warp_sum(dbp);
          if (lane == 0) p.dbeta_part[part] = dbp;
        }
        // dD = G + k dp^T; dk = b G w + D dp; dg = <dD, D>; G <- a dD
        float rk[16];
        float dgp = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float kk = s_k[16 * kg + i];
          rk[i] = 0.f;
#pragma unroll
          for (int c = 0; c < kC; ++c) {
            const float D = a * S[i][c], dD = fmaf(kk, dp[c], G[i][c]);
            rk[i] = fmaf(b * G[i][c], w[c], fmaf(D, dp[c], rk[i]));
            dgp = fmaf(dD, D, dgp);
            G[i][c] = a * dD;
          }
        }
        {
          const float dki = warp_rows16(rk);
          if (lane < 16) p.dk_part[part * kDim + 16 * kg + lane] = dki;
        }
        dgp = warp_sum(dgp);
        if (lane == 0) s_red[kg] = dgp;
        __syncthreads();
        if (tid == 0) {
          float tot = 0.f;
#pragma unroll
          for (int j = 0; j < kBwdThreads / 32; ++j) tot += s_red[j];
          p.dg_part[part] = tot;
        }
      }
    }
    if (p.dh0) {
      float* d = p.dh0 + (static_cast<int64_t>(s) * p.nv + h) * kDim * kDim + (16 * kg) * kDim + col;
#pragma unroll
      for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int c = 0; c < kC; ++c) d[i * kDim + c] = G[i][c];
    }
    __syncthreads();
  }
}

// Sums the column-split parts: dq[r][kh] and dk[r][kh] over the splits and the value
// heads of key head kh; dg[r][h] and dbeta[r][h] over the splits.
__global__ void gdn_backward_reduce_kernel(const BwdParams p, float* dq, float* dk, int64_t rows) {
  const int group = p.nv / p.nk, ns = p.nsplit;
  const int64_t n = rows * p.nk * kDim, m = rows * p.nv;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n + m; i += stride) {
    if (i < n) {
      const int64_t r = i / (static_cast<int64_t>(p.nk) * kDim);
      const int kh = static_cast<int>((i / kDim) % p.nk), e = static_cast<int>(i % kDim);
      float sq = 0.f, sk = 0.f;
      for (int j = 0; j < group; ++j)
        for (int sp = 0; sp < ns; ++sp) {
          const int64_t o = ((r * p.nv + kh * group + j) * ns + sp) * kDim + e;
          sq += p.dq_part[o];
          sk += p.dk_part[o];
        }
      dq[i] = sq;
      dk[i] = sk;
    } else {
      const int64_t rh = i - n;
      float sg = 0.f, sb = 0.f;
      for (int sp = 0; sp < ns; ++sp) {
        sg += p.dg_part[rh * ns + sp];
        sb += p.dbeta_part[rh * ns + sp];
      }
      p.dg_out[rh] = sg;
      p.dbeta_out[rh] = sb;
    }
  }
}

}  // namespace gdn

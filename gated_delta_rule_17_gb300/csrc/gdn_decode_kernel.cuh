// Single-token GDN decode step for sm_103a.
//
// The recurrent update that follows the prefill in serving (the state the
// GDN prefill op carries in and out, ssm_gdn_a3.rs, `gdn_prefill_fla`
// problem arguments): for every sequence b and value head h, with one new
// token (q, k, v, g, beta),
//
//     S' = e^g S;   r = k^T S';   S <- S' + beta k (v - r)^T;   o = S^T q / sqrt(dk)
//
// It is bound by the state's HBM traffic (64 KB read and written per
// (sequence, head)); the arithmetic is three 128 x 128 matrix-vector passes,
// so it runs on the CUDA cores. One CTA per (sequence, head): 256 threads,
// thread (kg, vg) owns the 16 x 4 block S[16 kg : 16 kg + 16, 4 vg : 4 vg + 4]
// in registers, loaded and stored as float4 rows, so every warp moves whole
// 512-byte row segments. The two reductions over k go through shared memory.
#pragma once
#include "gdn_common.cuh"

namespace gdn {

constexpr int kDecodeThreads = 256;

struct DecodeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const float* g;
  const float* beta;
  void* state;  // float[B][nv][128][128], or float*[B] when state_is_table
  __nv_bfloat16* out;
  int64_t q_stride, k_stride, v_stride, g_stride, beta_stride, out_stride;
  int B, nk, nv;
  int state_is_table;
  int qk_l2norm;  // fused prologue: normalise the q and k rows first
};

__global__ void __launch_bounds__(kDecodeThreads)
gdn_decode_kernel(const DecodeParams p) {
  __shared__ float s_k[kDim], s_q[kDim];
  __shared__ __align__(16) float s_part[8][kDim];  // per-k-group partial sums over k
  __shared__ float s_norm[2][4];                   // fused prologue: per-warp sums of squares
  const int tid = threadIdx.x;
  const int vg = tid & 31, kg = tid >> 5;  // v = 4 vg .. 4 vg + 3, k = 16 kg .. 16 kg + 15
  const int h = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.nv));
  const int b = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.nv));
  const int kh = h / (p.nv / p.nk);

  float* base = p.state_is_table ? reinterpret_cast<float* const*>(p.state)[b]
                                 : reinterpret_cast<float*>(p.state) + static_cast<int64_t>(b) * p.nv * kDim * kDim;
  float* S = base + static_cast<int64_t>(h) * kDim * kDim;
  // the state block first, so that its HBM latency overlaps the token's loads
  float4 s[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) s[i] = *reinterpret_cast<const float4*>(S + (16 * kg + i) * kDim + 4 * vg);
  if (tid < kDim) {
    s_k[tid] = __bfloat162float(p.k[b * p.k_stride + kh * kDim + tid]);
    s_q[tid] = __bfloat162float(p.q[b * p.q_stride + kh * kDim + tid]);
  }
  if (p.qk_l2norm) {  // 1 / |k|, 1 / |q| (warps 0-3 hold the two rows)
    __syncthreads();
    if (tid < kDim) {
      float sk = s_k[tid] * s_k[tid], sq = s_q[tid] * s_q[tid];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
      }
      if ((tid & 31) == 0) {
        s_norm[0][tid >> 5] = sk;
        s_norm[1][tid >> 5] = sq;
      }
    }
    __syncthreads();
    if (tid < kDim) {
      const float rk = 1.f / sqrtf(s_norm[0][0] + s_norm[0][1] + s_norm[0][2] + s_norm[0][3] + kL2Eps);
      const float rq = 1.f / sqrtf(s_norm[1][0] + s_norm[1][1] + s_norm[1][2] + s_norm[1][3] + kL2Eps);
      s_k[tid] *= rk;
      s_q[tid] *= rq;
    }
  }
  const float a = __expf(p.g[b * p.g_stride + h]);
  const float bt = p.beta[b * p.beta_stride + h];

  // decayed state block and its partial k^T S'
  __syncthreads();
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
    const float kk = s_k[16 * kg + i];
    r.x = fmaf(kk, s[i].x, r.x); r.y = fmaf(kk, s[i].y, r.y);
    r.z = fmaf(kk, s[i].z, r.z); r.w = fmaf(kk, s[i].w, r.w);
  }
  *reinterpret_cast<float4*>(&s_part[kg][4 * vg]) = r;
  __syncthreads();
  // delta = beta (v - k^T S') for this thread's 4 columns
  float4 rs = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 t = *reinterpret_cast<const float4*>(&s_part[j][4 * vg]);
    rs.x += t.x; rs.y += t.y; rs.z += t.z; rs.w += t.w;
  }
  const __nv_bfloat16* vrow = p.v + b * p.v_stride + h * kDim + 4 * vg;
  const float4 d = make_float4(bt * (__bfloat162float(vrow[0]) - rs.x), bt * (__bfloat162float(vrow[1]) - rs.y),
                               bt * (__bfloat162float(vrow[2]) - rs.z), bt * (__bfloat162float(vrow[3]) - rs.w));
  // S <- S' + k delta^T, stored back; partial S^T q
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float kk = s_k[16 * kg + i], qq = s_q[16 * kg + i];
    s[i].x = fmaf(kk, d.x, s[i].x); s[i].y = fmaf(kk, d.y, s[i].y);
    s[i].z = fmaf(kk, d.z, s[i].z); s[i].w = fmaf(kk, d.w, s[i].w);
    *reinterpret_cast<float4*>(S + (16 * kg + i) * kDim + 4 * vg) = s[i];
    o.x = fmaf(qq, s[i].x, o.x); o.y = fmaf(qq, s[i].y, o.y);
    o.z = fmaf(qq, s[i].z, o.z); o.w = fmaf(qq, s[i].w, o.w);
  }
  __syncthreads();  // every thread has read its partial of k^T S'
  *reinterpret_cast<float4*>(&s_part[kg][4 * vg]) = o;
  __syncthreads();
  if (tid < 32) {
    float4 os = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 t = *reinterpret_cast<const float4*>(&s_part[j][4 * tid]);
      os.x += t.x; os.y += t.y; os.z += t.z; os.w += t.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(os.x * kInvSqrtD, os.y * kInvSqrtD);
    __nv_bfloat162 hi = __floats2bfloat162_rn(os.z * kInvSqrtD, os.w * kInvSqrtD);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&lo);
    w.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p.out + b * p.out_stride + h * kDim + 4 * tid) = w;
  }
}

}  // namespace gdn

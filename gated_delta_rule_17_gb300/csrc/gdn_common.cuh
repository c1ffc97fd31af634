// Constants and small register-level helpers shared by the two GDN prefill
// kernels (the chunk-parallel WY solve and the fused state spine).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "tc.cuh"

namespace gdn {

constexpr int kDim = 128;   // dk == dv
constexpr int kChunk = 64;  // tokens per chunk

// Status bits written to the per-device status word.
constexpr unsigned kStatusBadSeqlens = 1u;
constexpr unsigned kStatusTimeout = 2u;
// An output or the final state came out non-finite: an operand left the range of the
// 16-bit tensor-core types (|v|, |S| and the intermediates must stay below ~6.5e4).
constexpr unsigned kStatusRange = 4u;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr float kInvSqrtD = 0.08838834764831845f;  // 1 / sqrt(128)

// Decays e^{gc_i - gc_j} are factorised as E_i F_j about the middle of the
// chunk's gate range when that range is at most this many nats, so that both
// factors stay within e^{+-60}; wider ranges evaluate each decay directly.
constexpr float kFactorisedRange = 120.f;

// fp32 64 x 64 work matrix with 16-byte chunks XOR-swizzled by row, so that
// float4 accesses by threads on different rows hit different banks; chunk k of a row
// is also XORed with k / 8, so that chunks k and k + 8 of one row (256 bytes apart,
// the same banks otherwise) land in different bank groups.
__device__ __forceinline__ int lf_idx(int r, int c) {
  return r * 64 + ((((c >> 2) ^ r ^ (c >> 5)) & 15) << 2) + (c & 3);
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

// (a, b) = hi + lo with hi = fp16(x), lo = fp16(x - hi): about 22 significant bits.
__device__ __forceinline__ void split_half2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 x = __floats2half2_rn(a, b);
  const float2 xf = __half22float2(x);
  const __half2 y = __floats2half2_rn(a - xf.x, b - xf.y);
  hi = *reinterpret_cast<const uint32_t*>(&x);
  lo = *reinterpret_cast<const uint32_t*>(&y);
}

// (a, b) = hi + lo with hi = bf16(x), lo = bf16(x - hi): about 16 significant bits,
// with fp32's exponent range.
__device__ __forceinline__ void split_bf162(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 x = __floats2bfloat162_rn(a, b);
  const float2 xf = __bfloat1622float2(x);
  const __nv_bfloat162 y = __floats2bfloat162_rn(a - xf.x, b - xf.y);
  hi = *reinterpret_cast<const uint32_t*>(&x);
  lo = *reinterpret_cast<const uint32_t*>(&y);
}

// Fused prologue: a head row is scaled by 1 / sqrt(sum(x^2) + kL2Eps).
constexpr float kL2Eps = 1e-6f;

// Sum of squares of the 8 bf16 values in a 16-byte chunk.
__device__ __forceinline__ float sumsq_bf16x8(const uint4 raw) {
  float f[8];
  unpack_bf16x8(raw, f);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s = fmaf(f[i], f[i], s);
  return s;
}

// Inclusive in-chunk prefix of the log-gates held by one warp, lane l holding
// tokens 2l and 2l+1 (padding tokens carry g = 0).
struct GatePrefix {
  float gca, gcb;  // gc of tokens 2l and 2l+1
  float first;     // gc of token 0
  float last;      // gc of token 63 (= that of the last real token)
};

__device__ __forceinline__ GatePrefix gate_prefix(float g0, float g1) {
  const int lane = threadIdx.x & 31;
  const float pair = g0 + g1;
  float incl = pair;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  GatePrefix r;
  r.gca = incl - pair + g0;
  r.gcb = incl;
  r.last = __shfl_sync(0xffffffffu, incl, 31);
  r.first = __shfl_sync(0xffffffffu, r.gca, 0);
  return r;
}

}  // namespace gdn

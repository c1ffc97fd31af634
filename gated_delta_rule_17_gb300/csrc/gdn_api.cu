// C ABI of the chunked gated-delta-rule prefill (declared in include/gdn_prefill.h).
//
// Host side: validates every argument before anything is enqueued (each
// rejection names the guard, in the spirit of the GDN prefill op's named
// guards, ssm_gdn_a3.rs `gdn_tc_spine_reject`), encodes the TMA descriptors
// for q, k, v and the output, and enqueues at most three kernels on the
// caller's stream: the varlen schedule (sequences ordered by decreasing
// length and the chunk prefix over them, validating cu_seqlens on the
// device), the chunk-parallel WY solve and the fused spine kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <utility>

#include "gdn_prefill.h"
#include "gdn_prefill_kernel.cuh"
#include "gdn_wy_kernel.cuh"
#include "gdn_decode_kernel.cuh"
#include "gdn_bwd_dstates_tc.cuh"
#include "gdn_bwd_grads_tc.cuh"

namespace {

thread_local char g_err[512] = "";
thread_local int g_launches = 0;
thread_local cudaEvent_t g_timing[3] = {nullptr, nullptr, nullptr};  // gdn_set_timing_events
// gdn_set_test_hooks: wait limit (ns), consumer delay (ns), skipped hand-off chunk
struct TestHooks {
  int64_t wait_ns = 0, delay_ns = 0;
  int skip_chunk = -1;
  bool active() const { return wait_ns > 0 || delay_ns > 0 || skip_chunk >= 0; }
};
thread_local TestHooks g_hooks;

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

__device__ unsigned g_status;  // per-device status word (bits gdn::kStatus*)

constexpr int kMaxDevices = 64;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
  bool attrs = false;
  unsigned* status = nullptr;
  cudaStream_t copy_in = nullptr, copy_out = nullptr;  // gdn_prefill_host's copy streams
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.attrs) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
      return fail(GDN_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major, minor);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    for (const void* f : {reinterpret_cast<const void*>(gdn::gdn_prefill_kernel<true, false>),
                          reinterpret_cast<const void*>(gdn::gdn_prefill_kernel<true, false, true>),
                          reinterpret_cast<const void*>(gdn::gdn_prefill_kernel<true, true>),
                          reinterpret_cast<const void*>(gdn::gdn_prefill_kernel<false, false>),
                          reinterpret_cast<const void*>(gdn::gdn_prefill_kernel<false, false, false, true>),
                          reinterpret_cast<const void*>(gdn::gdn_prefill_kernel<false, true>)}) {
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, gdn::Plan::DYN_SMEM);
      if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    }
    e = cudaFuncSetAttribute(gdn::gdn_wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, gdn::WyPlan::DYN_SMEM);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    const std::pair<const void*, int> bwd[] = {
        {reinterpret_cast<const void*>(gdn::gdn_bwd_dstates_tc_kernel), gdn::DsPlan::DYN_SMEM},
        {reinterpret_cast<const void*>(gdn::gdn_bwd_grads_tc_kernel), gdn::GtPlan::DYN_SMEM}};
    for (const auto& f : bwd) {
      e = cudaFuncSetAttribute(f.first, cudaFuncAttributeMaxDynamicSharedMemorySize, f.second);
      if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    }
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
    d.attrs = true;
  }
  *out = &d;
  return GDN_OK;
}

// Sequences ordered by decreasing length (ties by index), so the longest
// chains start first, and cu_chunks[s] = the number of 64-token chunks in
// sequences 0..s-1 (a negative length counts as none); also validates
// cu_seqlens. One thread per sequence.
__global__ void gdn_schedule_kernel(const int32_t* cu, int B, int T, int32_t* order, int32_t* cu_chunks,
                                    unsigned* status) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= B) return;
  const int a = cu[s], b = cu[s + 1];
  if (a < 0 || b < a || b > T || (s == 0 && a != 0) || (s == B - 1 && b != T)) atomicOr(status, gdn::kStatusBadSeqlens);
  const int len = b - a;
  int rank = 0, before = 0;
  for (int o = 0; o < B; ++o) {
    const int lo = cu[o + 1] - cu[o];
    rank += (lo > len) || (lo == len && o < s);
    if (o <= s && lo > 0) before += (lo + gdn::kChunk - 1) / gdn::kChunk;
  }
  order[rank] = s;
  cu_chunks[s + 1] = before;
  if (s == 0) cu_chunks[0] = 0;
}

// ---- segment-parallel schedule ---------------------------------------------------
// A dense batch with few (sequence, head) chains and long sequences leaves most SMs
// idle in the serial spine. The state map of a run of chunks is affine,
// S_end = M S_start + N (the spine recurrence of ssm_gdn_a3.rs, `gdn_prefill_fla`
// doc comment, stage 2, is linear in S), so each sequence is cut into G segments
// of L chunks:
//   phase 1: for every segment g = 0 .. G-2 the output-free spine kernel runs twice,
//            from S = I with v = 0 (giving M_g) and from S = 0 (giving N_g);
//   combine: X_{g+1} = M_g X_g + N_g in fp32, g = 0 .. G-2 (X_0 = the carried-in
//            state, X_{G-1} lands in the caller's state);
//   phase 2: every segment runs from X_g with its output rows.
// Phase 1 takes chains * 2 (G - 1) CTAs, so G is the largest count with that within
// the SM count, at least kSegMinChunks chunks per segment and at most kSegMaxCount.
constexpr int kSegMinChunks = 8;
constexpr int kSegMaxCount = 8;
constexpr int64_t kStateFloats = static_cast<int64_t>(gdn::kDim) * gdn::kDim;

struct SegPlan {
  int G = 0, L = 0;  // G >= 2 segments of L chunks (the last may be shorter); G = 0: serial
};

SegPlan seg_plan(int B, int T, int nv, int sms) {
  SegPlan sp;
  const int64_t chains = static_cast<int64_t>(B) * nv;
  const int nchunks = static_cast<int>((static_cast<int64_t>(T) + gdn::kChunk - 1) / gdn::kChunk);
  if (chains <= 0 || chains * 2 > sms) return sp;
  int G = static_cast<int>(sms / (2 * chains) + 1);
  if (G > nchunks / kSegMinChunks) G = nchunks / kSegMinChunks;
  if (G > kSegMaxCount) G = kSegMaxCount;
  if (G < 2) return sp;
  const int L = (nchunks + G - 1) / G;
  G = (nchunks + L - 1) / L;
  if (G < 2) return sp;
  sp.G = G;
  sp.L = L;
  return sp;
}

// Workspace of the segment schedule: two segment tables (4 int32 per entry), two
// state-pointer tables, then the X_0..X_{G-2}, M_0..M_{G-2} and N_0..N_{G-2} states.
struct SegLayout {
  size_t tab1 = 0, tab2 = 0, ptr1 = 0, ptr2 = 0, bufs = 0, total = 0;
  int n1 = 0, n2 = 0;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

SegLayout seg_layout(const SegPlan& sp, int B, int nv) {
  SegLayout l;
  if (sp.G < 2) return l;
  l.n1 = B * 2 * (sp.G - 1);
  l.n2 = B * sp.G;
  l.tab1 = 0;
  l.tab2 = align256(l.tab1 + 16 * static_cast<size_t>(l.n1));
  l.ptr1 = align256(l.tab2 + 16 * static_cast<size_t>(l.n2));
  l.ptr2 = align256(l.ptr1 + 8 * static_cast<size_t>(l.n1));
  l.bufs = align256(l.ptr2 + 8 * static_cast<size_t>(l.n2));
  l.total = l.bufs + 3 * static_cast<size_t>(sp.G - 1) * B * nv * kStateFloats * sizeof(float);
  return l;
}

// SM count for the plan: the current device's, or GB300's 152 where no device is
// visible (the workspace query works on a host without a GPU).
int plan_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
    return sms;
  cudaGetLastError();
  return 152;
}

struct SegArgs {
  int B, T, nv, G, L;
  int32_t* tab1;
  int32_t* tab2;
  float** ptr1;
  float** ptr2;
  float* X;  // [G-1][B][nv][128][128]: the states entering segments 0 .. G-2
  float* M;  // [G-1][B][nv][128][128]
  float* N;  // [G-1][B][nv][128][128]
  void* state;  // the caller's state (contiguous, or a table of B pointers)
  int state_is_table;
};

__device__ __forceinline__ float* user_state(const SegArgs& a, int b) {
  return a.state_is_table ? reinterpret_cast<float* const*>(a.state)[b]
                          : reinterpret_cast<float*>(a.state) + static_cast<int64_t>(b) * a.nv * kStateFloats;
}

// Builds both segment tables and pointer tables, sets M = I and N = 0, and copies the
// carried-in state into X_0. Grid-stride over the state buffers.
__global__ void gdn_segment_setup_kernel(const SegArgs a) {
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int per1 = 2 * (a.G - 1), per2 = a.G;
  const int64_t seg_rows = static_cast<int64_t>(a.L) * gdn::kChunk;
  const int64_t head = static_cast<int64_t>(a.nv) * kStateFloats;  // floats per (b) state
  auto seg_len = [&](int g) -> int {
    const int64_t r = static_cast<int64_t>(a.T) - g * seg_rows;
    return static_cast<int>(r < seg_rows ? r : seg_rows);
  };
  auto buf = [&](float* base, int g, int b) { return base + (static_cast<int64_t>(g) * a.B + b) * head; };
  if (tid < static_cast<int64_t>(a.B) * per1) {
    const int b = static_cast<int>(tid / per1), j = static_cast<int>(tid % per1);
    const int g = j >> 1;
    const bool is_m = (j & 1) == 0;
    int32_t* e = a.tab1 + 4 * tid;
    e[0] = static_cast<int32_t>(static_cast<int64_t>(b) * a.T + g * seg_rows);
    e[1] = seg_len(g);
    e[2] = gdn::kSegNoOutput | (is_m ? gdn::kSegZeroValues : 0);
    e[3] = 0;
    a.ptr1[tid] = buf(is_m ? a.M : a.N, g, b);
  }
  if (tid < static_cast<int64_t>(a.B) * per2) {
    const int b = static_cast<int>(tid / per2), g = static_cast<int>(tid % per2);
    int32_t* e = a.tab2 + 4 * tid;
    e[0] = static_cast<int32_t>(static_cast<int64_t>(b) * a.T + g * seg_rows);
    e[1] = seg_len(g);
    e[2] = 0;
    e[3] = 0;
    a.ptr2[tid] = g < a.G - 1 ? buf(a.X, g, b) : user_state(a, b);
  }
  const int64_t nbuf = static_cast<int64_t>(a.G - 1) * a.B * head;
  for (int64_t i = tid; i < nbuf; i += nthreads) {
    const int64_t w = i % kStateFloats;
    a.M[i] = (w / gdn::kDim == w % gdn::kDim) ? 1.f : 0.f;
    a.N[i] = 0.f;
  }
  for (int64_t i = tid; i < static_cast<int64_t>(a.B) * head; i += nthreads) {
    const int b = static_cast<int>(i / head);
    a.X[i] = user_state(a, b)[i % head];  // X_0 is the first block of X
  }
}

// X_{g+1} = M_g X_g + N_g for every (sequence, head), fp32 on the CUDA cores
// (128 x 128 x 128 per head). CTA = one 64 x 64 output tile; thread = 4 x 4.
constexpr int kCombineThreads = 256;
__global__ void __launch_bounds__(kCombineThreads) gdn_segment_combine_kernel(const SegArgs a, int g) {
  __shared__ float sa[64][17];
  __shared__ __align__(16) float sb[16][64];
  const int tile = blockIdx.x & 3, bh = blockIdx.x >> 2;
  const int b = bh / a.nv, h = bh % a.nv;
  const int r0 = (tile >> 1) * 64, c0 = (tile & 1) * 64;
  const int64_t head = static_cast<int64_t>(a.nv) * kStateFloats;
  const int64_t off = (static_cast<int64_t>(g) * a.B + b) * head + static_cast<int64_t>(h) * kStateFloats;
  const float* Mh = a.M + off;
  const float* Nh = a.N + off;
  const float* Xin = a.X + off;
  float* Xout = g + 1 < a.G - 1 ? a.X + off + static_cast<int64_t>(a.B) * head
                                : user_state(a, b) + static_cast<int64_t>(h) * kStateFloats;
  const int tid = threadIdx.x, tr = (tid >> 4) * 4, tc = (tid & 15) * 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < gdn::kDim; k0 += 16) {
    for (int i = tid; i < 64 * 16; i += kCombineThreads) {
      const int r = i >> 4, c = i & 15;
      sa[r][c] = Mh[(r0 + r) * gdn::kDim + k0 + c];
      sb[i >> 6][i & 63] = Xin[(k0 + (i >> 6)) * gdn::kDim + c0 + (i & 63)];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 bv = *reinterpret_cast<const float4*>(&sb[kk][tc]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float av = sa[tr + i][kk];
        acc[i][0] = fmaf(av, bv.x, acc[i][0]);
        acc[i][1] = fmaf(av, bv.y, acc[i][1]);
        acc[i][2] = fmaf(av, bv.z, acc[i][2]);
        acc[i][3] = fmaf(av, bv.w, acc[i][3]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t o = static_cast<int64_t>(r0 + tr + i) * gdn::kDim + c0 + tc + j;
      Xout[o] = acc[i][j] + Nh[o];
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int make_map(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int64_t stride_elems, const char* name) {
  auto fn = encode_fn();
  if (!fn) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride_elems) * 2};
  cuuint32_t box[2] = {64, 64}, estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(GDN_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, static_cast<int>(r));
  return GDN_OK;
}

struct Resolved {
  int64_t q, k, v, g, beta, out;
  int table;
  int l2norm;
};

int validate(const void* q, const void* k, const void* v, const float* g, const float* beta, void* state,
             void* out, int B, int T, int nk, int nv, int dk, int dv, const gdn_strides_t* st, Resolved* r) {
  if (B < 0) return fail(GDN_ERR_ARG, "B = %d is negative", B);
  if (T < 0) return fail(GDN_ERR_ARG, "T = %d is negative", T);
  if (nk <= 0 || nv <= 0) return fail(GDN_ERR_ARG, "head counts nk = %d, nv = %d must be positive", nk, nv);
  if (nv % nk != 0) return fail(GDN_ERR_UNSUPPORTED, "nv = %d is not a multiple of nk = %d (GQA groups)", nv, nk);
  if (dk != gdn::kDim || dv != gdn::kDim)
    return fail(GDN_ERR_UNSUPPORTED, "head dims dk = %d, dv = %d differ from the compile-time tile (128, 128)", dk, dv);
  r->q = st ? st->q : static_cast<int64_t>(nk) * dk;
  r->k = st ? st->k : static_cast<int64_t>(nk) * dk;
  r->v = st ? st->v : static_cast<int64_t>(nv) * dv;
  r->g = st ? st->g : nv;
  r->beta = st ? st->beta : nv;
  r->out = st ? st->out : static_cast<int64_t>(nv) * dv;
  r->table = st ? st->state_is_table : 0;
  r->l2norm = st ? st->qk_l2norm : 0;
  if (r->q < static_cast<int64_t>(nk) * dk || r->q % 8) return fail(GDN_ERR_ARG, "q row stride %lld must be >= nk*dk and a multiple of 8", (long long)r->q);
  if (r->k < static_cast<int64_t>(nk) * dk || r->k % 8) return fail(GDN_ERR_ARG, "k row stride %lld must be >= nk*dk and a multiple of 8", (long long)r->k);
  if (r->v < static_cast<int64_t>(nv) * dv || r->v % 8) return fail(GDN_ERR_ARG, "v row stride %lld must be >= nv*dv and a multiple of 8", (long long)r->v);
  if (r->out < static_cast<int64_t>(nv) * dv || r->out % 8) return fail(GDN_ERR_ARG, "out row stride %lld must be >= nv*dv and a multiple of 8", (long long)r->out);
  if (r->g < nv) return fail(GDN_ERR_ARG, "g row stride %lld must be >= nv", (long long)r->g);
  if (r->beta < nv) return fail(GDN_ERR_ARG, "beta row stride %lld must be >= nv", (long long)r->beta);
  if (r->table != 0 && r->table != 1) return fail(GDN_ERR_ARG, "state_is_table must be 0 or 1");
  if (r->l2norm != 0 && r->l2norm != 1) return fail(GDN_ERR_ARG, "qk_l2norm must be 0 or 1");
  if (B == 0 || T == 0) return GDN_OK;  // nothing to read or write
  if (!q || !k || !v || !g || !beta || !state || !out) return fail(GDN_ERR_ARG, "a required pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(state))
    return fail(GDN_ERR_ARG, "q, k, v, out and the state must be 16-byte aligned");
  return GDN_OK;
}

// WY launch geometry. Items: dense batches every (chunk, v-head); varlen an upper
// bound on them (sum of ceil(len / 64) <= T / 64 + B), whose excess CTAs exit at
// once. The kernel is persistent: a few CTAs per SM walk the items.
int wy_geometry(const DeviceInfo& d, int B, int T, int nv, bool varlen, int* items, int64_t* grid) {
  const int64_t chunks = varlen ? static_cast<int64_t>(T) / gdn::kChunk + B + 1
                                : static_cast<int64_t>((T + gdn::kChunk - 1) / gdn::kChunk) * B;
  if (chunks * nv + static_cast<int64_t>(d.sms) * gdn::kWyCtasPerSm > INT32_MAX)
    return fail(GDN_ERR_UNSUPPORTED, "%lld (chunk, head) items exceed the 2^31 item range", (long long)(chunks * nv));
  *items = static_cast<int>(chunks * nv);
  const int64_t slots = static_cast<int64_t>(d.sms) * gdn::kWyCtasPerSm;
  *grid = *items < slots ? *items : slots;
  return GDN_OK;
}

// One spine launch: the instantiation for output rows (or not) and the fused q/k norms (or
// not); the test instantiation when test hooks are set (output rows, no fused norms).
// `after_wy`: the launch directly follows the WY kernel in the stream and may start while
// that kernel still runs (programmatic stream serialisation). Its CTAs then take SMs as
// the WY kernel's CTAs leave them, set up, load their first tiles and issue their first
// Gram; every access to the T diag(beta) / output rows waits for the WY grid in the
// kernel (tc::grid_dependency_wait).
template <bool kOut, bool kNorm, bool kTest = false>
cudaError_t launch_spine_as(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const CUtensorMap& mt, const gdn::ChunkParams& p, int64_t grid, bool after_wy,
                            cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(gdn::kThreads);
  cfg.dynamicSmemBytes = gdn::Plan::DYN_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_wy ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gdn::gdn_prefill_kernel<kOut, kNorm, kTest>, mq, mk, mv, mt, p);
}

cudaError_t launch_spine(bool out_rows, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mt, const gdn::ChunkParams& p, int64_t grid, cudaStream_t stream,
                         bool after_wy = false) {
  if (out_rows) {
    if (g_hooks.active() && !p.qk_l2norm) return launch_spine_as<true, false, true>(mq, mk, mv, mt, p, grid, after_wy, stream);
    if (p.qk_l2norm) return launch_spine_as<true, true>(mq, mk, mv, mt, p, grid, after_wy, stream);
    return launch_spine_as<true, false>(mq, mk, mv, mt, p, grid, after_wy, stream);
  }
  if (p.qk_l2norm) return launch_spine_as<false, true>(mq, mk, mv, mt, p, grid, after_wy, stream);
  return launch_spine_as<false, false>(mq, mk, mv, mt, p, grid, after_wy, stream);
}

int launch(const void* q, const void* k, const void* v, const float* g, const float* beta, void* state, void* out,
           int B, int T, int nk, int nv, const Resolved& r, const int32_t* cu, int32_t* sched, cudaStream_t stream,
           void* seg_ws = nullptr, size_t seg_ws_bytes = 0, int c_begin = 0, int c_count = 0) {
  DeviceInfo* d = nullptr;
  if (int rc = device_info(&d)) return rc;
  const int64_t rows = cu ? static_cast<int64_t>(T) : static_cast<int64_t>(B) * T;
  if (rows > INT32_MAX) return fail(GDN_ERR_UNSUPPORTED, "%lld token rows exceed the 2^31 TMA coordinate range", (long long)rows);
  CUtensorMap mq, mk, mv, mt;
  if (int rc = make_map(&mq, q, static_cast<int64_t>(nk) * gdn::kDim, rows, r.q, "q")) return rc;
  if (int rc = make_map(&mk, k, static_cast<int64_t>(nk) * gdn::kDim, rows, r.k, "k")) return rc;
  if (int rc = make_map(&mv, v, static_cast<int64_t>(nv) * gdn::kDim, rows, r.v, "v")) return rc;
  // the output rows, read back as 16-bit T diag(beta) tiles
  if (int rc = make_map(&mt, out, static_cast<int64_t>(nv) * gdn::kDim, rows, r.out, "out")) return rc;
  int32_t* order = cu ? sched : nullptr;
  int32_t* cu_chunks = cu ? sched + B : nullptr;

  gdn::WyParams w;
  w.g = g;
  w.beta = beta;
  w.tb = static_cast<uint16_t*>(out);
  w.cu_seqlens = cu;
  w.cu_chunks = cu_chunks;
  w.status = d->status;
  w.g_stride = r.g;
  w.beta_stride = r.beta;
  w.out_stride = r.out;
  w.B = B;
  w.T = T;
  w.nk = nk;
  w.nv = nv;
  w.chunks_per_seq = (T + gdn::kChunk - 1) / gdn::kChunk;
  w.chunk_begin = 0;
  w.qk_l2norm = r.l2norm;
  w.t_only = 0;
  int64_t wy_grid = 0;
  if (int rc = wy_geometry(*d, B, T, nv, cu != nullptr, &w.items, &wy_grid)) return rc;
  if (c_count > 0 && !cu) {  // dense: only the chunk range [c_begin, c_begin + c_count) of every sequence
    w.chunk_begin = c_begin;
    w.chunks_per_seq = c_count;
    w.items = static_cast<int>(static_cast<int64_t>(B) * c_count * nv);
    const int64_t slots = static_cast<int64_t>(d->sms) * gdn::kWyCtasPerSm;
    wy_grid = w.items < slots ? w.items : slots;
  }

  gdn::ChunkParams p;
  p.g = g;
  p.state = state;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.cu_seqlens = cu;
  p.order = order;
  p.status = d->status;
  p.g_stride = r.g;
  p.out_stride = r.out;
  p.B = B;
  p.T = T;
  p.nk = nk;
  p.nv = nv;
  p.state_is_table = r.table;
  p.qk_l2norm = r.l2norm;
  p.seg = nullptr;
  p.chunk_begin = c_count > 0 && !cu ? c_begin : 0;
  p.chunk_count = c_count > 0 && !cu ? c_count : 0;
  p.test_wait_ns = g_hooks.wait_ns > 0 ? g_hooks.wait_ns : static_cast<int64_t>(gdn::kWaitLimitNs);
  p.test_delay_ns = g_hooks.delay_ns;
  p.test_skip_chunk = g_hooks.skip_chunk;
  int launches = 0;
  if (cu) {
    gdn_schedule_kernel<<<(B + 255) / 256, 256, 0, stream>>>(cu, B, T, order, cu_chunks, d->status);
    ++launches;
  }
  if (g_timing[0]) cudaEventRecord(g_timing[0], stream);
  gdn::gdn_wy_kernel<<<static_cast<unsigned>(wy_grid), gdn::kWyThreads, gdn::WyPlan::DYN_SMEM, stream>>>(mk, w);
  ++launches;
  if (g_timing[1]) cudaEventRecord(g_timing[1], stream);
  // one CTA per (sequence, v-head); CTAs of the same sequence and GQA group are
  // adjacent so their shared q/k tiles meet in L2
  const SegPlan sp = cu ? SegPlan() : seg_plan(B, T, nv, d->sms);
  const SegLayout sl = seg_layout(sp, B, nv);
  if (sp.G >= 2 && seg_ws && seg_ws_bytes >= sl.total) {
    // segment-parallel schedule (see seg_plan): setup, phase 1, the combine steps, phase 2
    char* w8 = static_cast<char*>(seg_ws);
    SegArgs a;
    a.B = B;
    a.T = T;
    a.nv = nv;
    a.G = sp.G;
    a.L = sp.L;
    a.tab1 = reinterpret_cast<int32_t*>(w8 + sl.tab1);
    a.tab2 = reinterpret_cast<int32_t*>(w8 + sl.tab2);
    a.ptr1 = reinterpret_cast<float**>(w8 + sl.ptr1);
    a.ptr2 = reinterpret_cast<float**>(w8 + sl.ptr2);
    const size_t blk = static_cast<size_t>(sp.G - 1) * B * nv * kStateFloats;
    a.X = reinterpret_cast<float*>(w8 + sl.bufs);
    a.M = a.X + blk;
    a.N = a.M + blk;
    a.state = state;
    a.state_is_table = r.table;
    gdn_segment_setup_kernel<<<d->sms * 4, 256, 0, stream>>>(a);
    ++launches;
    gdn::ChunkParams ps = p;
    ps.cu_seqlens = nullptr;
    ps.order = nullptr;
    ps.state_is_table = 1;
    ps.T = static_cast<int>(rows);
    ps.seg = a.tab1;
    ps.state = a.ptr1;
    ps.B = sl.n1;
    if (cudaError_t e = launch_spine(false, mq, mk, mv, mt, ps, static_cast<int64_t>(sl.n1) * nv, stream))
      return fail(GDN_ERR_CUDA, "spine launch: %s", cudaGetErrorString(e));
    ++launches;
    for (int gs = 0; gs <= sp.G - 2; ++gs) {
      gdn_segment_combine_kernel<<<static_cast<unsigned>(B * nv * 4), kCombineThreads, 0, stream>>>(a, gs);
      ++launches;
    }
    ps.seg = a.tab2;
    ps.state = a.ptr2;
    ps.B = sl.n2;
    if (cudaError_t e = launch_spine(true, mq, mk, mv, mt, ps, static_cast<int64_t>(sl.n2) * nv, stream))
      return fail(GDN_ERR_CUDA, "spine launch: %s", cudaGetErrorString(e));
    ++launches;
  } else {
    const int64_t grid = static_cast<int64_t>(B) * nv;
    if (grid > INT32_MAX) return fail(GDN_ERR_UNSUPPORTED, "grid of %lld CTAs too large", (long long)grid);
    // Overlapped with the WY kernel's tail unless an event must separate the two, and only
    // where placement cannot matter. A dependent launch puts the spine's CTAs on the first
    // SMs the WY kernel frees, and those come in groups: a grid that covers part of the
    // GPU then lands on fewer, fuller GPCs, whose SMs share the instruction cache behind
    // their own, and its chain runs slower (measured at T = 8192: 64, 96 and 128 CTAs
    // lost 22-79 us against a serialised launch; 8, 32, 152 and 160 CTAs gained 3-9 us).
    const bool dependent = g_timing[1] == nullptr && (grid >= d->sms || grid * 4 <= d->sms);
    if (cudaError_t e = launch_spine(true, mq, mk, mv, mt, p, grid, stream, dependent))
      return fail(GDN_ERR_CUDA, "spine launch: %s", cudaGetErrorString(e));
    ++launches;
  }
  if (g_timing[2]) cudaEventRecord(g_timing[2], stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  g_launches = launches;
  return GDN_OK;
}

// varlen: the sequence order (B int32) followed by the chunk prefix (B + 1 int32);
// dense: the segment schedule's tables and states when seg_plan cuts the sequences
// (0 when it does not)
size_t workspace_bytes(int B, int T, int nv, int varlen) {
  if (B <= 0) return 0;
  if (!varlen) return seg_layout(seg_plan(B, T, nv, plan_sms()), B, nv).total;
  return ((2 * static_cast<size_t>(B) + 1) * sizeof(int32_t) + 255) & ~static_cast<size_t>(255);
}

// ---- allocation-free entry point -------------------------------------------------
// Scratch for gdn_prefill_noalloc: the varlen schedule (the sequence order
// and the chunk prefix, 2B + 1 int32) lives in this file-scope device array
// instead of a workspace. Every GPU that loads the library holds it until the
// process exits.
constexpr int kNoAllocMaxSeqs = GDN_NOALLOC_MAX_SEQS;
static __device__ __align__(256) int32_t g_noalloc_order[2 * kNoAllocMaxSeqs + 1];
int32_t* g_noalloc_ptr[kMaxDevices] = {};

// Device address of g_noalloc_order on the current device, looked up once
// per device. In host code the array's name only stands in for the symbol;
// the kernel must be given the address cudaGetSymbolAddress returns.
int noalloc_scratch(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_order);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetSymbolAddress(schedule scratch): %s", cudaGetErrorString(e));
    g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return GDN_OK;
}

// ---- backward -------------------------------------------------------------------
// Scratch of the chunked backward: the varlen schedule; T (16-bit, rows x nv x 128),
// u and du' (fp16, same shape); each chunk's S0 and dS_end (fp16 128 x 128 per
// (chunk slot, v-head), rows / 64 + B + 1 slots).
struct BwdLayout {
  size_t sched = 0, tm = 0, u = 0, du = 0, s0 = 0, ds = 0, total = 0;
};

BwdLayout bwd_layout(int B, int T, int nv, int varlen) {
  BwdLayout l;
  const size_t rows = varlen ? static_cast<size_t>(T) : static_cast<size_t>(B) * T;
  const size_t slots = rows / gdn::kChunk + B + 1;
  const size_t row16 = rows * nv * gdn::kDim * 2;
  const size_t state16 = slots * nv * static_cast<size_t>(kStateFloats) * 2;
  l.sched = 0;
  l.tm = align256(varlen ? (2 * static_cast<size_t>(B) + 1) * sizeof(int32_t) : 0);
  l.u = align256(l.tm + row16);
  l.du = align256(l.u + row16);
  l.s0 = align256(l.du + row16);
  l.ds = align256(l.s0 + state16);
  l.total = align256(l.ds + state16);
  return l;
}

// ---- end-to-end entry point from page-locked host memory (gdn_prefill_host) ---------

// Device staging: packed copies of q, k, v, g, beta, the state and the output rows,
// cu_seqlens, then the op's own workspace; 256-byte aligned parts.
struct HostLayout {
  size_t q = 0, k = 0, v = 0, g = 0, beta = 0, state = 0, out = 0, cu = 0, ws = 0, ws_bytes = 0, total = 0;
};

HostLayout host_layout(int B, int T, int nk, int nv, bool varlen) {
  HostLayout l;
  const size_t rows = varlen ? static_cast<size_t>(T) : static_cast<size_t>(B) * T;
  const size_t qk = rows * nk * gdn::kDim * 2, vo = rows * nv * gdn::kDim * 2, gb = rows * nv * sizeof(float);
  l.k = align256(l.q + qk);
  l.v = align256(l.k + qk);
  l.g = align256(l.v + vo);
  l.beta = align256(l.g + gb);
  l.state = align256(l.beta + gb);
  l.out = align256(l.state + static_cast<size_t>(B) * nv * kStateFloats * sizeof(float));
  l.cu = align256(l.out + vo);
  l.ws = align256(l.cu + (varlen ? (static_cast<size_t>(B) + 1) * sizeof(int32_t) : 0));
  l.ws_bytes = workspace_bytes(B, T, nv, varlen);
  l.total = align256(l.ws + l.ws_bytes);
  return l;
}

int check_pinned(const void* p, const char* name) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(GDN_ERR_ARG, "%s: cudaPointerGetAttributes: %s", name, cudaGetErrorString(e));
  }
  if (a.type != cudaMemoryTypeHost)
    return fail(GDN_ERR_ARG, "%s must be page-locked host memory (cudaHostAlloc or cudaHostRegister)", name);
  return GDN_OK;
}

int copy_streams(DeviceInfo* d) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  for (cudaStream_t* s : {&d->copy_in, &d->copy_out}) {
    if (*s) continue;
    cudaError_t e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaStreamCreateWithFlags: %s", cudaGetErrorString(e));
  }
  return GDN_OK;
}

// Rows [r0, r1) of every sequence of a dense [B][T][row_bytes] tensor, in one strided
// copy (one block of rows per sequence; per sequence when the pitch is too wide).
cudaError_t copy_rows(void* dst, const void* src, size_t row_bytes, int B, int T, int r0, int r1, cudaMemcpyKind kind,
                      cudaStream_t s) {
  const size_t pitch = static_cast<size_t>(T) * row_bytes, off = static_cast<size_t>(r0) * row_bytes;
  const size_t width = static_cast<size_t>(r1 - r0) * row_bytes;
  if (pitch < (static_cast<size_t>(1) << 31))
    return cudaMemcpy2DAsync(static_cast<char*>(dst) + off, pitch, static_cast<const char*>(src) + off, pitch, width,
                             static_cast<size_t>(B), kind, s);
  for (int b = 0; b < B; ++b)
    if (cudaError_t e = cudaMemcpyAsync(static_cast<char*>(dst) + b * pitch + off,
                                        static_cast<const char*>(src) + b * pitch + off, width, kind, s))
      return e;
  return cudaSuccess;
}

// Chunk ranges of the pipelined path: a dense batch of at least 32 chunks per sequence
// that does not take the segment schedule is cut into 2-8 ranges of >= 16 chunks, so
// each range's copies in overlap the op and the copies out of the ranges before it.
// (B=4 T=8192 nv=32, ms per call: 1 range 4.73, 4 ranges 3.50, 8 ranges 3.34, 16 ranges
// 3.36, 32 ranges 3.61.)
int host_ranges(int B, int T, int nv, int sms) {
  const int nchunks = static_cast<int>((static_cast<int64_t>(T) + gdn::kChunk - 1) / gdn::kChunk);
  if (nchunks < 32 || seg_plan(B, T, nv, sms).G >= 2) return 1;
  const int n = nchunks / 16;
  return n < 2 ? 2 : (n > 8 ? 8 : n);
}

}  // namespace

extern "C" {

size_t gdn_prefill_workspace_bytes(int B, int T, int nv, int dk, int dv, int varlen) {
  (void)dk;
  (void)dv;
  if (T < 0 || nv <= 0) return 0;
  return workspace_bytes(B, T, nv, varlen);
}

int gdn_prefill_ex(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   void* h_state_inout, void* out, int B, int T, int nk, int nv, int dk, int dv,
                   const gdn_strides_t* strides, const int32_t* cu_seqlens, void* workspace, size_t workspace_bytes_,
                   void* stream) {
  g_err[0] = 0;
  g_launches = 0;
  Resolved r;
  if (int rc = validate(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, dk, dv, strides, &r)) return rc;
  if (B == 0 || (T == 0 && !cu_seqlens)) return GDN_OK;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return fail(GDN_ERR_ARG, "workspace must be 256-byte aligned");
  if (cu_seqlens) {
    const size_t need = workspace_bytes(B, T, nv, 1);
    if (workspace_bytes_ < need) return fail(GDN_ERR_ARG, "workspace of %zu bytes is smaller than the %zu required", workspace_bytes_, need);
    if (need && !workspace) return fail(GDN_ERR_ARG, "workspace is NULL but %zu bytes are required", need);
    if (T == 0) return GDN_OK;  // varlen with no rows: every sequence is empty
    return launch(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, r, cu_seqlens, static_cast<int32_t*>(workspace),
                  static_cast<cudaStream_t>(stream));
  }
  // dense: the workspace is optional; with enough of it long sequences run segment-parallel
  return launch(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, r, nullptr, nullptr,
                static_cast<cudaStream_t>(stream), workspace, workspace ? workspace_bytes_ : 0);
}

int gdn_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta, void* h_state_inout,
                void* out, int B, int T, int nk, int nv, int dk, int dv, const gdn_strides_t* strides,
                const int32_t* cu_seqlens, void* stream) {
  g_err[0] = 0;
  g_launches = 0;
  Resolved r;
  if (int rc = validate(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, dk, dv, strides, &r)) return rc;
  if (B == 0 || T == 0) return GDN_OK;
  const size_t need = workspace_bytes(B, T, nv, cu_seqlens != nullptr);
  void* ws = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (need) {
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaMallocAsync(%zu): %s", need, cudaGetErrorString(e));
  }
  int rc = cu_seqlens ? launch(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, r, cu_seqlens, static_cast<int32_t*>(ws), s)
                      : launch(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, r, nullptr, nullptr, s, ws, need);
  if (ws) {
    cudaError_t e = cudaFreeAsync(ws, s);
    if (e != cudaSuccess && rc == GDN_OK) rc = fail(GDN_ERR_CUDA, "cudaFreeAsync: %s", cudaGetErrorString(e));
  }
  return rc;
}

int gdn_prefill_noalloc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        void* h_state_inout, void* out, int B, int T, int nk, int nv, int dk, int dv,
                        const gdn_strides_t* strides, const int32_t* cu_seqlens, void* stream) {
  g_err[0] = 0;
  g_launches = 0;
  Resolved r;
  if (int rc = validate(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, dk, dv, strides, &r)) return rc;
  if (B == 0 || T == 0) return GDN_OK;
  int32_t* order = nullptr;
  if (cu_seqlens) {
    if (B > kNoAllocMaxSeqs)
      return fail(GDN_ERR_UNSUPPORTED, "gdn_prefill_noalloc handles at most %d sequences per varlen call, got B = %d",
                  kNoAllocMaxSeqs, B);
    if (int rc = noalloc_scratch(&order)) return rc;
  }
  return launch(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, r, cu_seqlens, order,
                static_cast<cudaStream_t>(stream));
}

size_t gdn_prefill_host_scratch_bytes(int B, int T, int nk, int nv, int dk, int dv, int varlen) {
  if (B < 0 || T < 0 || nk <= 0 || nv <= 0 || dk != gdn::kDim || dv != gdn::kDim) return 0;
  return host_layout(B, T, nk, nv, varlen != 0).total;
}

int gdn_prefill_host(const void* q, const void* k, const void* v, const float* g, const float* beta,
                     void* h_state_inout, void* out, int B, int T, int nk, int nv, int dk, int dv,
                     const gdn_strides_t* strides, const int32_t* cu_seqlens, void* scratch, size_t scratch_bytes,
                     void* stream) {
  g_err[0] = 0;
  g_launches = 0;
  Resolved r;
  if (int rc = validate(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, dk, dv, strides, &r)) return rc;
  if (r.table) return fail(GDN_ERR_UNSUPPORTED, "gdn_prefill_host takes a contiguous state (state_is_table = 0)");
  if (r.q != static_cast<int64_t>(nk) * dk || r.k != static_cast<int64_t>(nk) * dk || r.v != static_cast<int64_t>(nv) * dv ||
      r.out != static_cast<int64_t>(nv) * dv || r.g != nv || r.beta != nv)
    return fail(GDN_ERR_UNSUPPORTED, "gdn_prefill_host takes packed rows (q, k: nk*dk; v, out: nv*dv; g, beta: nv)");
  if (B == 0 || T == 0) return GDN_OK;
  if (scratch && (reinterpret_cast<uintptr_t>(scratch) & 255u)) return fail(GDN_ERR_ARG, "scratch must be 256-byte aligned");
  const bool varlen = cu_seqlens != nullptr;
  const HostLayout l = host_layout(B, T, nk, nv, varlen);
  if (scratch && scratch_bytes < l.total)
    return fail(GDN_ERR_ARG, "scratch of %zu bytes is smaller than the %zu required", scratch_bytes, l.total);
  const std::pair<const void*, const char*> host[] = {{q, "q"}, {k, "k"}, {v, "v"}, {g, "g"}, {beta, "beta"},
                                                      {h_state_inout, "h_state_inout"}, {out, "out"},
                                                      {cu_seqlens ? cu_seqlens : q, "cu_seqlens"}};
  for (const auto& h : host)
    if (int rc = check_pinned(h.first, h.second)) return rc;
  DeviceInfo* d = nullptr;
  if (int rc = device_info(&d)) return rc;
  if (int rc = copy_streams(d)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(scratch);
  if (!base) {
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&base), l.total, s);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaMallocAsync(%zu): %s", l.total, cudaGetErrorString(e));
  }
  void *dq = base + l.q, *dkk = base + l.k, *dvv = base + l.v, *dstate = base + l.state, *dout = base + l.out;
  float *dg = reinterpret_cast<float*>(base + l.g), *dbeta = reinterpret_cast<float*>(base + l.beta);
  int32_t* dcu = varlen ? reinterpret_cast<int32_t*>(base + l.cu) : nullptr;
  void* dws = l.ws_bytes ? base + l.ws : nullptr;
  Resolved packed = r;  // the staging rows are packed like the host rows
  const size_t rows = varlen ? static_cast<size_t>(T) : static_cast<size_t>(B) * T;
  const size_t bq = rows * nk * dk * 2, bv = rows * nv * dv * 2, bg = rows * nv * sizeof(float);
  const size_t bs = static_cast<size_t>(B) * nv * kStateFloats * sizeof(float);
  const int nr = varlen ? 1 : host_ranges(B, T, nv, d->sms);
  int rc = GDN_OK, launches = 0;
  cudaError_t e = cudaSuccess;
  auto h2d = [&](void* dst, const void* src, size_t n, cudaStream_t st) {
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st);
  };
  if (nr == 1) {
    // one pass: everything in, the op, everything out, in stream order
    h2d(dq, q, bq, s);
    h2d(dkk, k, bq, s);
    h2d(dvv, v, bv, s);
    h2d(dg, g, bg, s);
    h2d(dbeta, beta, bg, s);
    h2d(dstate, h_state_inout, bs, s);
    if (varlen) h2d(dcu, cu_seqlens, (static_cast<size_t>(B) + 1) * sizeof(int32_t), s);
    if (e != cudaSuccess) rc = fail(GDN_ERR_CUDA, "host to device copy: %s", cudaGetErrorString(e));
    if (rc == GDN_OK) {
      rc = varlen ? launch(dq, dkk, dvv, dg, dbeta, dstate, dout, B, T, nk, nv, packed, dcu, static_cast<int32_t*>(dws), s)
                  : launch(dq, dkk, dvv, dg, dbeta, dstate, dout, B, T, nk, nv, packed, nullptr, nullptr, s, dws, l.ws_bytes);
      launches = g_launches;
    }
    if (rc == GDN_OK) {
      e = cudaMemcpyAsync(out, dout, bv, cudaMemcpyDeviceToHost, s);
      if (e == cudaSuccess) e = cudaMemcpyAsync(h_state_inout, dstate, bs, cudaMemcpyDeviceToHost, s);
      if (e != cudaSuccess) rc = fail(GDN_ERR_CUDA, "device to host copy: %s", cudaGetErrorString(e));
    }
  } else {
    // pipelined: range i's rows are copied in on copy_in, its WY solve and spine run on
    // `stream` once they have landed, and its output rows go back on copy_out once the
    // spine is done, while the next range's rows are already coming in. Events order
    // the three streams; no kernel waits for another.
    const int nchunks = static_cast<int>((static_cast<int64_t>(T) + gdn::kChunk - 1) / gdn::kChunk);
    cudaEvent_t ev[2 * 8 + 3] = {};
    const int nev = 2 * nr + 3;  // start, (in, op) per range, end of copy_in, end of copy_out
    for (int i = 0; i < nev && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(ev[0], s);  // the staging is ours from here
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d->copy_in, ev[0], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d->copy_out, ev[0], 0);
    h2d(dstate, h_state_inout, bs, d->copy_in);
    for (int i = 0; i < nr && e == cudaSuccess && rc == GDN_OK; ++i) {
      const int c0 = static_cast<int>(static_cast<int64_t>(nchunks) * i / nr);
      const int c1 = static_cast<int>(static_cast<int64_t>(nchunks) * (i + 1) / nr);
      const int r0 = c0 * gdn::kChunk, r1 = c1 * gdn::kChunk < T ? c1 * gdn::kChunk : T;
      const std::pair<std::pair<void*, const void*>, size_t> parts[] = {
          {{dq, q}, static_cast<size_t>(nk) * dk * 2}, {{dkk, k}, static_cast<size_t>(nk) * dk * 2},
          {{dvv, v}, static_cast<size_t>(nv) * dv * 2}, {{dg, g}, nv * sizeof(float)},
          {{dbeta, beta}, nv * sizeof(float)}};
      for (const auto& pt : parts)
        if (e == cudaSuccess)
          e = copy_rows(pt.first.first, pt.first.second, pt.second, B, T, r0, r1, cudaMemcpyHostToDevice, d->copy_in);
      if (e == cudaSuccess) e = cudaEventRecord(ev[1 + 2 * i], d->copy_in);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev[1 + 2 * i], 0);
      if (e != cudaSuccess) break;
      rc = launch(dq, dkk, dvv, dg, dbeta, dstate, dout, B, T, nk, nv, packed, nullptr, nullptr, s, nullptr, 0, c0,
                  c1 - c0);
      launches += g_launches;
      if (rc != GDN_OK) break;
      e = cudaEventRecord(ev[2 + 2 * i], s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(d->copy_out, ev[2 + 2 * i], 0);
      if (e == cudaSuccess)
        e = copy_rows(out, dout, static_cast<size_t>(nv) * dv * 2, B, T, r0, r1, cudaMemcpyDeviceToHost, d->copy_out);
    }
    if (e == cudaSuccess && rc == GDN_OK) e = cudaMemcpyAsync(h_state_inout, dstate, bs, cudaMemcpyDeviceToHost, d->copy_out);
    // the call ends on `stream` once both copy streams have (also after an error, so that
    // nothing uses the staging once `stream` passes the call)
    for (int j = 0; j < 2; ++j) {
      cudaEvent_t end = ev[nev - 2 + j];
      if (!end) continue;
      cudaError_t je = cudaEventRecord(end, j == 0 ? d->copy_in : d->copy_out);
      if (je == cudaSuccess) je = cudaStreamWaitEvent(s, end, 0);
      if (je != cudaSuccess && e == cudaSuccess) e = je;
    }
    for (int i = 0; i < nev; ++i)
      if (ev[i]) cudaEventDestroy(ev[i]);  // released once the work that records it completes
    if (e != cudaSuccess && rc == GDN_OK) rc = fail(GDN_ERR_CUDA, "pipelined copies: %s", cudaGetErrorString(e));
  }
  if (!scratch) {
    cudaError_t fe = cudaFreeAsync(base, s);
    if (fe != cudaSuccess && rc == GDN_OK) rc = fail(GDN_ERR_CUDA, "cudaFreeAsync: %s", cudaGetErrorString(fe));
  }
  if (rc == GDN_OK) g_launches = launches;
  return rc;
}

int gdn_prefill_check(void* stream) {
  g_err[0] = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  DeviceInfo* d = nullptr;
  if (int rc = device_info(&d)) return rc;
  unsigned st = 0;
  e = cudaMemcpy(&st, d->status, sizeof st, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
  if (st) {
    const unsigned zero = 0;
    e = cudaMemcpy(d->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "clearing the status word: %s", cudaGetErrorString(e));
  }
  if (st & gdn::kStatusTimeout) return fail(GDN_ERR_TIMEOUT, "a bounded on-device wait expired (status 0x%x)", st);
  if (st & gdn::kStatusBadSeqlens)
    return fail(GDN_ERR_DEVICE_STATUS, "cu_seqlens is malformed: not non-decreasing from 0 to T (status 0x%x)", st);
  if (st & gdn::kStatusRange)
    return fail(GDN_ERR_RANGE,
                "an output or final state is not finite: v, the state or an intermediate left the fp16 operand "
                "range (|x| < 65504) (status 0x%x)", st);
  return GDN_OK;
}

int gdn_decode(const void* q, const void* k, const void* v, const float* g, const float* beta, void* h_state_inout,
               void* out, int B, int nk, int nv, int dk, int dv, const gdn_strides_t* strides, void* stream) {
  g_err[0] = 0;
  g_launches = 0;
  Resolved r;
  if (int rc = validate(q, k, v, g, beta, h_state_inout, out, B, 1, nk, nv, dk, dv, strides, &r)) return rc;
  if (B == 0) return GDN_OK;
  DeviceInfo* d = nullptr;
  if (int rc = device_info(&d)) return rc;
  const int64_t grid = static_cast<int64_t>(B) * nv;
  if (grid > INT32_MAX) return fail(GDN_ERR_UNSUPPORTED, "grid of %lld CTAs too large", (long long)grid);
  gdn::DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.g = g;
  p.beta = beta;
  p.state = h_state_inout;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.q_stride = r.q;
  p.k_stride = r.k;
  p.v_stride = r.v;
  p.g_stride = r.g;
  p.beta_stride = r.beta;
  p.out_stride = r.out;
  p.B = B;
  p.nk = nk;
  p.nv = nv;
  p.state_is_table = r.table;
  p.qk_l2norm = r.l2norm;
  gdn::gdn_decode_kernel<<<static_cast<unsigned>(grid), gdn::kDecodeThreads, 0,
                           static_cast<cudaStream_t>(stream)>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  g_launches = 1;
  return GDN_OK;
}

size_t gdn_prefill_backward_workspace_bytes(int B, int T, int nv, int dk, int dv, int varlen) {
  (void)dk;
  (void)dv;
  if (B <= 0 || T <= 0 || nv <= 0) return 0;
  return bwd_layout(B, T, nv, varlen).total;
}

int gdn_prefill_backward(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const void* h0, const float* dout, const float* dST, float* dq, float* dk, float* dv,
                         float* dg, float* dbeta, float* dh0, int B, int T, int nk, int nv, int dk_dim, int dv_dim,
                         const gdn_strides_t* strides, const int32_t* cu_seqlens, void* workspace,
                         size_t workspace_bytes_, void* stream) {
  g_err[0] = 0;
  g_launches = 0;
  Resolved r;
  // dout stands in for `out` in the shared checks (contiguous [rows][nv][128] rows)
  gdn_strides_t st{};
  if (strides) st = *strides;
  else {
    st.q = static_cast<int64_t>(nk) * dk_dim;
    st.k = st.q;
    st.v = static_cast<int64_t>(nv) * dv_dim;
    st.g = nv;
    st.beta = nv;
  }
  st.out = static_cast<int64_t>(nv) * dv_dim;
  if (int rc = validate(q, k, v, g, beta, const_cast<void*>(h0), const_cast<float*>(dout), B, T, nk, nv, dk_dim, dv_dim, &st, &r))
    return rc;
  if (r.l2norm) return fail(GDN_ERR_UNSUPPORTED, "the backward takes already normalised q and k (qk_l2norm = 0)");
  if (B == 0 || T == 0) return GDN_OK;
  if (!dq || !dk || !dv || !dg || !dbeta) return fail(GDN_ERR_ARG, "a gradient output pointer is NULL");
  if (!aligned16(dq) || !aligned16(dk) || !aligned16(dv) || (dST && !aligned16(dST)) || (dh0 && !aligned16(dh0)))
    return fail(GDN_ERR_ARG, "dq, dk, dv, dS_T and dh0 must be 16-byte aligned");
  DeviceInfo* d = nullptr;
  if (int rc = device_info(&d)) return rc;
  const int64_t rows = cu_seqlens ? static_cast<int64_t>(T) : static_cast<int64_t>(B) * T;
  if (rows > INT32_MAX) return fail(GDN_ERR_UNSUPPORTED, "%lld token rows exceed the 2^31 TMA coordinate range", (long long)rows);
  const BwdLayout l = bwd_layout(B, T, nv, cu_seqlens != nullptr);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap mq, mk, mv;
  if (int rc = make_map(&mq, q, static_cast<int64_t>(nk) * gdn::kDim, rows, r.q, "q")) return rc;
  if (int rc = make_map(&mk, k, static_cast<int64_t>(nk) * gdn::kDim, rows, r.k, "k")) return rc;
  if (int rc = make_map(&mv, v, static_cast<int64_t>(nv) * gdn::kDim, rows, r.v, "v")) return rc;
  gdn::WyParams w;
  int64_t wy_grid = 0;
  if (int rc = wy_geometry(*d, B, T, nv, cu_seqlens != nullptr, &w.items, &wy_grid)) return rc;
  // (chunk, key head) items: the WY kernel's chunk count (or its varlen bound) times nk
  const int64_t grad_items = static_cast<int64_t>(w.items) / nv * nk;
  if (static_cast<int64_t>(B) * nv > INT32_MAX) return fail(GDN_ERR_UNSUPPORTED, "too many (sequence, head) chains");
  void* ws = workspace;
  if (ws) {
    if (workspace_bytes_ < l.total)
      return fail(GDN_ERR_ARG, "workspace of %zu bytes is smaller than the %zu required", workspace_bytes_, l.total);
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(GDN_ERR_ARG, "workspace must be 256-byte aligned");
  } else {
    cudaError_t e = cudaMallocAsync(&ws, l.total, s);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaMallocAsync(%zu): %s", l.total, cudaGetErrorString(e));
  }
  char* w8 = static_cast<char*>(ws);
  // the WY kernel's T rows (16-bit), read back by the forward chain's copies
  CUtensorMap mt;
  if (int rc = make_map(&mt, w8 + l.tm, static_cast<int64_t>(nv) * gdn::kDim, rows, static_cast<int64_t>(nv) * gdn::kDim,
                        "T")) {
    if (!workspace) cudaFreeAsync(ws, s);
    return rc;
  }
  int32_t* sched = cu_seqlens ? reinterpret_cast<int32_t*>(w8 + l.sched) : nullptr;
  int32_t* order = sched;
  int32_t* cu_chunks = sched ? sched + B : nullptr;

  w.g = g;
  w.beta = beta;
  w.tb = reinterpret_cast<uint16_t*>(w8 + l.tm);
  w.cu_seqlens = cu_seqlens;
  w.cu_chunks = cu_chunks;
  w.status = d->status;
  w.g_stride = r.g;
  w.beta_stride = r.beta;
  w.out_stride = static_cast<int64_t>(nv) * gdn::kDim;
  w.B = B;
  w.T = T;
  w.nk = nk;
  w.nv = nv;
  w.chunks_per_seq = (T + gdn::kChunk - 1) / gdn::kChunk;
  w.chunk_begin = 0;
  w.qk_l2norm = 0;
  w.t_only = 1;

  gdn::BwdChunkParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.g = g;
  p.beta = beta;
  p.h0 = h0;
  p.dout = dout;
  p.dst = dST;
  p.tm = w.tb;
  p.ubuf = reinterpret_cast<__half*>(w8 + l.u);
  p.dubuf = reinterpret_cast<__half*>(w8 + l.du);
  p.s0buf = reinterpret_cast<__half*>(w8 + l.s0);
  p.dsbuf = reinterpret_cast<__half*>(w8 + l.ds);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dg = dg;
  p.dbeta = dbeta;
  p.dh0 = dh0;
  p.cu_seqlens = cu_seqlens;
  p.order = order;
  p.cu_chunks = cu_chunks;
  p.status = d->status;
  p.q_stride = r.q;
  p.k_stride = r.k;
  p.v_stride = r.v;
  p.g_stride = r.g;
  p.beta_stride = r.beta;
  p.B = B;
  p.T = T;
  p.nk = nk;
  p.nv = nv;
  p.state_is_table = r.table;

  int launches = 0;
  if (cu_seqlens) {
    gdn_schedule_kernel<<<(B + 255) / 256, 256, 0, s>>>(cu_seqlens, B, T, order, cu_chunks, d->status);
    ++launches;
  }
  gdn::gdn_wy_kernel<<<static_cast<unsigned>(wy_grid), gdn::kWyThreads, gdn::WyPlan::DYN_SMEM, s>>>(mk, w);
  const unsigned chains = static_cast<unsigned>(static_cast<int64_t>(B) * nv);
  // the forward chain: the output-free spine, storing each chunk's entry state and u
  gdn::ChunkParams fc{};
  fc.g = g;
  fc.state = const_cast<void*>(h0);
  fc.out = nullptr;
  fc.cu_seqlens = cu_seqlens;
  fc.order = order;
  fc.status = d->status;
  fc.g_stride = r.g;
  fc.out_stride = 0;
  fc.B = B;
  fc.T = T;
  fc.nk = nk;
  fc.nv = nv;
  fc.state_is_table = r.table;
  fc.qk_l2norm = 0;
  fc.seg = nullptr;
  fc.test_wait_ns = static_cast<int64_t>(gdn::kWaitLimitNs);
  fc.test_delay_ns = 0;
  fc.test_skip_chunk = -1;
  fc.beta = beta;
  fc.beta_stride = r.beta;
  fc.s0buf = p.s0buf;
  fc.ubuf = p.ubuf;
  gdn::gdn_prefill_kernel<false, false, false, true><<<chains, gdn::kThreads, gdn::Plan::DYN_SMEM, s>>>(mq, mk, mv, mt, fc);
  gdn::gdn_bwd_dstates_tc_kernel<<<chains, gdn::kDsThreads, gdn::DsPlan::DYN_SMEM, s>>>(mq, mk, p);
  gdn::gdn_bwd_grads_tc_kernel<<<static_cast<unsigned>(grad_items), gdn::kGtThreads, gdn::GtPlan::DYN_SMEM, s>>>(p);
  launches += 4;
  int rc = GDN_OK;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) rc = fail(GDN_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  if (!workspace) {
    e = cudaFreeAsync(ws, s);
    if (e != cudaSuccess && rc == GDN_OK) rc = fail(GDN_ERR_CUDA, "cudaFreeAsync: %s", cudaGetErrorString(e));
  }
  if (rc == GDN_OK) g_launches = launches;
  return rc;
}

const char* gdn_last_error(void) { return g_err; }

int gdn_last_launch_count(void) { return g_launches; }

int gdn_set_test_hooks(int64_t wait_limit_ns, int64_t consumer_delay_ns, int skip_hand_off_chunk) {
  g_err[0] = 0;
  if (wait_limit_ns < 0 || consumer_delay_ns < 0 || skip_hand_off_chunk < -1)
    return fail(GDN_ERR_ARG, "test hooks: limits must be >= 0 and the skipped chunk >= -1");
  if (consumer_delay_ns > 100000000)
    return fail(GDN_ERR_ARG, "test hooks: a consumer delay above 100 ms per chunk is refused");
  g_hooks.wait_ns = wait_limit_ns;
  g_hooks.delay_ns = consumer_delay_ns;
  g_hooks.skip_chunk = skip_hand_off_chunk;
  return GDN_OK;
}

void gdn_set_timing_events(void* before_wy, void* before_spine, void* after_spine) {
  g_timing[0] = static_cast<cudaEvent_t>(before_wy);
  g_timing[1] = static_cast<cudaEvent_t>(before_spine);
  g_timing[2] = static_cast<cudaEvent_t>(after_spine);
}

}  // extern "C"

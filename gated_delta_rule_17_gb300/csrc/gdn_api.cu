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

#include "gdn_prefill.h"
#include "gdn_prefill_kernel.cuh"
#include "gdn_wy_kernel.cuh"
#include "gdn_decode_kernel.cuh"

namespace {

thread_local char g_err[512] = "";
thread_local int g_launches = 0;
thread_local cudaEvent_t g_timing[3] = {nullptr, nullptr, nullptr};  // gdn_set_timing_events

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
    e = cudaFuncSetAttribute(gdn::gdn_prefill_kernel<>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gdn::Plan::DYN_SMEM);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    e = cudaFuncSetAttribute(gdn::gdn_wy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, gdn::WyPlan::DYN_SMEM);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
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

int launch(const void* q, const void* k, const void* v, const float* g, const float* beta, void* state, void* out,
           int B, int T, int nk, int nv, const Resolved& r, const int32_t* cu, int32_t* sched, cudaStream_t stream) {
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
  w.qk_l2norm = r.l2norm;
  // dense: every chunk of every sequence; varlen: an upper bound on the chunk
  // count (sum of ceil(len / 64) <= T / 64 + B), the excess CTAs exit at once
  const int64_t wy_chunks = cu ? static_cast<int64_t>(T) / gdn::kChunk + B + 1
                               : static_cast<int64_t>(w.chunks_per_seq) * B;
  if (wy_chunks * nv + static_cast<int64_t>(d->sms) * gdn::kWyCtasPerSm > INT32_MAX)
    return fail(GDN_ERR_UNSUPPORTED, "%lld (chunk, head) items exceed the 2^31 item range", (long long)(wy_chunks * nv));
  w.items = static_cast<int>(wy_chunks * nv);
  // persistent: a few CTAs per SM walk the items
  const int64_t wy_grid = w.items < static_cast<int64_t>(d->sms) * gdn::kWyCtasPerSm
                              ? w.items : static_cast<int64_t>(d->sms) * gdn::kWyCtasPerSm;

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
  const int64_t grid = static_cast<int64_t>(B) * nv;
  if (grid > INT32_MAX) return fail(GDN_ERR_UNSUPPORTED, "grid of %lld CTAs too large", (long long)grid);
  gdn::gdn_prefill_kernel<><<<static_cast<unsigned>(grid), gdn::kThreads, gdn::Plan::DYN_SMEM, stream>>>(mq, mk, mv, mt,
                                                                                                      p);
  ++launches;
  if (g_timing[2]) cudaEventRecord(g_timing[2], stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  g_launches = launches;
  return GDN_OK;
}

// varlen: the sequence order (B int32) followed by the chunk prefix (B + 1 int32)
size_t workspace_bytes(int B, int varlen) {
  if (!varlen || B <= 0) return 0;
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

}  // namespace

extern "C" {

size_t gdn_prefill_workspace_bytes(int B, int T, int nv, int dk, int dv, int varlen) {
  (void)T;
  (void)nv;
  (void)dk;
  (void)dv;
  return workspace_bytes(B, varlen);
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
  const size_t need = workspace_bytes(B, cu_seqlens != nullptr);
  if (workspace_bytes_ < need) return fail(GDN_ERR_ARG, "workspace of %zu bytes is smaller than the %zu required", workspace_bytes_, need);
  if (need && !workspace) return fail(GDN_ERR_ARG, "workspace is NULL but %zu bytes are required", need);
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return fail(GDN_ERR_ARG, "workspace must be 256-byte aligned");
  if (T == 0) return GDN_OK;  // varlen with no rows: every sequence is empty
  return launch(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, r, cu_seqlens, static_cast<int32_t*>(workspace),
                static_cast<cudaStream_t>(stream));
}

int gdn_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta, void* h_state_inout,
                void* out, int B, int T, int nk, int nv, int dk, int dv, const gdn_strides_t* strides,
                const int32_t* cu_seqlens, void* stream) {
  g_err[0] = 0;
  g_launches = 0;
  Resolved r;
  if (int rc = validate(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, dk, dv, strides, &r)) return rc;
  if (B == 0 || T == 0) return GDN_OK;
  const size_t need = workspace_bytes(B, cu_seqlens != nullptr);
  void* ws = nullptr;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (need) {
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaMallocAsync(%zu): %s", need, cudaGetErrorString(e));
  }
  int rc = launch(q, k, v, g, beta, h_state_inout, out, B, T, nk, nv, r, cu_seqlens, static_cast<int32_t*>(ws), s);
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

const char* gdn_last_error(void) { return g_err; }

int gdn_last_launch_count(void) { return g_launches; }

void gdn_set_timing_events(void* before_wy, void* before_spine, void* after_spine) {
  g_timing[0] = static_cast<cudaEvent_t>(before_wy);
  g_timing[1] = static_cast<cudaEvent_t>(before_spine);
  g_timing[2] = static_cast<cudaEvent_t>(after_spine);
}

}  // extern "C"

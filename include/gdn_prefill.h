/*
 * gdn_prefill.h -- C ABI of the GB300 (sm_103a) chunked gated-delta-rule
 * prefill forward.
 *
 * The operation (GDN prefill op, ssm_gdn_a3.rs, doc comment and problem
 * arguments of `gdn_prefill_fla`): for every sequence s and value head h,
 * with key/query head kh = h / (nv / nk), run the recurrence
 *
 *     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t / sqrt(dk)
 *
 * over the tokens of s, starting from the carried-in state S_0 = h_state[s][h]
 * and leaving S_T there. It is evaluated in chunks of 64 tokens in WY form:
 * a per-chunk triangular solve (the op's recompute_wu stage), a serial state
 * spine over chunks (its chunk_delta_h stage) and the chunk-parallel output
 * (its chunk_fwd_o stage). Here the triangular solve runs chunk-parallel in
 * one kernel (a CTA per chunk and v-head) and hands T diag(beta) to a second,
 * fused kernel (a CTA per sequence and v-head) that forms the WY products,
 * runs the spine and writes the output, so the state and the other stage
 * hand-offs stay on chip.
 *
 * All entry points are plain C; pointers marked "device" are CUDA device
 * (or managed) addresses on the current device, `stream` is a cudaStream_t
 * passed as void* (NULL = legacy default stream).
 */
#ifndef GDN_PREFILL_H
#define GDN_PREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. Host-detectable errors launch nothing. */
enum {
  GDN_OK = 0,
  GDN_ERR_ARG = 1,           /* a NULL pointer, a negative size, a bad stride or alignment */
  GDN_ERR_UNSUPPORTED = 2,   /* dk/dv other than 128, nv not a multiple of nk, no sm_103 device */
  GDN_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (message names it) */
  GDN_ERR_DEVICE_STATUS = 4, /* a kernel found malformed cu_seqlens (reported by gdn_prefill_check) */
  GDN_ERR_TIMEOUT = 5,       /* a bounded on-device wait expired (reported by gdn_prefill_check) */
  GDN_ERR_RANGE = 6          /* an output or final state came out non-finite: an operand left the
                                fp16 range (reported by gdn_prefill_check) */
};

/*
 * Row strides, in elements, between consecutive token rows of each tensor
 * (the op's qk_stride / v_stride / gb_stride arguments; the packed conv layout
 * uses qk_stride = v_stride = conv width and a g/beta stride of 2*nv), and
 * the prologue option.
 *   q, k : bf16 elements; multiple of 8 (16-byte rows for TMA); >= nk*dk
 *   v    : bf16 elements; multiple of 8; >= nv*dv
 *   g, beta : fp32 elements; >= nv
 *   out  : bf16 elements; multiple of 8; >= nv*dv
 *   state_is_table : 0 -> h_state_inout is float[B][nv][dk][dv];
 *                    1 -> h_state_inout is a device array of B device
 *                         pointers, each to one float[nv][dk][dv]
 *   qk_l2norm : 0 -> q and k rows are used as given (already L2-normalised
 *                    by the caller);
 *               1 -> fused prologue: every head row of q and of k is
 *                    normalised inside the kernels, x / sqrt(sum(x^2) + 1e-6)
 *                    in fp32, before any use (the input tensors are not
 *                    modified)
 * Passing NULL for the struct means packed rows (q = k = nk*dk, v = out =
 * nv*dv, g = beta = nv), a contiguous state and no prologue.
 */
typedef struct {
  int64_t q, k, v;
  int64_t g, beta;
  int64_t out;
  int32_t state_is_table;
  int32_t qk_l2norm;
} gdn_strides_t;

/*
 * Enqueue the prefill on `stream` and return; no host synchronisation.
 *
 *   q, k    : device bf16, row r holds nk heads of dk values (head kh at
 *             column kh*dk); rows are already L2-normalised by the caller.
 *   v       : device bf16, row r holds nv heads of dv values.
 *   g       : device fp32 log-decay per (row, v-head), finite and <= 0
 *             (exp(g) is the decay; -inf is not supported).
 *   beta    : device fp32 write strength per (row, v-head), in [0, 1].
 *   h_state_inout : device fp32 state, see state_is_table; read as S_0 and
 *             overwritten with S_T of each sequence, k-major ([dk][dv]).
 *   out     : device bf16 [rows][nv][dv] at row stride strides->out;
 *             every row of every sequence is written, nothing else. The
 *             call also uses these rows as its hand-off between the two
 *             kernels (each chunk's T diag(beta) sits in its own tokens'
 *             rows until their outputs replace it), so `out` must not
 *             overlap any input, and its contents are defined only once the
 *             stream has passed the call.
 *   B, T    : dense (cu_seqlens == NULL): B sequences of T tokens, row
 *             r = b*T + t. Varlen: B sequences packed into T rows in total,
 *             sequence s owns rows [cu_seqlens[s], cu_seqlens[s+1]).
 *   nk, nv  : key/query and value head counts, nv % nk == 0; v-head h reads
 *             q/k head h / (nv / nk).
 *   dk, dv  : must both be 128.
 *   cu_seqlens : device int32 [B+1] (non-decreasing, cu[0] = 0, cu[B] = T)
 *             or NULL. Malformed offsets are detected on the device: the
 *             affected sequences write nothing and gdn_prefill_check reports
 *             GDN_ERR_DEVICE_STATUS.
 *   stream  : cudaStream_t as void*.
 * Numerics: products run on the tensor cores with fp16 operands (split into
 * hi + lo pairs where the output needs it) and fp32 accumulation; the
 * triangular solve and the state are carried in fp32. Inputs must keep |v|,
 * |S| and intermediate values inside the fp16 range (|x| < 65504). This is
 * narrower than bf16's range, so it is checked: an operand outside it turns
 * into inf or NaN on conversion, which reaches the outputs or the final state,
 * and any non-finite value there sets the device status bit that
 * gdn_prefill_check reports as GDN_ERR_RANGE (the state and outputs of that
 * call are then not usable).
 * Allocation: needs gdn_prefill_workspace_bytes() of device scratch, which
 * this call allocates and frees stream-ordered (cudaMallocAsync /
 * cudaFreeAsync); use gdn_prefill_ex to supply it instead.
 * Buffers are owned by the caller and must stay valid until the stream
 * reaches the end of this work. q/k/v/out must be 16-byte aligned.
 */
int gdn_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta,
                void* h_state_inout, void* out, int B, int T, int nk, int nv, int dk, int dv,
                const gdn_strides_t* strides, const int32_t* cu_seqlens, void* stream);

/* Bytes of device scratch gdn_prefill_ex needs for these sizes. Varlen
 * batches: a schedule of 2B + 1 int32 (the sequence order and the chunk
 * prefix over the sequences), rounded up to 256 bytes. Dense batches: 0, or,
 * when the batch has few (sequence, head) chains for the device's SM count and
 * long sequences (at least 2 segments of 8 chunks; B * nv * 2 <= SMs), the
 * segment-parallel schedule's scratch: two segment tables and pointer tables
 * (under 4 KB for small B) plus 3 (G - 1) fp32 states of nv x 128 x 128 per
 * sequence, G being the segment count. The state map of a run of chunks is
 * affine in the entry state (the spine stage of ssm_gdn_a3.rs
 * `gdn_prefill_fla`), so the library computes the segments' maps in
 * parallel, chains the segment entry states, and then runs every segment in
 * parallel. The SM count is the current device's,
 * or 152 when no device is visible. */
size_t gdn_prefill_workspace_bytes(int B, int T, int nv, int dk, int dv, int varlen);

/* gdn_prefill with caller-provided scratch (the GDN prefill op likewise takes
 * its scratch from the caller: ssm_gdn_a3.rs, `gdn_prefill_fla` arguments, the
 * caller-owned `gdn_fla_scratch` buffer arena): `workspace` is a device buffer
 * of at least gdn_prefill_workspace_bytes(...) bytes (may be NULL when that
 * is 0), 256-byte aligned, not used by other work until the stream passes
 * this call. Allocates nothing. Varlen batches require the full size (else
 * GDN_ERR_ARG). For dense batches the workspace is optional: with at least
 * the queried size the segment-parallel schedule runs, with less (or NULL)
 * the serial one; both meet the same tolerances. */
int gdn_prefill_ex(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   void* h_state_inout, void* out, int B, int T, int nk, int nv, int dk, int dv,
                   const gdn_strides_t* strides, const int32_t* cu_seqlens, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Allocation-free variant of gdn_prefill for callers that cannot allocate
 * device memory during the call -- for example a serving process whose
 * device memory is reserved up front by its own allocator, or a latency
 * bound loop where a cudaMalloc could block or fail. It has no counterpart
 * in the GDN prefill op; it exists only so those callers can use the library.
 * Same arguments and semantics as gdn_prefill. The varlen schedule it needs
 * lives in a static device array of 2 * GDN_NOALLOC_MAX_SEQS + 1 int32
 * entries (128 KiB) that each GPU holds from library load until process exit; varlen
 * calls with B > GDN_NOALLOC_MAX_SEQS return GDN_ERR_UNSUPPORTED, dense
 * calls have no limit. It calls no cudaMalloc, cudaFree or other allocating
 * routine. The first call on a device looks up that array's device address
 * (cudaGetSymbolAddress) with the device current; make that first call
 * before any stream capture. All calls on a device share the one array and
 * it keeps the last call's contents (every entry a call uses is rewritten
 * by that call): calls that overlap on the GPU, e.g. on two streams, race on
 * it and must be serialised by the caller. */
#define GDN_NOALLOC_MAX_SEQS 16384
int gdn_prefill_noalloc(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        void* h_state_inout, void* out, int B, int T, int nk, int nv, int dk, int dv,
                        const gdn_strides_t* strides, const int32_t* cu_seqlens, void* stream);

/* End-to-end prefill from page-locked host memory: gdn_prefill over inputs
 * and outputs that live on the host. It has no counterpart in the GDN prefill
 * op, which runs on device buffers; it exists for callers whose tensors are on
 * the host, and is how the library measures its end-to-end throughput.
 *   q, k, v, g, beta, h_state_inout, out, cu_seqlens : host buffers allocated
 *             with cudaHostAlloc / cudaMallocHost or registered with
 *             cudaHostRegister (else GDN_ERR_ARG), laid out as for gdn_prefill
 *             with packed rows (strides NULL or equal to the packed widths) and
 *             a contiguous state (state_is_table 0; else GDN_ERR_UNSUPPORTED).
 *             qk_l2norm is honoured. cu_seqlens may be NULL (dense).
 *   scratch : device buffer of gdn_prefill_host_scratch_bytes() bytes,
 *             256-byte aligned, or NULL (the call then allocates and frees it
 *             stream-ordered on `stream`).
 * Enqueues on `stream` and returns: the copies in, the op and the copies out.
 * A dense batch of at least 32 chunks per sequence that does not take the
 * segment schedule is cut into 2-8 ranges of whole chunks, and the library
 * pipelines them over two internal streams of its own: range i's rows are
 * copied in, its WY solve and spine run on `stream` (the state carried from
 * range to range on the device), and its output rows are copied out while
 * range i + 1's rows come in. The results equal gdn_prefill's bit for bit.
 * Every copy is ordered after the work already on `stream` when the call is
 * made, and `stream` passes the call only after the last copy out, so the
 * usual stream semantics hold: the host buffers must stay valid and unchanged
 * (out and the state unread) until then. Numerics, errors and the device
 * status word are as for gdn_prefill; gdn_last_launch_count counts the
 * kernels (two per range). */
size_t gdn_prefill_host_scratch_bytes(int B, int T, int nk, int nv, int dk, int dv, int varlen);
int gdn_prefill_host(const void* q, const void* k, const void* v, const float* g, const float* beta,
                     void* h_state_inout, void* out, int B, int T, int nk, int nv, int dk, int dv,
                     const gdn_strides_t* strides, const int32_t* cu_seqlens, void* scratch, size_t scratch_bytes,
                     void* stream);

/* Single-token decode step, the recurrent update that follows a prefill in
 * serving (same recurrence and state as gdn_prefill, one token per sequence):
 * for every sequence b and value head h, with kh = h / (nv / nk),
 *     S' = exp(g) S;  S <- S' + beta k (v - k^T S')^T;  o = S^T q / sqrt(dk)
 * on row b of q, k, v, g, beta and out (row strides as for gdn_prefill; the
 * state is h_state_inout[b][h], contiguous or through the pointer table).
 * Same argument rules, numerics (fp32 state, fp32 arithmetic, bf16 output),
 * ownership and error codes as gdn_prefill; allocates nothing; one launch. */
int gdn_decode(const void* q, const void* k, const void* v, const float* g, const float* beta, void* h_state_inout,
               void* out, int B, int nk, int nv, int dk, int dv, const gdn_strides_t* strides, void* stream);

/* Timing hook for profiling harnesses: every later call on this host thread
 * records the given events (cudaEvent_t as void*, created by the caller) on
 * its stream before the WY-solve kernel, between the two kernels and after
 * the spine kernel, so each kernel's device time can be read with
 * cudaEventElapsedTime. Any NULL leaves that point unrecorded; all NULL
 * switches the hook off. The events must outlive the calls that record them.
 * Without the between-kernels event, the spine kernel of a call that has no
 * segment schedule, and whose grid covers every SM or at most a quarter of
 * them, is launched with programmatic stream serialisation: it may start on
 * SMs the WY kernel has left and overlap that kernel's tail (its reads of the
 * WY output wait for the WY grid to complete). With that event set, the two
 * kernels run one after the other. */
void gdn_set_timing_events(void* before_wy, void* before_spine, void* after_spine);

/* Backward of the prefill (the training pass): gradients of a loss L with
 * respect to every input of the recurrence S_t = e^{g_t}(I - beta_t k_t k_t^T)
 * S_{t-1} + beta_t k_t v_t^T, o_t = S_t^T q_t / sqrt(dk) (the forward of
 * ssm_gdn_a3.rs `gdn_prefill_fla`), given dL/do and dL/dS_T. Computed in the
 * same chunked form as the forward: the per-chunk WY inverse T, a forward chain
 * storing each chunk's entry state, a reverse chain storing each chunk's state
 * gradient, and the per-chunk gradients, all on the tensor cores (fp16 or bf16
 * operands, hi + lo pairs where they carry a chain, fp32 accumulation and chain
 * states). The forward's outputs are not needed.
 * Enqueues 4 kernels (5 with cu_seqlens). Scratch: 6 bytes per (row, v-head,
 * column) plus 64 KB per (64-row chunk, v-head).
 *   q, k, v, g, beta, strides, cu_seqlens, B, T, nk, nv, dk, dv: as gdn_prefill
 *             (qk_l2norm must be 0: pass the normalised q and k).
 *   h0     : the INITIAL state (gdn_prefill updates its state in place, so keep a
 *            copy), fp32 [B][nv][128][128] or a table of B pointers (state_is_table).
 *   dout   : fp32 [rows][nv][128], dL/do.
 *   dST    : fp32 [B][nv][128][128] (dL/dS_T) or NULL for zero.
 *   dq, dk : fp32 [rows][nk][128] (summed over the value heads of each key head).
 *   dv     : fp32 [rows][nv][128].      dg, dbeta : fp32 [rows][nv].
 *   dh0    : fp32 [B][nv][128][128] (dL/dS_0) or NULL.
 *   (A well-formed cu_seqlens covers every row; with a malformed one the rows
 *   of the rejected sequences hold unspecified values and the status word says so.)
 *   workspace : device scratch of gdn_prefill_backward_workspace_bytes(...) bytes,
 *            256-byte aligned, or NULL to allocate it stream-ordered.
 * dq, dk, dv, dST and dh0 must be 16-byte aligned. Returns GDN_OK or an error code. */
size_t gdn_prefill_backward_workspace_bytes(int B, int T, int nv, int dk, int dv, int varlen);
int gdn_prefill_backward(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const void* h0, const float* dout, const float* dST, float* dq, float* dk, float* dv,
                         float* dg, float* dbeta, float* dh0, int B, int T, int nk, int nv, int dk_dim, int dv_dim,
                         const gdn_strides_t* strides, const int32_t* cu_seqlens, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Synchronise `stream`, then read and clear the current device's status word
 * that kernels set on malformed cu_seqlens (GDN_ERR_DEVICE_STATUS), on an
 * expired bounded wait (GDN_ERR_TIMEOUT) or on a non-finite output or final
 * state (GDN_ERR_RANGE). The word is shared by all calls on the device since
 * the last check. The device-side counterpart of the op's host guards
 * (ssm_gdn_a3.rs, the named-reject guards around `gdn_tc_spine_reject`):
 * what only the kernels can see is reported here instead of silently. After
 * GDN_ERR_TIMEOUT the call's output rows and state are incomplete (output rows
 * may still hold the WY hand-off words); the next call is unaffected. */
int gdn_prefill_check(void* stream);

/* Message for the last error returned on the calling thread, naming the
 * argument or guard that rejected the call ("" after success); the op's
 * named-reject guards (ssm_gdn_a3.rs, `gdn_tc_spine_reject` and the reasons it
 * logs) likewise name what rejected a launch. Thread-local; valid until the
 * next call on the same thread. */
const char* gdn_last_error(void);

/* Number of kernel launches the last successful call on this thread enqueued
 * (the op's dispatch in ssm_gdn_a3.rs, `gdn_prefill_fla`, is a fixed sequence
 * of stage launches; here 2 for a dense batch, 3 with cu_seqlens, more on the
 * segment-parallel schedule). A measurement aid: bench harnesses count the
 * kernels they time with it. */
int gdn_last_launch_count(void);

/* Test hooks, for the library's own tests only (no counterpart in the op):
 * later gdn_prefill* calls on this host thread run a separate test build of
 * the spine kernel (dense or varlen, without the fused q/k norms) that
 *   - uses wait_limit_ns (> 0) instead of the 2 s limit of every bounded wait,
 *   - makes its consumer warps sleep consumer_delay_ns before the hand-off
 *     wait of every odd chunk (the producer warps then run ahead), and
 *   - skips the producer's hand-off arrival of chunk skip_hand_off_chunk
 *     (>= 0), so that the waits on it expire and the call reports
 *     GDN_ERR_TIMEOUT through gdn_prefill_check.
 * All three off (0, 0, -1) returns to the normal kernel. Delays above 100 ms
 * per chunk are refused (GDN_ERR_ARG). Nothing faults or hangs: expired waits
 * unwind the kernel, which frees its tensor memory and returns. */
int gdn_set_test_hooks(int64_t wait_limit_ns, int64_t consumer_delay_ns, int skip_hand_off_chunk);

#ifdef __cplusplus
}
#endif

#endif /* GDN_PREFILL_H */

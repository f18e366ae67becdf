/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention prefill forward.
 *
 * The operation ("NVIDIA Kernel Design Agents optimize Kimi Delta Attention",
 * sections 01 RESULTS and 03 REWARD HACKING; "Autoresearch on Kimi Delta
 * Attention", section THE MECHANISM): for every sequence s and head h, a dk x dv
 * fp32 state S starts at h0[s,h] (or zero) and, for each token t in order,
 *     qh = q_t / sqrt(|q_t|^2 + KDA_L2_EPS),  kh = k_t / sqrt(|k_t|^2 + KDA_L2_EPS)
 *     S  = (I - beta_t kh kh^T) Diag(exp(g_t)) S + beta_t kh v_t^T
 *     o_t = scale * S^T qh
 * and hT[s,h] receives the final S.  The library computes this chunkwise (64
 * tokens per chunk): the state moves from chunk to chunk in order, in fp32; the
 * work inside a chunk is matrix products on the tensor cores with fp32
 * accumulators, bf16 operands for most, and tf32 inputs for the state update
 * (whose rounding would persist in the state).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers, row-major and contiguous:
 *       q, k : [B, T, H, dk]  (dtype = qkv_dtype)     g : [B, T, H, dk] fp32
 *       v, o : [B, T, H, dv]  (dtype = qkv_dtype)     beta : [B, T, H] fp32
 *       h0, hT : [N, H, dk, dv] fp32
 *   - Fixed length: cu_seqlens == NULL and N == num_seqs == B.
 *     Varlen: B == 1, T = total tokens, cu_seqlens is a DEVICE int32 array of
 *     num_seqs + 1 non-decreasing offsets with cu_seqlens[0] == 0 and
 *     cu_seqlens[num_seqs] == T.  Zero-length sequences are legal (hT = h0).
 *   - Legal inputs: g <= 0 and finite (any depth: deep decays underflow to zero,
 *     never overflow); beta in [0, 1]; any sequence length.
 *   - The caller owns every buffer.  The library allocates no device memory and
 *     keeps no state between calls other than cached device attributes.  All work
 *     is enqueued on `stream`; the call returns without synchronising.
 *   - No exception crosses this boundary and no kernel traps.  Host-side checks
 *     return a status before anything is launched; conditions only the device can
 *     see (malformed cu_seqlens) set an error word in the workspace, read back by
 *     kda_fwd_check().
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (a cudaStream_t); 0 is the legacy default stream. */
typedef void* kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null required pointer, bad size, non-finite scale */
    KDA_ERR_UNSUPPORTED = 2,  /* dk or dv not in {64, 128}, unknown dtype */
    KDA_ERR_ALIGNMENT = 3,    /* a tensor pointer is not 16-byte aligned */
    KDA_ERR_WORKSPACE = 4,    /* workspace null, too small or not 256-byte aligned */
    KDA_ERR_CUDA = 5,         /* a CUDA runtime call failed (launch, attribute, copy) */
    KDA_ERR_DEVICE = 6,       /* the device reported malformed input (kda_fwd_check) */
    KDA_ERR_TOO_LARGE = 7     /* kda_fwd_noalloc: needs more than KDA_NOALLOC_SCRATCH_BYTES */
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_FP32 = 1 } kda_dtype;

/* L2-normalisation epsilon: x / sqrt(sum(x^2) + KDA_L2_EPS).  The pages name the
 * normalisation of q and k but not its epsilon; 1e-6 is the reading taken. */
#define KDA_L2_EPS 1e-6f

/* Tokens per chunk of the chunkwise form (fixed). */
#define KDA_CHUNK 64

/* Device error word bits (kda_fwd_check). */
#define KDA_DEVERR_CU_SEQLENS 0x1u   /* cu_seqlens not 0-based, decreasing, or != T */
#define KDA_DEVERR_TIMEOUT 0x2u      /* a kernel's bounded wait ran out (it left early) */
#define KDA_DEVERR_PLAN 0x4u         /* the schedule did not fit its workspace (a library
                                        fault: the state recurrence did not run) */

/*
 * Bytes of device workspace kda_fwd needs for these sizes (0 on bad sizes).
 * B, T, H: batch, tokens per batch row, heads; num_seqs: N (== B when fixed length).
 * The workspace holds a schedule of chunks and the per-chunk factors of the
 * chunkwise form and, where few long chains may be cut into segments (dk = dv =
 * 128, N * H <= 64), a region for the segments' start states and maps (up to 20 MB);
 * a smaller workspace of at least the rest runs the chains whole.  Its contents are
 * scratch and need no initialisation.
 */
size_t kda_fwd_workspace_size(int B, int T, int H, int dk, int dv, int num_seqs);

/*
 * The KDA prefill forward.  Writes o (dtype qkv_dtype) and, when hT is not NULL,
 * the final states.  h0 may be NULL (zero initial state).  scale multiplies the
 * output (the usual choice is dk^-1/2).  workspace must be 256-byte aligned and at
 * least kda_fwd_workspace_size(...) bytes.  q, k, v, g, o must be 16-byte aligned.
 * Returns KDA_OK once the work is enqueued, or an error status with nothing
 * enqueued.  Calls that share a workspace must be ordered on one stream.
 */
kda_status kda_fwd(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                   const float* g, const float* beta, const float* h0,
                   const int32_t* cu_seqlens, int num_seqs,
                   int B, int T, int H, int dk, int dv, float scale,
                   void* o, float* hT,
                   void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * Synchronises `stream`, then reads the device error word that the last kda_fwd
 * on this workspace left.  Returns KDA_OK, KDA_ERR_DEVICE (and *device_error gets
 * the KDA_DEVERR_* bits, if device_error is not NULL) or KDA_ERR_CUDA.
 */
kda_status kda_fwd_check(const void* workspace, kda_stream_t stream, uint32_t* device_error);

/* Static, human-readable name of a status. */
const char* kda_status_string(kda_status status);

/* Number of kernel launches kda_fwd enqueues for these sizes under the current
 * pipeline setting, with a workspace of kda_fwd_workspace_size bytes (for launch
 * counts): 2 with the fused pipeline (schedule, fused); with the split one 3
 * (schedule, factors, state), 4 when it leaves the choice between the tiled and the
 * 128-column state kernels to the device (both launched), 5 with segments chosen on
 * the host (schedule, factors, pass A, scan, pass C), 6 when the device decides on
 * segments (the tiled state kernel, then the three segment kernels). */
int kda_fwd_launch_count(int B, int T, int H, int dk, int dv, int num_seqs);

/*
 * kda_fwd with the gate g stored as fp32 (g_dtype = KDA_FP32, exactly kda_fwd) or
 * bf16 (g_dtype = KDA_BF16, which needs qkv_dtype = KDA_BF16): a bf16 gate halves
 * the gate's bytes, the largest input at d = 128 ("NVIDIA Kernel Design Agents
 * optimize Kimi Delta Attention", section 01 RESULTS, names the inputs and their
 * dtypes; the gate's dtype is left open there).  The computation is the same, from
 * the gate values as stored.  Other statuses as kda_fwd; an unsupported
 * combination of dtypes is KDA_ERR_UNSUPPORTED.
 */
kda_status kda_fwd_ex(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                      const void* g, kda_dtype g_dtype, const float* beta, const float* h0,
                      const int32_t* cu_seqlens, int num_seqs,
                      int B, int T, int H, int dk, int dv, float scale,
                      void* o, float* hT,
                      void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_fwd_ex, and in addition cudaEventRecord(events[i], stream) just before its
 * i-th kernel launch and events[n] after the last one, n = kda_fwd_launch_count(...),
 * so that a profiler can time each kernel on the stream it runs on.  `events`
 * holds n + 1 caller-created cudaEvent_t handles.  Same arguments and statuses as
 * kda_fwd_ex (KDA_ERR_CUDA if an event record fails).
 */
kda_status kda_fwd_profiled(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                            const void* g, kda_dtype g_dtype, const float* beta, const float* h0,
                            const int32_t* cu_seqlens, int num_seqs,
                            int B, int T, int H, int dk, int dv, float scale,
                            void* o, float* hT,
                            void* workspace, size_t workspace_bytes, kda_stream_t stream,
                            void* const* events);

/*
 * Pipelines of the forward (both compute the same operation; their kernels differ,
 * so results may differ in the last bits):
 *   fused: a schedule kernel, then one persistent cooperative kernel in which some
 *     CTAs produce the per-chunk factors and the others run the state recurrence
 *     over whole (sequence, head) chains, consuming each chunk's factors as soon as
 *     they are published.  Applies to dk = dv = 128, batches of at most 2048
 *     sequences and 65536 (sequence, head) pairs, on a device with 2 to 1025 SMs.
 *   split: a schedule kernel, a factor kernel over every chunk, then a state kernel:
 *     over (sequence, head, value-column tile) chains, or, with dk = dv = 128 where
 *     that is predicted faster, over whole (sequence, head) chains of 128 columns.
 *     The state kernel is chosen on the host for equal-length chains and by the
 *     schedule kernel from the chain lengths for varlen batches of at least 512
 *     (sequence, head) pairs (both are then launched; the one not chosen leaves at
 *     once).  Few long chains (dk = dv = 128, at most 64 (sequence, head) pairs, a
 *     workspace of kda_fwd_workspace_size bytes) are cut into segments where that is
 *     predicted faster: a first pass runs each chain's first segment and, for every
 *     middle segment, its state map and its state from zero; a scan kernel gives
 *     each segment's start state; a second pass reruns the later segments from
 *     those (exact up to rounding: the chunk step is affine in the state).  The
 *     segment length is chosen on the host for equal-length chains, by the schedule
 *     kernel for varlen batches of at least 2048 tokens (the tiled state kernel is
 *     then launched too, and the kernels not chosen leave at once).  Applies to
 *     every size.
 * KDA_PIPELINE_AUTO (default) takes the fused pipeline where it applies and was
 * measured faster on GB300: fixed-length batches (or a single sequence) with
 * 32 <= B * H <= 256 for which the split pipeline would not take the 128-column
 * chain kernel; every other size takes the split one.  KDA_PIPELINE_FUSED
 * takes it wherever it applies, KDA_PIPELINE_SPLIT never, KDA_PIPELINE_SPLIT_WHOLE
 * never and never cuts chains into segments.  The setting is process-wide (an
 * atomic; calls already enqueued keep theirs); it exists for measurement and
 * testing.
 */
typedef enum {
    KDA_PIPELINE_AUTO = 0,
    KDA_PIPELINE_FUSED = 1,
    KDA_PIPELINE_SPLIT = 2,
    KDA_PIPELINE_SPLIT_WHOLE = 3
} kda_pipeline;
void kda_set_pipeline(kda_pipeline pipeline);
kda_pipeline kda_get_pipeline(void);

/* 1 if kda_fwd takes the fused pipeline for these sizes under the current setting
 * (on the current device), else 0.  B == 1 with num_seqs != 1 is a varlen batch. */
int kda_fwd_uses_fused(int B, int T, int H, int dk, int dv, int num_seqs);

/* Size of the device scratch array built into the library for kda_fwd_noalloc. */
#define KDA_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * kda_fwd for callers that cannot allocate device memory.  The pages describe no
 * such entry point; it exists for users of this library, not for the method.
 *
 * Some callers cannot obtain device memory where they run the forward: a plugin
 * inside a host engine that owns every device allocation, code on a path where
 * an allocation's latency or failure is not acceptable, or a runtime whose
 * allocator this library cannot reach.  This entry point takes the same inputs
 * and outputs as kda_fwd but no workspace: it uses a device array of
 * KDA_NOALLOC_SCRATCH_BYTES (32 MiB) built into the library, which every GPU that
 * loads the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Limits and behaviour:
 *   - Problems whose workspace (kda_fwd_workspace_size) exceeds the array are
 *     refused with KDA_ERR_TOO_LARGE before anything is launched; at d = 128 the
 *     array holds about 310 (chunk, head) pairs, e.g. 1,024 tokens x 19 heads.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, and each call's kernels
 *     overwrite it completely before reading it, so nothing needs clearing
 *     between calls.  Calls whose work overlaps on the GPU (different streams
 *     without ordering, or host threads racing) corrupt each other's results:
 *     order them on one stream.
 *   - Conditions only the device can see (malformed cu_seqlens, a bounded wait
 *     that ran out) set the error word in the built-in array; read it with
 *     kda_fwd_noalloc_check() after the call.
 * Statuses are kda_fwd's, plus KDA_ERR_TOO_LARGE.
 */
kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                           const float* g, const float* beta, const float* h0,
                           const int32_t* cu_seqlens, int num_seqs,
                           int B, int T, int H, int dk, int dv, float scale,
                           void* o, float* hT, kda_stream_t stream);

/*
 * The kda_fwd_check of kda_fwd_noalloc: synchronises `stream`, then reads the
 * device error word that the last kda_fwd_noalloc on the current device left in
 * the built-in scratch array.  Returns KDA_OK, KDA_ERR_DEVICE (and *device_error,
 * if not NULL, gets the KDA_DEVERR_* bits) or KDA_ERR_CUDA.  Allocates nothing.
 * The word belongs to the last call on this device, whichever stream made it.
 */
kda_status kda_fwd_noalloc_check(kda_stream_t stream, uint32_t* device_error);

/*
 * One recurrence step per sequence: single-token decode ("Autoresearch on Kimi
 * Delta Attention", section THE MECHANISM: the per-token state update that the
 * chunked prefill batches).  For every sequence n and head h, with S = h_in[n,h]
 * (zeros when h_in is NULL) and that sequence's one token:
 *     qh = q / sqrt(|q|^2 + KDA_L2_EPS),  kh = k / sqrt(|k|^2 + KDA_L2_EPS)
 *     S' = (I - beta kh kh^T) Diag(exp(g)) S + beta kh v^T,   o = scale * S'^T qh
 * h_out[n,h] receives S'.  Every step is fp32 (no tensor cores: the work is one
 * read and one write of the state, bound by HBM bandwidth).
 *
 * Layouts (DEVICE pointers, row-major, contiguous, 16-byte aligned):
 *     q, k : [N, H, dk] (qkv_dtype)   g : [N, H, dk] fp32   beta : [N, H] fp32
 *     v, o : [N, H, dv] (qkv_dtype)   h_in, h_out : [N, H, dk, dv] fp32
 * h_out may be h_in itself (update in place); otherwise the two must not overlap
 * (KDA_ERR_INVALID_ARG).  No workspace; nothing is allocated.  Same legal inputs
 * as kda_fwd.  Statuses: KDA_ERR_INVALID_ARG (null pointer, N < 0, H <= 0,
 * non-finite scale, overlapping states), KDA_ERR_UNSUPPORTED, KDA_ERR_ALIGNMENT,
 * KDA_ERR_CUDA; KDA_OK with nothing enqueued when N == 0.
 */
kda_status kda_decode(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                      const float* g, const float* beta, const float* h_in, float* h_out,
                      int N, int H, int dk, int dv, float scale, void* o, kda_stream_t stream);

/*
 * Backward pass ("Autoresearch on Kimi Delta Attention", sections THE MECHANISM and
 * OPTIMIZATION TRACE: the training-side workload, the state's gradient carried
 * backwards through the chunks): for the forward of kda_fwd on the same inputs,
 * the gradients of  L = sum(o * dout) + sum(h_T * dhT)  with respect to q, k, v, g,
 * beta and h0 (through the L2 normalisations of q and k and alpha = exp(g)).
 *
 * Layouts as kda_fwd (DEVICE pointers, row-major, contiguous, 16-byte aligned):
 *     q, k, dout-like : q, k [B, T, H, dk], v and dout [B, T, H, dv] (qkv_dtype)
 *     g : [B, T, H, dk] fp32      beta : [B, T, H] fp32
 *     h0 : [N, H, dk, dv] fp32 or NULL (zero initial state)
 *     dhT : [N, H, dk, dv] fp32 or NULL (no gradient through h_T)
 * Outputs (fp32, written in full): dq, dk : [B, T, H, dk]; dv : [B, T, H, dv];
 *     dg : [B, T, H, dk]; dbeta : [B, T, H]; dh0 : [N, H, dk, dv] or NULL (not wanted).
 * cu_seqlens as kda_fwd.  Workspace: kda_bwd_workspace_size bytes (for the current
 * device), 256-byte aligned, caller-owned scratch; it holds the state at every
 * chunk start and, per CTA, the states of one chunk.
 *
 * Computation: one CTA per (sequence, head, 32 value columns) at a time (the value
 * columns never mix in the recurrence), fp32 state in registers, fp32 arithmetic
 * on the CUDA cores: the forward recomputed with checkpoints at chunk starts, then
 * every chunk in reverse (its states recomputed, then its tokens in reverse).  The
 * sums over value columns (dq, dk, dg, dbeta) are added tile by tile into the
 * zeroed outputs, so their last bits may differ between runs.  Launches: the
 * schedule kernel, four memsets of those outputs, the backward, a kernel applying
 * the L2 normalisations' derivatives.  Statuses as kda_fwd (malformed cu_seqlens:
 * the device error word, kda_fwd_check).
 */
size_t kda_bwd_workspace_size(int B, int T, int H, int dk, int dv, int num_seqs);
kda_status kda_bwd(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                   const float* g, const float* beta, const float* h0,
                   const int32_t* cu_seqlens, int num_seqs,
                   int B, int T, int H, int dk, int dv, float scale,
                   const void* dout, const float* dhT,
                   float* dq, float* dk_out, float* dv_out, float* dg, float* dbeta, float* dh0,
                   void* workspace, size_t workspace_bytes, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */

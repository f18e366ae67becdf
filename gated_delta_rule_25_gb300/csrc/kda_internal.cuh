// Internal definitions shared by the KDA kernels and the C-ABI layer.
//
// Workspace (caller-owned, 256-byte aligned), carved as:
//   [0, 256)        header: u32 error word, i32 total chunk count, i32 work counter
//   seq_first       int32[N + 1]: index of the first chunk of each sequence
//   order           int32[N]:     sequences by decreasing chunk count (longest first)
//   chunks          int4[Cmax]:   {sequence, first token row, valid rows L, 0}
//   plist           int32[Cmax*H]: the order in which the fused pipeline produces
//                                 (chunk, head) items, each as chunk * H + head
//   ready           u32[Cmax*H]:  per (chunk, head): 1 once its factors are published
//   factors         per (chunk, head): the factors of the chunkwise form
//   (segments, when they may apply: dk = dv = 128 and N * H <= kSegPairs)
//   seg_a, seg_c    int4[kSegTasks] each: the two chain passes' task lists
//   seg_scan        int4[kSegPairs]: the scan's (pair, E slot, F slot, segments)
//   seg_e, seg_f    fp32[slots][dk * dv] and [slots][dk * (dk + kMapPad)]: segment
//                   start states and maps (F^T, rows padded)
//
// Per (chunk, head) factor block, every part a multiple of 256 bytes:
//   WQ  [128 x dk] bf16, M-major operand layout: rows 0-63
//                                       w = (I + A)^-1 Diag(beta) (kh * exp(Gamma)), rows
//                                       64-127 qh * exp(Gamma) (one M = 128 operand)
//   KT  [dk x 64] fp32, tf32 operand layout  (kh * exp(Gamma_last - Gamma))^T
//   P   [64 x 64] bf16, operand layout  sum_c qh_ic kh_jc exp(Gamma_ic - Gamma_jc), j <= i
//   U0  [dv/32][8][64][4] fp32          u = (I + A)^-1 Diag(beta) v, in 32-column
//                                       slabs (one contiguous slab per value tile)
//   GL  [dk] fp32                       exp(Gamma_last)
// KT and u feed the state update, the one product whose rounding persists in the
// state, so they are kept in fp32 and that product runs on tf32 inputs.
//
// "Operand layout" is the K-major, unswizzled tensor-core shared-memory layout for
// an R x K tile: core matrices of 8 rows x 16 contiguous bytes (8 bf16 or 4 fp32
// elements of K), core matrix (row block rb, k block kb) at byte ((kb * R/8) + rb)
// * 128.  A bulk copy of the block lands in shared memory ready for tcgen05.mma,
// with descriptor leading byte offset (between core matrices adjacent in K) = R/8 *
// 128 and stride byte offset (between core matrices adjacent in rows) = 128.
// "M-major operand layout" (WQ): core matrices of 8 K-columns x 16 contiguous bytes
// (8 bf16 elements of M), core matrix (row block mb, k block kb) at byte ((mb *
// dk/8) + kb) * 128; descriptor leading byte offset (K-adjacent) 128, stride byte
// offset (M-adjacent) dk/8 * 128, and the instruction's A-major bit set.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace kda {

constexpr int kChunk = 64;
constexpr int kNV = 32;  // value columns per state-recurrence chain

// Device error word bits (mirrors of the KDA_DEVERR_* values of kda.h).
constexpr unsigned kDevErrCuSeqlens = 0x1u;
constexpr unsigned kDevErrTimeout = 0x2u;
constexpr unsigned kDevErrPlan = 0x4u;

// Element index of (row r, value column n) in the slabbed U0 block (fp32): one
// slab of kChunk x kNV per value tile, inside it groups of 4 columns, each a
// column-group-major [kChunk][4] array, so that consecutive rows of a 4-column
// group are consecutive 16-byte words (conflict-free for a warp of rows).
__host__ __device__ inline int u0_index(int r, int n) {
    return (((n / kNV) * (kNV / 4) + (n % kNV) / 4) * kChunk + r) * 4 + (n & 3);
}

struct Dims {
    int B, T, H, dk, dv, N;
    bool varlen;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Upper bound on the number of chunks over all sequences.
__host__ __device__ inline long long max_chunks(const Dims& d) {
    if (d.varlen) return (long long)d.T / kChunk + d.N;
    return (long long)d.B * ((d.T + kChunk - 1) / kChunk);
}

struct FactorLayout {
    size_t wq, kt, p, u0, gl, bytes;
    __host__ __device__ explicit FactorLayout(int dk, int dv) {
        size_t off = 0;
        wq = off; off += align256(size_t(2 * kChunk) * dk * 2);
        kt = off; off += align256(size_t(dk) * kChunk * 4);
        p = off;  off += align256(size_t(kChunk) * kChunk * 2);
        u0 = off; off += align256(size_t(kChunk) * dv * 4);
        gl = off; off += align256(size_t(dk) * 4);
        bytes = off;
    }
};

// Exact inter-chunk split ("segments") of few long chains, in the split pipeline
// (dk = dv = 128, at most kSegPairs (sequence, head) pairs): each chain is cut into
// segments of L chunks; the chunk step S <- M_c S + D_c is affine, so a middle
// segment k is the map S -> F_k S + Z_k (F_k the product of its M_c, Z_k its state
// from zero).  Pass A runs segment 0 from h0 and F_k, Z_k of the middle segments,
// all at once; a scan then gives every segment's start state; pass C reruns
// segments 1.. from those, writing the outputs and h_T.
constexpr int kSegPairs = 64;    // (sequence, head) pairs, at most
constexpr int kSegTasks = 1024;  // tasks of one pass, at most
constexpr int kSegSlots = 160;   // segment start states (and maps), at most
constexpr int kMapPad = 8;       // a map F^T is stored with rows of dk + kMapPad floats
// Task kinds (int4 {first chunk, chunks, sequence * H + head, kind | last << 3 | slot << 4}).
constexpr int kTaskWhole = 0;  // a whole chain: h0 -> outputs, h_T
constexpr int kTaskHead = 1;   // segment 0: h0 -> outputs, end state to E[slot]
constexpr int kTaskMapF = 2;   // a middle segment's map: identity, u = 0 -> F[slot]
constexpr int kTaskMapZ = 3;   // a middle segment from zero -> E[slot]
constexpr int kTaskTail = 4;   // segment k >= 1: E[slot] -> outputs (h_T when last)

__host__ __device__ inline bool seg_layout_applies(const Dims& d) {
    return d.dk == 128 && d.dv == 128 && (long long)d.N * d.H <= kSegPairs;
}

struct WsLayout {
    size_t header, seq_first, order, chunks, plist, ready, factors, total;
    size_t seg_a, seg_c, seg_scan, seg_e, seg_f, total_seg;
    long long cmax;
    int seg_slots;  // capacity of seg_e and seg_f (0: no segment region)
    size_t factor_bytes;
    __host__ __device__ explicit WsLayout(const Dims& d) {
        cmax = max_chunks(d);
        FactorLayout f(d.dk, d.dv);
        factor_bytes = f.bytes;
        size_t off = 0;
        header = off;    off += 256;
        seq_first = off; off += align256(size_t(d.N + 1) * 4);
        order = off;     off += align256(size_t(d.N) * 4);
        chunks = off;    off += align256(size_t(cmax) * 16);
        plist = off;     off += align256(size_t(cmax) * d.H * 4);
        ready = off;     off += align256(size_t(cmax) * d.H * 4);
        factors = off;   off += size_t(cmax) * d.H * f.bytes;
        total = off;
        const long long pairs_chunks = cmax * d.H;
        seg_slots = seg_layout_applies(d) ? (int)(pairs_chunks < kSegSlots ? pairs_chunks : kSegSlots) : 0;
        off = align256(off);
        seg_a = off;     off += seg_slots ? size_t(kSegTasks) * 16 : 0;
        seg_c = off;     off += seg_slots ? size_t(kSegTasks) * 16 : 0;
        seg_scan = off;  off += seg_slots ? size_t(kSegPairs) * 16 : 0;
        seg_e = off;     off += size_t(seg_slots) * d.dk * d.dv * 4;
        seg_f = off;     off += size_t(seg_slots) * d.dk * (d.dk + kMapPad) * 4;
        total_seg = seg_slots ? off : total;
    }
};

// Element index of (r, k) in an R x K bf16 tile stored in the operand layout.
__host__ __device__ inline int op_index(int r, int k, int R) {
    return (((k >> 3) * (R >> 3) + (r >> 3)) << 6) + ((r & 7) << 3) + (k & 7);
}

// Element index of (r, k) in an R x K fp32 (tf32 operand) tile in the operand layout.
__host__ __device__ inline int op_index32(int r, int k, int R) {
    return (((k >> 2) * (R >> 3) + (r >> 3)) << 5) + ((r & 7) << 2) + (k & 3);
}

struct Header {
    uint32_t error;
    int32_t total_chunks;
    int32_t next_item;  // work counter of the persistent state kernel (reset per call)
    int32_t n_chain;    // fused pipeline: CTAs that run state chains (0: none)
    int32_t chain128;   // split pipeline: 1 when the 128-column chain kernel runs the
                        // state recurrence (and the factors' u is in its layout)
    int32_t seg;        // split pipeline: 1 when segmented chains run the recurrence
                        // (the factors' u then in the 128-column layout too)
    int32_t seg_na, seg_nc, seg_ns;  // tasks of pass A and C, pairs of the scan
    int32_t seg_len;    // chunks per segment
};

// Longest-first ranking covers up to this many sequences (identity order beyond);
// the fused pipeline needs the ranking, so it takes batches of at most this many.
constexpr int kRankMax = 2048;

// Raises a kernel's dynamic shared-memory limit once per device (the attribute
// call is kept out of later calls, which may run under stream capture).
// Bookkeeping is per kernel (keyed by its address) and per device.
cudaError_t ensure_smem_raw(const void* kern, size_t bytes);

// Number of SMs of the current device (cached per device; 152 on GB300).
int num_sms();

template <typename Kernel>
cudaError_t ensure_smem(Kernel kern, size_t bytes) {
    return ensure_smem_raw(reinterpret_cast<const void*>(kern), bytes);
}

// Launchers (each enqueues on `stream`; return cudaGetLastError()).
// Split pipeline.  c128_mode: 0, the tiled state kernel runs (value tiles of
// split_nv_for columns); 1, the 128-column chain kernel runs; 2 (varlen, dk = dv =
// 128), the schedule kernel picks one of the two from the chain lengths and the
// other leaves at once.
cudaError_t launch_schedule(const Dims& d, const int32_t* cu_seqlens, uint8_t* ws, int split_nv,
                            int c128_mode, int seg_len, cudaStream_t stream);
// For equal-length chains (a fixed-length batch or one sequence): whether the
// 128-column chain kernel is predicted faster.
bool chain128_pick_uniform(const Dims& d);
cudaError_t launch_prep_tc(const Dims& d, bool qkv_bf16, bool g_bf16, const void* q, const void* k,
                           const void* v, const void* g, const float* beta, uint8_t* ws,
                           cudaStream_t stream);
cudaError_t launch_chain(const Dims& d, bool qkv_bf16, const float* h0, float scale, void* o,
                         float* hT, uint8_t* ws, cudaStream_t stream);
// Value-tile width of the split state kernel for these sizes (16, 32 or 64).
int split_nv_for(const Dims& d);
// The split pipeline's 128-column chain kernel (dk = dv = 128), which runs only when
// the schedule kernel chose it (Header::chain128); and whether it applies at all.
cudaError_t launch_chain128(const Dims& d, bool qkv_bf16, const float* h0, float scale, void* o,
                            float* hT, uint8_t* ws, cudaStream_t stream);
bool chain128_applies(const Dims& d);

// Segmented chains (split pipeline, seg_layout_applies and a workspace of
// WsLayout::total_seg bytes).  seg_pick_uniform: for chains of equal length, the
// segment length predicted fastest, or 0 where the unsegmented state kernel is
// predicted faster.  The schedule kernel's seg_len: > 0 use it, 0 none, -1 decide
// from the chain lengths.  launch_seg_pass(pass 0 = A, 1 = C) and launch_seg_scan
// run only when the schedule kernel set Header::seg (they leave at once otherwise).
int seg_pick_uniform(const Dims& d);
cudaError_t launch_seg_pass(const Dims& d, bool qkv_bf16, int pass, const float* h0, float scale,
                            void* o, float* hT, uint8_t* ws, cudaStream_t stream);
cudaError_t launch_seg_scan(const Dims& d, uint8_t* ws, cudaStream_t stream);

// Backward pass: workspace bytes for the current device (after the schedule's
// tables), and the launch (after launch_schedule has filled the tables).
size_t bwd_workspace_bytes(const Dims& d);
cudaError_t launch_bwd(const Dims& d, bool qkv_bf16, const int32_t* cu, const void* q, const void* k,
                       const void* v, const float* g, const float* beta, const float* h0, const void* dout,
                       const float* dhT, float scale, float* dq, float* dk, float* dv, float* dg,
                       float* dbeta, float* dh0, uint8_t* ws, cudaStream_t stream);

// Fused pipeline.  The schedule kernel, given fused_grid > 0, also picks how many of
// the fused kernel's fused_grid CTAs run state chains (production_ratio: the time to
// produce one item's factors over the time of one chain step), lays out the
// production order and clears the ready flags; the fused kernel produces factors on
// the other CTAs while the chain CTAs consume them as they are published.
cudaError_t launch_schedule_fused(const Dims& d, const int32_t* cu_seqlens, uint8_t* ws,
                                  int fused_grid, float production_ratio, cudaStream_t stream);
cudaError_t launch_fused(const Dims& d, bool qkv_bf16, bool g_bf16, const void* q, const void* k,
                         const void* v, const void* g, const float* beta, const float* h0,
                         float scale, void* o, float* hT, uint8_t* ws, cudaStream_t stream);
// Grid and item-time ratio the fused pipeline uses for these sizes (grid 0: the
// fused pipeline does not apply).
int fused_grid(const Dims& d);
float fused_ratio(const Dims& d, bool qkv_bf16);

}  // namespace kda

// Backward pass of the KDA forward: the gradients of sum(o * do) + sum(h_T * dh_T)
// with respect to q, k, v, g, beta and h0 ("Autoresearch on Kimi Delta Attention",
// sections THE MECHANISM and OPTIMIZATION TRACE: the training-side workload carries
// the state's gradient backwards through the chunks).
//
// The value columns of the state never mix in the recurrence (S[:, n] evolves from
// kh, alpha, beta and v[n] alone), and neither do those of its gradient, so the
// work item is one (sequence, head, tile of NVT = 32 or 64 columns; 64 once 32-column
// items would fill the SMs more than twice, so that each token's barriers are shared
// by more work): a persistent grid takes items in steps of its size.  4 * dk threads
// per CTA: thread (c, qd) holds row c of the tile's fp32 state S and of its gradient
// dS, columns qd, qd + 4, ... of the tile
// (interleaved, so that the four threads of a row read consecutive words of a
// shared vector).  Per item:
//   1. forward over the chain, the tile's state at the start of every 64-token
//      chunk saved (a checkpoint in the workspace);
//   2. chunks in reverse: the chunk's states S_{t-1} recomputed from its checkpoint
//      into the CTA's scratch (and r_t = v_t - P_t^T kh_t kept in shared memory),
//      then tokens in reverse, each step the derivative of
//        P = Diag(alpha_t) S_{t-1},  r = v_t - P^T kh,  S_t = P + beta_t kh r^T,
//        o_t = scale S_t^T qh:
//        dS += scale qh do^T;  dqh = scale S_t do;  dbeta = kh . (dS r);
//        dkh = beta dS r - P dr;  dr = beta dS^T kh = dv_t;  dP = dS - kh dr^T;
//        dalpha = rowsum(dP * S_{t-1});  dg = dalpha * alpha;  dS <- Diag(alpha) dP;
//      the sums over value columns (dqh, dkh, dalpha, dbeta) are the tile's share,
//      added into the zeroed outputs (so the last bits of dq, dk, dg and dbeta may
//      differ between runs: the tiles' shares arrive in any order);
//   3. dh0 = dS (the tile's columns).
// A last kernel turns dkh and dqh into dk and dq through the L2 normalisations'
// derivatives, dk = (dkh - kh (kh . dkh)) / |k|_eps.  All arithmetic is fp32 on the
// CUDA cores; a sum over the state's rows is a warp butterfly and one pass through
// shared memory, a sum over a row a shuffle among the row's four threads.
#include <cuda_bf16.h>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr float kEps = 1e-6f;  // the L2-normalisation epsilon of the forward

__device__ __forceinline__ float ld_in(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float ld_in(const float* p) { return *p; }

// Vectors over a tile's columns are kept permuted and padded: column n at
// vidx(n) = (n % 4) (NC + 4) + n / 4 (NC = NVT / 4), so that the NC columns of
// thread qd (n = 4 i + qd) are contiguous and the four threads of a row read them by
// 16-byte loads in distinct banks.
template <int NVT>
__host__ __device__ constexpr int vpad() { return 4 * (NVT / 4 + 4); }
template <int NVT>
__device__ __forceinline__ int vidx(int n) { return (n & 3) * (NVT / 4 + 4) + (n >> 2); }

// Shared memory of one CTA: the current chunk's per-token vectors and the
// reduction scratch.
template <int DK, int NVT>
struct __align__(16) BwdSmem {
    float kh[kChunk][DK], qh[kChunk][DK], al[kChunk][DK];
    float v[kChunk][vpad<NVT>()], dout[kChunk][vpad<NVT>()], r[kChunk][vpad<NVT>()];
    float red[DK / 8][NVT];  // per-warp partial column sums (natural order)
    float vec[vpad<NVT>()];  // a finished column sum
    float bpart[kChunk][DK / 8];
    float beta[kChunk];
};

// Value columns per work item for these sizes (on this device).
int bwd_nvt(const Dims& d) {
    const long long items32 = (long long)d.N * d.H * (d.dv / 32);
    return d.dv >= 64 && items32 > 2LL * num_sms() ? 64 : 32;
}

// Workspace: the forward's schedule (header, sequence table, chunk table), then the
// checkpoints (per (chunk, head): the state at the chunk's start) and each CTA's
// scratch (the tile's states S_{t-1} of one chunk).
struct BwdLayout {
    size_t ckpt, scratch, total;
    __host__ __device__ BwdLayout(const Dims& d, int grid, int nvt) {
        const WsLayout W(d);
        ckpt = align256(W.plist);
        scratch = ckpt + size_t(W.cmax) * d.H * d.dk * d.dv * 4;
        total = scratch + size_t(grid) * kChunk * d.dk * nvt * 4;
    }
};

template <int DK, int DV, int NVT, typename TIn>
__global__ void __launch_bounds__(DK * 4, 1)
    bwd_kernel(Dims d, const int32_t* __restrict__ cu, const TIn* __restrict__ q, const TIn* __restrict__ k,
               const TIn* __restrict__ v, const float* __restrict__ g, const float* __restrict__ beta,
               const float* __restrict__ h0, const TIn* __restrict__ dout, const float* __restrict__ dhT,
               float scale, float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
               float* __restrict__ dg, float* __restrict__ dbeta, float* __restrict__ dh0,
               uint8_t* __restrict__ ws) {
    constexpr int NT = DK * 4, NC = NVT / 4, NW = NT / 32, NTILE = DV / NVT;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    BwdSmem<DK, NVT>& sm = *reinterpret_cast<BwdSmem<DK, NVT>*>(smem_raw);
    const WsLayout W(d);
    const BwdLayout L(d, (int)gridDim.x, NVT);
    const Header* hdr = reinterpret_cast<const Header*>(ws + W.header);
    if (hdr->error) return;  // malformed cu_seqlens (reported in the error word)
    const int32_t* seq_first = reinterpret_cast<const int32_t*>(ws + W.seq_first);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid >> 2, qd = tid & 3, n0 = qd * NC;  // n0: this thread's slots in a saved state
    const int H = d.H;
    const size_t st = size_t(DK) * DV;
    float* ckpt_all = reinterpret_cast<float*>(ws + L.ckpt);
    float* scr = reinterpret_cast<float*>(ws + L.scratch) + size_t(blockIdx.x) * kChunk * DK * NVT;

    // Sum over the state's rows of f x[i] (column 4 i + qd of the tile), for every
    // column: the result lands in sm.vec.  Inside a warp (8 rows) a butterfly: at each
    // of three shuffle distances a thread keeps half of its remaining slots and hands
    // the other half to its partner, ending with one slot summed over the warp's rows;
    // then one pass through shared memory over the warps.  Two barriers; callers read
    // sm.vec after it returns.
    const bool b2 = (lane >> 4) & 1, b1 = (lane >> 3) & 1, b0 = (lane >> 2) & 1;
    const int slot0 = (b2 ? NC / 2 : 0) + (b1 ? NC / 4 : 0) + (b0 ? NC / 8 : 0);
    auto col_sum = [&](const float (&x)[NC], float f) {
        float y[NC / 2], z[NC / 4], w[NC / 8];
#pragma unroll
        for (int i = 0; i < NC / 2; ++i) {
            const float lo = f * x[i], hi = f * x[i + NC / 2];
            y[i] = (b2 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b2 ? lo : hi, 16);
        }
#pragma unroll
        for (int i = 0; i < NC / 4; ++i) {
            const float send = b1 ? y[i] : y[i + NC / 4];
            z[i] = (b1 ? y[i + NC / 4] : y[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int i = 0; i < NC / 8; ++i) {
            const float send = b0 ? z[i] : z[i + NC / 8];
            w[i] = (b0 ? z[i + NC / 8] : z[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
        }
#pragma unroll
        for (int i = 0; i < NC / 8; ++i) sm.red[warp][4 * (slot0 + i) + qd] = w[i];
        __syncthreads();
        if (tid < NVT) {
            float s = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) s += sm.red[w2][tid];
            sm.vec[vidx<NVT>(tid)] = s;
        }
        __syncthreads();
    };
    // This thread's columns of a permuted vector: four of them (i = 4 j .. 4 j + 3)
    // by one 16-byte load.
    auto vq = [&](const float* vecp, int j) {
        return reinterpret_cast<const float4*>(vecp + qd * (NC + 4))[j];
    };
    auto row_sum = [&](float x) {  // over the row's four threads
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        return x;
    };
    // One step of the forward on this thread's columns: S <- P + beta kh (v - P^T kh).
    auto fwd_step = [&](float (&S)[NC], int tt, bool keep_r) {
        const float a = sm.al[tt][c], kc = sm.kh[tt][c], be = sm.beta[tt];
        col_sum(S, a * kc);  // P^T kh, P = Diag(alpha) S
        if (keep_r && tid < NVT) sm.r[tt][vidx<NVT>(tid)] = sm.v[tt][vidx<NVT>(tid)] - sm.vec[vidx<NVT>(tid)];
#pragma unroll
        for (int j = 0; j < NC / 4; ++j) {
            const float4 vv = vq(sm.v[tt], j), pk = vq(sm.vec, j);
            S[4 * j] = fmaf(be * kc, vv.x - pk.x, a * S[4 * j]);
            S[4 * j + 1] = fmaf(be * kc, vv.y - pk.y, a * S[4 * j + 1]);
            S[4 * j + 2] = fmaf(be * kc, vv.z - pk.z, a * S[4 * j + 2]);
            S[4 * j + 3] = fmaf(be * kc, vv.w - pk.w, a * S[4 * j + 3]);
        }
    };
    // The chunk's per-token vectors into shared memory (warp w takes tokens w, w + NW,
    // ...): kh (normalised), alpha, the tile's v and beta; with `full` also qh and the
    // tile's do.
    auto load_chunk = [&](int b, int t0, int rows, int h, int col0, bool full) {
        for (int tt = warp; tt < rows; tt += NW) {
            const size_t row = (size_t)b * d.T + t0 + tt;
            const size_t ok = (row * H + h) * DK, ov = (row * H + h) * DV + col0;
            float ss = 0.f, sq = 0.f, kk[DK / 32], qq[DK / 32];
#pragma unroll
            for (int i = 0; i < DK / 32; ++i) {
                const int ch = lane + 32 * i;
                kk[i] = ld_in(k + ok + ch);
                ss += kk[i] * kk[i];
                qq[i] = full ? ld_in(q + ok + ch) : 0.f;
                sq += qq[i] * qq[i];
                sm.al[tt][ch] = expf(g[ok + ch]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ss += __shfl_xor_sync(0xffffffffu, ss, o);
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
            }
            const float rk = 1.f / sqrtf(ss + kEps), rq = 1.f / sqrtf(sq + kEps);
#pragma unroll
            for (int i = 0; i < DK / 32; ++i) {
                sm.kh[tt][lane + 32 * i] = kk[i] * rk;
                if (full) sm.qh[tt][lane + 32 * i] = qq[i] * rq;
            }
#pragma unroll
            for (int i = 0; i < NVT / 32; ++i) {
                sm.v[tt][vidx<NVT>(lane + 32 * i)] = ld_in(v + ov + lane + 32 * i);
                if (full) sm.dout[tt][vidx<NVT>(lane + 32 * i)] = ld_in(dout + ov + lane + 32 * i);
            }
            if (lane == 0) sm.beta[tt] = beta[row * H + h];
        }
        __syncthreads();
    };

    const int items = d.N * H * NTILE;
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int chain = item / NTILE, tile = item - chain * NTILE;
        const int s = chain / H, h = chain - s * H, col0 = tile * NVT;
        int b, bos, eos;
        if (d.varlen) {
            b = 0;
            bos = cu[s];
            eos = cu[s + 1];
        } else {
            b = s;
            bos = 0;
            eos = d.T;
        }
        const int len = eos - bos, nch = (len + kChunk - 1) / kChunk;
        float* ck = ckpt_all + ((size_t)seq_first[s] * H + h) * st + (size_t)c * DV + col0 + n0;  // + j H st
        const size_t rbase = ((size_t)s * H + h) * st + (size_t)c * DV + col0 + qd;  // + 4 i: column 4 i + qd
        float S[NC], dS[NC];
#pragma unroll
        for (int i = 0; i < NC; ++i) S[i] = h0 ? h0[rbase + 4 * i] : 0.f;
        // -------- 1. forward, checkpoints at chunk starts
        for (int j = 0; j < nch; ++j) {
            float* cj = ck + (size_t)j * H * st;
#pragma unroll
            for (int i = 0; i < NC; i += 4) *reinterpret_cast<float4*>(cj + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
            const int t0 = bos + j * kChunk, rows = eos - t0 < kChunk ? eos - t0 : kChunk;
            __syncthreads();  // the previous chunk's vectors are no longer read
            load_chunk(b, t0, rows, h, col0, false);
            for (int tt = 0; tt < rows; ++tt) fwd_step(S, tt, false);
        }
        // -------- 2. chunks in reverse
#pragma unroll
        for (int i = 0; i < NC; ++i) dS[i] = dhT ? dhT[rbase + 4 * i] : 0.f;
        for (int j = nch - 1; j >= 0; --j) {
            const int t0 = bos + j * kChunk, rows = eos - t0 < kChunk ? eos - t0 : kChunk;
            const float* cj = ck + (size_t)j * H * st;
#pragma unroll
            for (int i = 0; i < NC; i += 4) {
                const float4 w4 = *reinterpret_cast<const float4*>(cj + i);
                S[i] = w4.x; S[i + 1] = w4.y; S[i + 2] = w4.z; S[i + 3] = w4.w;
            }
            __syncthreads();  // the previous chunk's vectors are no longer read
            load_chunk(b, t0, rows, h, col0, true);
            // the chunk's states S_{t-1} into the scratch, and r_t
            for (int tt = 0; tt < rows; ++tt) {
                float* sp = scr + (size_t)tt * DK * NVT + (size_t)c * NVT + n0;
#pragma unroll
                for (int i = 0; i < NC; i += 4) *reinterpret_cast<float4*>(sp + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
                fwd_step(S, tt, true);
            }
            __syncthreads();  // sm.r complete
            // tokens in reverse; each step's S_{t-1} loads during the step before
            float nxt[NC];
            auto load_prev = [&](int tt) {
                const float* sp = scr + (size_t)tt * DK * NVT + (size_t)c * NVT + n0;
#pragma unroll
                for (int i = 0; i < NC; i += 4) {
                    const float4 w4 = *reinterpret_cast<const float4*>(sp + i);
                    nxt[i] = w4.x; nxt[i + 1] = w4.y; nxt[i + 2] = w4.z; nxt[i + 3] = w4.w;
                }
            };
            if (rows > 0) load_prev(rows - 1);
            for (int tt = rows - 1; tt >= 0; --tt) {
                const size_t row = (size_t)b * d.T + t0 + tt;
                float Sp[NC];
#pragma unroll
                for (int i = 0; i < NC; ++i) Sp[i] = nxt[i];
                if (tt > 0) load_prev(tt - 1);
                const float a = sm.al[tt][c], kc = sm.kh[tt][c], qc = sm.qh[tt][c], be = sm.beta[tt];
                float dqh = 0.f, u = 0.f;
#pragma unroll
                for (int j = 0; j < NC / 4; ++j) {
                    const float4 r4 = vq(sm.r[tt], j), d4 = vq(sm.dout[tt], j);
                    const float rr[4] = {r4.x, r4.y, r4.z, r4.w}, dd[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 4 * j + e;
                        const float St = fmaf(be * kc, rr[e], a * Sp[i]);
                        dS[i] = fmaf(scale * qc, dd[e], dS[i]);
                        dqh = fmaf(St, dd[e], dqh);
                        u = fmaf(dS[i], rr[e], u);
                    }
                }
                col_sum(dS, kc);  // sm.vec = dS^T kh
                float dkh2 = 0.f, dal = 0.f;
#pragma unroll
                for (int j = 0; j < NC / 4; ++j) {
                    const float4 c4 = vq(sm.vec, j);
                    const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 4 * j + e;
                        const float dr = be * cs[e];
                        const float P = a * Sp[i];
                        const float dP = fmaf(-kc, dr, dS[i]);
                        dkh2 = fmaf(-P, dr, dkh2);
                        dal = fmaf(dP, Sp[i], dal);
                        dS[i] = a * dP;
                    }
                }
                dqh = row_sum(dqh);
                u = row_sum(u);
                dkh2 = row_sum(dkh2);
                dal = row_sum(dal);
                if (qd == 0) {  // this tile's shares of the sums over value columns
                    const size_t ok = (row * H + h) * DK + c;
                    atomicAdd(dk + ok, fmaf(be, u, dkh2));  // dkh; normalised by the last kernel
                    atomicAdd(dq + ok, scale * dqh);         // dqh; the same
                    atomicAdd(dg + ok, dal * a);
                }
                if (tid < NVT) dv[(row * H + h) * DV + col0 + tid] = be * sm.vec[vidx<NVT>(tid)];
                float bp = qd == 0 ? kc * u : 0.f;  // this warp's rows' share of dbeta
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) bp += __shfl_xor_sync(0xffffffffu, bp, o);
                if (lane == 0) sm.bpart[tt][warp] = bp;
            }
            __syncthreads();  // the dbeta parts of the chunk are written
            for (int tt = tid; tt < rows; tt += NT) {
                float sb = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < NW; ++w2) sb += sm.bpart[tt][w2];
                atomicAdd(dbeta + ((size_t)b * d.T + t0 + tt) * H + h, sb);
            }
        }
        // -------- 3. the gradient of the initial state (this tile's columns)
        if (dh0) {
#pragma unroll
            for (int i = 0; i < NC; ++i) dh0[rbase + 4 * i] = dS[i];
        }
        __syncthreads();  // the chunk vectors and scratch are free for the next item
    }
}

// dk = (dkh - kh (kh . dkh)) / |k|_eps and dq likewise, in place: one warp per
// (token, head) row.
template <int DK, typename TIn>
__global__ void __launch_bounds__(256) bwd_finish_kernel(Dims d, const TIn* __restrict__ q,
                                                         const TIn* __restrict__ k, float* __restrict__ dq,
                                                         float* __restrict__ dk, const uint8_t* __restrict__ ws) {
    const Header* hdr = reinterpret_cast<const Header*>(ws + WsLayout(d).header);
    if (hdr->error) return;
    const long long rowsH = (long long)d.B * d.T * d.H;
    const long long rw = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (rw >= rowsH) return;
    const size_t o = (size_t)rw * DK;
    float kk[DK / 32], qq[DK / 32], xk[DK / 32], xq[DK / 32], ss = 0.f, sq = 0.f;
#pragma unroll
    for (int i = 0; i < DK / 32; ++i) {
        const int ch = lane + 32 * i;
        kk[i] = ld_in(k + o + ch);
        qq[i] = ld_in(q + o + ch);
        xk[i] = dk[o + ch];
        xq[i] = dq[o + ch];
        ss += kk[i] * kk[i];
        sq += qq[i] * qq[i];
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, s);
        sq += __shfl_xor_sync(0xffffffffu, sq, s);
    }
    const float rk = 1.f / sqrtf(ss + kEps), rq = 1.f / sqrtf(sq + kEps);
    float dotk = 0.f, dotq = 0.f;
#pragma unroll
    for (int i = 0; i < DK / 32; ++i) {
        dotk = fmaf(kk[i] * rk, xk[i], dotk);
        dotq = fmaf(qq[i] * rq, xq[i], dotq);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
        dotk += __shfl_xor_sync(0xffffffffu, dotk, s);
        dotq += __shfl_xor_sync(0xffffffffu, dotq, s);
    }
#pragma unroll
    for (int i = 0; i < DK / 32; ++i) {
        const int ch = lane + 32 * i;
        dk[o + ch] = rk * fmaf(-kk[i] * rk, dotk, xk[i]);
        dq[o + ch] = rq * fmaf(-qq[i] * rq, dotq, xq[i]);
    }
}

int bwd_grid(const Dims& d) {
    const long long items = (long long)d.N * d.H * (d.dv / bwd_nvt(d));
    const int sms = num_sms();
    return (int)(items < sms ? (items > 0 ? items : 1) : sms);
}

template <int DK, int DV, int NVT, typename TIn>
cudaError_t launch_bwd_t(const Dims& d, const int32_t* cu, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* h0, const void* dout,
                         const float* dhT, float scale, float* dq, float* dk, float* dv, float* dg,
                         float* dbeta, float* dh0, uint8_t* ws, cudaStream_t stream) {
    static_assert(DV % NVT == 0 && NVT % 32 == 0, "value tiles of whole warps of columns");
    auto kern = bwd_kernel<DK, DV, NVT, TIn>;
    const size_t smem = sizeof(BwdSmem<DK, NVT>);
    static_assert(sizeof(BwdSmem<DK, NVT>) <= 227 * 1024, "backward shared memory");
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const size_t tok = (size_t)d.B * d.T * d.H;
    if (tok > 0) {  // the sums over value tiles are added into these
        if ((e = cudaMemsetAsync(dq, 0, tok * DK * 4, stream)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(dk, 0, tok * DK * 4, stream)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(dg, 0, tok * DK * 4, stream)) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(dbeta, 0, tok * 4, stream)) != cudaSuccess) return e;
    }
    if ((long long)d.N * d.H == 0) return cudaSuccess;
    kern<<<bwd_grid(d), DK * 4, smem, stream>>>(d, cu, static_cast<const TIn*>(q), static_cast<const TIn*>(k),
                                                 static_cast<const TIn*>(v), g, beta, h0,
                                                 static_cast<const TIn*>(dout), dhT, scale, dq, dk, dv, dg,
                                                 dbeta, dh0, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (tok == 0) return cudaSuccess;
    bwd_finish_kernel<DK, TIn><<<(unsigned)((tok + 7) / 8), 256, 0, stream>>>(
        d, static_cast<const TIn*>(q), static_cast<const TIn*>(k), dq, dk, ws);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(const Dims& d) { return BwdLayout(d, bwd_grid(d), bwd_nvt(d)).total; }

cudaError_t launch_bwd(const Dims& d, bool qkv_bf16, const int32_t* cu, const void* q, const void* k,
                       const void* v, const float* g, const float* beta, const float* h0, const void* dout,
                       const float* dhT, float scale, float* dq, float* dk, float* dv, float* dg,
                       float* dbeta, float* dh0, uint8_t* ws, cudaStream_t stream) {
    using bf = __nv_bfloat16;
#define KDA_BWD_CASE(DK_, DV_, NVT_)                                                                  \
    if (d.dk == DK_ && d.dv == DV_ && bwd_nvt(d) == NVT_)                                              \
        return qkv_bf16 ? launch_bwd_t<DK_, DV_, NVT_, bf>(d, cu, q, k, v, g, beta, h0, dout, dhT, scale,   \
                                                            dq, dk, dv, dg, dbeta, dh0, ws, stream)    \
                        : launch_bwd_t<DK_, DV_, NVT_, float>(d, cu, q, k, v, g, beta, h0, dout, dhT,      \
                                                               scale, dq, dk, dv, dg, dbeta, dh0, ws, stream);
    KDA_BWD_CASE(64, 64, 32)
    KDA_BWD_CASE(64, 64, 64)
    KDA_BWD_CASE(64, 128, 32)
    KDA_BWD_CASE(64, 128, 64)
    KDA_BWD_CASE(128, 64, 32)
    KDA_BWD_CASE(128, 64, 64)
    KDA_BWD_CASE(128, 128, 32)
    KDA_BWD_CASE(128, 128, 64)
#undef KDA_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda

// Backward pass of the KDA forward: the gradients of sum(o * do) + sum(h_T * dh_T)
// with respect to q, k, v, g, beta and h0 ("Autoresearch on Kimi Delta Attention",
// sections THE MECHANISM and OPTIMIZATION TRACE: the training-side workload carries
// the state's gradient backwards through the chunks).
//
// One CTA per (sequence, head) chain at a time (persistent, chains in steps of the
// grid), 4 * dk threads: thread (c, qd) holds row c of the fp32 state S (dk x dv) and
// of its gradient dS, value columns qd, qd + 4, qd + 8, ... (interleaved, so that the
// four threads of a row read consecutive words of a shared vector).  Per chain:
//   1. forward over the chain, the state at the start of every 64-token chunk saved
//      (a checkpoint in the workspace);
//   2. chunks in reverse: the chunk's states S_{t-1} recomputed from its checkpoint
//      into the CTA's scratch (and r_t = v_t - P_t^T kh_t kept in shared memory),
//      then tokens in reverse, each step the derivative of
//        P = Diag(alpha_t) S_{t-1},  r = v_t - P^T kh,  S_t = P + beta_t kh r^T,
//        o_t = scale S_t^T qh:
//        dS += scale qh do^T;  dqh = scale S_t do;  dbeta = kh . (dS r);
//        dkh = beta dS r - P dr;  dr = beta dS^T kh = dv_t;  dP = dS - kh dr^T;
//        dalpha = rowsum(dP * S_{t-1});  dg = dalpha * alpha;  dS <- Diag(alpha) dP;
//      and the L2 normalisations' derivatives dk = (dkh - kh (kh . dkh)) / |k|_eps
//      (the same for q) once the chunk is done;
//   3. dh0 = dS.
// All arithmetic is fp32 on the CUDA cores; every sum over the state's rows is a
// warp shuffle tree and one pass through shared memory, every sum over its columns
// a shuffle among the row's four threads.
#include <cuda_bf16.h>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {

namespace {

constexpr float kEps = 1e-6f;  // the L2-normalisation epsilon of the forward

__device__ __forceinline__ float ld_in(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float ld_in(const float* p) { return *p; }

// Shared memory of one CTA: the current chunk's per-token vectors and the
// reduction scratch.  Vectors over the value columns are kept permuted and padded:
// column n at vidx(n) = (n % 4) (dv/4 + 4) + n / 4, so that the dv/4 columns of
// thread qd (n = 4 i + qd) are contiguous and the four threads of a row read them by
// 16-byte loads in distinct banks.
template <int DV>
__host__ __device__ constexpr int vpad() { return 4 * (DV / 4 + 4); }
template <int DV>
__device__ __forceinline__ int vidx(int n) { return (n & 3) * (DV / 4 + 4) + (n >> 2); }

template <int DK, int DV>
struct __align__(16) BwdSmem {
    float kh[kChunk][DK], qh[kChunk][DK], al[kChunk][DK];
    float v[kChunk][vpad<DV>()], dout[kChunk][vpad<DV>()], r[kChunk][vpad<DV>()];
    float red[DK / 8][DV];  // per-warp partial column sums (natural order)
    float vec[vpad<DV>()];  // a finished column sum
    float bpart[kChunk][DK / 8];
    float rk[kChunk], rq[kChunk], beta[kChunk];
};

// Workspace: the forward's schedule (header, sequence table, chunk table), then the
// checkpoints (per (chunk, head): the state at the chunk's start) and each CTA's
// scratch (the states S_{t-1} of one chunk).
struct BwdLayout {
    size_t ckpt, scratch, total;
    __host__ __device__ BwdLayout(const Dims& d, int grid) {
        const WsLayout W(d);
        const size_t st = size_t(d.dk) * d.dv * 4;
        ckpt = align256(W.plist);
        scratch = ckpt + size_t(W.cmax) * d.H * st;
        total = scratch + size_t(grid) * kChunk * st;
    }
};

template <int DK, int DV, typename TIn>
__global__ void __launch_bounds__(DK * 4, 1)
    bwd_kernel(Dims d, const int32_t* __restrict__ cu, const TIn* __restrict__ q, const TIn* __restrict__ k,
               const TIn* __restrict__ v, const float* __restrict__ g, const float* __restrict__ beta,
               const float* __restrict__ h0, const TIn* __restrict__ dout, const float* __restrict__ dhT,
               float scale, float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
               float* __restrict__ dg, float* __restrict__ dbeta, float* __restrict__ dh0,
               uint8_t* __restrict__ ws) {
    constexpr int NT = DK * 4, NC = DV / 4, NW = NT / 32;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    BwdSmem<DK, DV>& sm = *reinterpret_cast<BwdSmem<DK, DV>*>(smem_raw);
    const WsLayout W(d);
    const BwdLayout L(d, (int)gridDim.x);
    const Header* hdr = reinterpret_cast<const Header*>(ws + W.header);
    if (hdr->error) return;  // malformed cu_seqlens (reported in the error word)
    const int32_t* seq_first = reinterpret_cast<const int32_t*>(ws + W.seq_first);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid >> 2, qd = tid & 3, n0 = qd * NC;  // n0: this thread's slots in a saved state
    const int H = d.H;
    const size_t st = size_t(DK) * DV;
    float* ckpt_all = reinterpret_cast<float*>(ws + L.ckpt);
    float* scr = reinterpret_cast<float*>(ws + L.scratch) + size_t(blockIdx.x) * kChunk * st;

    // Sum over the state's rows of f x[i] (column 4 i + qd), for every column: the result
    // lands in sm.vec.  Inside a warp (8 rows) a butterfly: at each of three shuffle
    // distances a thread keeps half of its remaining slots and hands the other half to
    // its partner, ending with NC / 8 slots summed over the warp's rows (NC - 4
    // shuffles in all instead of 3 NC); then one pass through shared memory over the
    // warps.  Two barriers; callers read sm.vec after it returns.
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
        if (tid < DV) {
            float s = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) s += sm.red[w2][tid];
            sm.vec[vidx<DV>(tid)] = s;
        }
        __syncthreads();
    };
    // This thread's NC columns (4 i + qd) of a permuted vector: four of them (i = 4 j
    // .. 4 j + 3) by one 16-byte load.
    auto vq = [&](const float* vecp, int j) {
        return reinterpret_cast<const float4*>(vecp + qd * (NC + 4))[j];
    };
    auto row_sum = [&](float x) {  // over the row's four threads
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        return x;
    };
    const int R = d.N * H;
    for (int chain = blockIdx.x; chain < R; chain += gridDim.x) {
        const int s = chain / H, h = chain - s * H;
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
        float* ck = ckpt_all + ((size_t)seq_first[s] * H + h) * st;  // chunk j at + j * H * st
        const size_t rbase = ((size_t)s * H + h) * st + (size_t)c * DV + qd;  // + 4 i: column 4 i + qd
        float S[NC], dS[NC];
#pragma unroll
        for (int i = 0; i < NC; ++i) S[i] = h0 ? h0[rbase + 4 * i] : 0.f;
        // -------- 1. forward, checkpoints at chunk starts
        for (int j = 0; j < nch; ++j) {
            float* cj = ck + (size_t)j * H * st + (size_t)c * DV + n0;
#pragma unroll
            for (int i = 0; i < NC; i += 4) *reinterpret_cast<float4*>(cj + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
            const int t0 = bos + j * kChunk, rows = eos - t0 < kChunk ? eos - t0 : kChunk;
            __syncthreads();  // the previous chunk's vectors are no longer read
            // k (normalised), alpha, v and beta of the chunk's tokens: warp w takes
            // tokens w, w + NW, ...
            for (int tt = warp; tt < rows; tt += NW) {
                const size_t row = (size_t)b * d.T + t0 + tt;
                float ss = 0.f, kk[DK / 32];
#pragma unroll
                for (int i = 0; i < DK / 32; ++i) {
                    const int ch = lane + 32 * i;
                    kk[i] = ld_in(k + (row * H + h) * DK + ch);
                    ss += kk[i] * kk[i];
                    sm.al[tt][ch] = expf(g[(row * H + h) * DK + ch]);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float rk = 1.f / sqrtf(ss + kEps);
#pragma unroll
                for (int i = 0; i < DK / 32; ++i) sm.kh[tt][lane + 32 * i] = kk[i] * rk;
#pragma unroll
                for (int i = 0; i < DV / 32; ++i)
                    sm.v[tt][vidx<DV>(lane + 32 * i)] = ld_in(v + (row * H + h) * DV + lane + 32 * i);
                if (lane == 0) sm.beta[tt] = beta[row * H + h];
            }
            __syncthreads();
            for (int tt = 0; tt < rows; ++tt) {
                const float a = sm.al[tt][c], kc = sm.kh[tt][c], be = sm.beta[tt];
                col_sum(S, a * kc);  // P^T kh, P = Diag(alpha) S
#pragma unroll
                for (int j = 0; j < NC / 4; ++j) {
                    const float4 vv = vq(sm.v[tt], j), pk = vq(sm.vec, j);
                    S[4 * j] = fmaf(be * kc, vv.x - pk.x, a * S[4 * j]);
                    S[4 * j + 1] = fmaf(be * kc, vv.y - pk.y, a * S[4 * j + 1]);
                    S[4 * j + 2] = fmaf(be * kc, vv.z - pk.z, a * S[4 * j + 2]);
                    S[4 * j + 3] = fmaf(be * kc, vv.w - pk.w, a * S[4 * j + 3]);
                }
            }
        }
        // -------- 2. chunks in reverse
#pragma unroll
        for (int i = 0; i < NC; ++i) dS[i] = dhT ? dhT[rbase + 4 * i] : 0.f;
        for (int j = nch - 1; j >= 0; --j) {
            const int t0 = bos + j * kChunk, rows = eos - t0 < kChunk ? eos - t0 : kChunk;
            const float* cj = ck + (size_t)j * H * st + (size_t)c * DV + n0;
#pragma unroll
            for (int i = 0; i < NC; i += 4) {
                const float4 w4 = *reinterpret_cast<const float4*>(cj + i);
                S[i] = w4.x; S[i + 1] = w4.y; S[i + 2] = w4.z; S[i + 3] = w4.w;
            }
            __syncthreads();  // the previous chunk's vectors are no longer read
            for (int tt = warp; tt < rows; tt += NW) {  // as above, with q (normalised) and do
                const size_t row = (size_t)b * d.T + t0 + tt;
                const size_t ok = (row * H + h) * DK, ov = (row * H + h) * DV;
                float ss = 0.f, sq = 0.f, kk[DK / 32], qq[DK / 32];
#pragma unroll
                for (int i = 0; i < DK / 32; ++i) {
                    const int ch = lane + 32 * i;
                    kk[i] = ld_in(k + ok + ch);
                    qq[i] = ld_in(q + ok + ch);
                    ss += kk[i] * kk[i];
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
                    sm.qh[tt][lane + 32 * i] = qq[i] * rq;
                }
#pragma unroll
                for (int i = 0; i < DV / 32; ++i) {
                    sm.v[tt][vidx<DV>(lane + 32 * i)] = ld_in(v + ov + lane + 32 * i);
                    sm.dout[tt][vidx<DV>(lane + 32 * i)] = ld_in(dout + ov + lane + 32 * i);
                }
                if (lane == 0) {
                    sm.rk[tt] = rk;
                    sm.rq[tt] = rq;
                    sm.beta[tt] = beta[row * H + h];
                }
            }
            __syncthreads();
            // the chunk's states S_{t-1} into the scratch, and r_t
            for (int tt = 0; tt < rows; ++tt) {
                float* sp = scr + (size_t)tt * st + (size_t)c * DV + n0;
#pragma unroll
                for (int i = 0; i < NC; i += 4) *reinterpret_cast<float4*>(sp + i) = make_float4(S[i], S[i + 1], S[i + 2], S[i + 3]);
                const float a = sm.al[tt][c], kc = sm.kh[tt][c], be = sm.beta[tt];
                col_sum(S, a * kc);  // P^T kh, P = Diag(alpha) S
                if (tid < DV) sm.r[tt][vidx<DV>(tid)] = sm.v[tt][vidx<DV>(tid)] - sm.vec[vidx<DV>(tid)];
#pragma unroll
                for (int j = 0; j < NC / 4; ++j) {
                    const float4 vv = vq(sm.v[tt], j), pk = vq(sm.vec, j);
                    S[4 * j] = fmaf(be * kc, vv.x - pk.x, a * S[4 * j]);
                    S[4 * j + 1] = fmaf(be * kc, vv.y - pk.y, a * S[4 * j + 1]);
                    S[4 * j + 2] = fmaf(be * kc, vv.z - pk.z, a * S[4 * j + 2]);
                    S[4 * j + 3] = fmaf(be * kc, vv.w - pk.w, a * S[4 * j + 3]);
                }
            }
            __syncthreads();  // sm.r complete
            // tokens in reverse; each step's S_{t-1} loads during the step before
            float nxt[NC];
            auto load_prev = [&](int tt) {
                const float* sp = scr + (size_t)tt * st + (size_t)c * DV + n0;
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
                if (qd == 0) {
                    const size_t ok = (row * H + h) * DK + c;
                    dk[ok] = fmaf(be, u, dkh2);  // dkh; normalised below
                    dq[ok] = scale * dqh;         // dqh; normalised below
                    dg[ok] = dal * a;
                }
                if (tid < DV) dv[(row * H + h) * DV + tid] = be * sm.vec[vidx<DV>(tid)];
                float bp = qd == 0 ? kc * u : 0.f;  // this warp's rows' share of dbeta
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) bp += __shfl_xor_sync(0xffffffffu, bp, o);
                if (lane == 0) sm.bpart[tt][warp] = bp;
            }
            __syncthreads();  // dkh, dqh and the dbeta parts of the chunk are written
            // dbeta, and the normalisations' derivatives, per token
            for (int tt = warp; tt < rows; tt += NW) {
                const size_t row = (size_t)b * d.T + t0 + tt;
                const size_t ok = (row * H + h) * DK;
                if (lane == 0) {
                    float sb = 0.f;
                    for (int w = 0; w < NW; ++w) sb += sm.bpart[tt][w];
                    dbeta[row * H + h] = sb;
                }
                float xk[DK / 32], xq[DK / 32], dotk = 0.f, dotq = 0.f;
#pragma unroll
                for (int i = 0; i < DK / 32; ++i) {
                    const int ch = lane + 32 * i;
                    xk[i] = dk[ok + ch];
                    xq[i] = dq[ok + ch];
                    dotk = fmaf(sm.kh[tt][ch], xk[i], dotk);
                    dotq = fmaf(sm.qh[tt][ch], xq[i], dotq);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    dotk += __shfl_xor_sync(0xffffffffu, dotk, o);
                    dotq += __shfl_xor_sync(0xffffffffu, dotq, o);
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < DK / 32; ++i) {
                    const int ch = lane + 32 * i;
                    dk[ok + ch] = sm.rk[tt] * fmaf(-sm.kh[tt][ch], dotk, xk[i]);
                    dq[ok + ch] = sm.rq[tt] * fmaf(-sm.qh[tt][ch], dotq, xq[i]);
                }
            }
        }
        // -------- 3. the gradient of the initial state
        if (dh0) {
#pragma unroll
            for (int i = 0; i < NC; ++i) dh0[rbase + 4 * i] = dS[i];
        }
        __syncthreads();  // the chunk vectors and scratch are free for the next chain
    }
}

int bwd_grid(const Dims& d) {
    const long long R = (long long)d.N * d.H;
    const int sms = num_sms();
    return (int)(R < sms ? (R > 0 ? R : 1) : sms);
}

template <int DK, int DV, typename TIn>
cudaError_t launch_bwd_t(const Dims& d, const int32_t* cu, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* h0, const void* dout,
                         const float* dhT, float scale, float* dq, float* dk, float* dv, float* dg,
                         float* dbeta, float* dh0, uint8_t* ws, cudaStream_t stream) {
    auto kern = bwd_kernel<DK, DV, TIn>;
    const size_t smem = sizeof(BwdSmem<DK, DV>);
    static_assert(sizeof(BwdSmem<DK, DV>) <= 227 * 1024, "backward shared memory");
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    if ((long long)d.N * d.H == 0) return cudaSuccess;
    kern<<<bwd_grid(d), DK * 4, smem, stream>>>(d, cu, static_cast<const TIn*>(q), static_cast<const TIn*>(k),
                                                 static_cast<const TIn*>(v), g, beta, h0,
                                                 static_cast<const TIn*>(dout), dhT, scale, dq, dk, dv, dg,
                                                 dbeta, dh0, ws);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_bytes(const Dims& d) { return BwdLayout(d, bwd_grid(d)).total; }

cudaError_t launch_bwd(const Dims& d, bool qkv_bf16, const int32_t* cu, const void* q, const void* k,
                       const void* v, const float* g, const float* beta, const float* h0, const void* dout,
                       const float* dhT, float scale, float* dq, float* dk, float* dv, float* dg,
                       float* dbeta, float* dh0, uint8_t* ws, cudaStream_t stream) {
    using bf = __nv_bfloat16;
#define KDA_BWD_CASE(DK_, DV_)                                                                        \
    if (d.dk == DK_ && d.dv == DV_)                                                                   \
        return qkv_bf16 ? launch_bwd_t<DK_, DV_, bf>(d, cu, q, k, v, g, beta, h0, dout, dhT, scale, dq, dk, \
                                                      dv, dg, dbeta, dh0, ws, stream)                  \
                        : launch_bwd_t<DK_, DV_, float>(d, cu, q, k, v, g, beta, h0, dout, dhT, scale, dq,  \
                                                         dk, dv, dg, dbeta, dh0, ws, stream);
    KDA_BWD_CASE(64, 64)
    KDA_BWD_CASE(64, 128)
    KDA_BWD_CASE(128, 64)
    KDA_BWD_CASE(128, 128)
#undef KDA_BWD_CASE
    return cudaErrorInvalidValue;
}

}  // namespace kda

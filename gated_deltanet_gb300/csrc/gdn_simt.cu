// fp32 CUDA-core engine of the chunked gated delta rule, plus the chunk-
// parallel split helpers (gate statistics for the warmup split, and the
// serial S* / M combine of the exact split).
//
// One CTA owns one (sequence, value head, 32-column value tile, segment) and
// walks its chunks serially with the [K x 32] fp32 state slice in shared
// memory.  Per chunk (C = 64 rows; all arithmetic fp32, gates in base 2):
//
//   1. gate cumsum          G_i = sum_{s<=i} g_s / ln 2   (per channel for gk)
//   2. gated K K^T, Q K^T    L_ij = beta_i sum_d k_id k_jd 2^(G_id-G_jd)  (j < i)
//                            P_ij =        sum_d q_id k_jd 2^(G_id-G_jd)  (j <= i)
//   3. inverse               X = (I + L)^-1 by column-parallel forward substitution
//   4. residual              R = diag(beta) (V - (K * 2^G) S)
//   5. WY / new values       V' = X R                         (= U - W S)
//   6. output                O = scale [ (Q * 2^G) S + P V' ]  (state before the chunk)
//   7. state                 S <- Diag(2^G_C) S + (K * 2^(G_C - G))^T V'
//
// Steps 4-5 are the FLA four-step form (FlashQLA blog, "Key problems", the
// W/U and V' lines) with U - W S factored as A diag(beta) (V - diag(gam) K S)
// ("A balanced solution", step 3); the per-channel gate follows the "KDA
// source walkthrough" (Akk/Aqk with exp(g_i - g_j) per channel, kg, qg, and
// the per-row state decay).  Rows past the end of a sequence are loaded as
// k = q = v = 0, g = 0, beta = 0, which makes them inert, so the decay to the
// chunk end uses the last valid token (same walkthrough, last_idx).
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {
using ptx::ex2;  // the MUFU base-2 exponential (a handful of ulp; inputs are log-gate sums)

constexpr int kBV = 32;
constexpr int kThreads = 256;
constexpr int kLd = 65;  // padded row length of the 64 x 64 tiles

__device__ __forceinline__ int rows_in_chunk(int64_t len, int c)
{
    const int64_t r = len - (int64_t)c * kChunk;
    return r < kChunk ? (int)r : kChunk;
}
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float *p, float x) { *p = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

template <int K, bool CHANNEL>
struct SimtLayout {
    static constexpr int KP = K + 1;
    static constexpr int oS = 0;                          // [K][kBV]   state slice
    static constexpr int oK = oS + K * kBV;               // [64][KP]   k, then k * 2^G (channel)
    static constexpr int oQ = oK + 64 * KP;               // [64][KP]   q, then q * 2^G (channel)
    static constexpr int oG = oQ + 64 * KP;               // [64][KP] or [64]: G, then k * 2^(G_C - G)
    static constexpr int oGC = oG + (CHANNEL ? 64 * KP : 64);  // [K] or [1]: G_C
    static constexpr int oV = oGC + (CHANNEL ? K : 4);    // [64][kBV]  v, then beta * R
    static constexpr int oVp = oV + 64 * kBV;             // [64][kBV]  V'
    static constexpr int oL = oVp + 64 * kBV;             // [64][kLd]  L
    static constexpr int oX = oL + 64 * kLd;              // [64][kLd]  X = (I + L)^-1
    static constexpr int oP = oX + 64 * kLd;              // [64][kLd]  P
    static constexpr int oB = oP + 64 * kLd;              // [64]       beta
    static constexpr int total = oB + 64;
};

template <typename DT, int K, bool CHANNEL>
__global__ void __launch_bounds__(kThreads) simt_scan_kernel(const ScanArgs a)
{
    using Lay = SimtLayout<K, CHANNEL>;
    constexpr int KP = Lay::KP;
    extern __shared__ float smem[];
    float *sS = smem + Lay::oS, *sK = smem + Lay::oK, *sQ = smem + Lay::oQ, *sG = smem + Lay::oG;
    float *sGC = smem + Lay::oGC, *sV = smem + Lay::oV, *sVp = smem + Lay::oVp;
    float *sL = smem + Lay::oL, *sX = smem + Lay::oX, *sP = smem + Lay::oP, *sB = smem + Lay::oB;

    const int tid = threadIdx.x;
    const int vt = blockIdx.x, seg = blockIdx.y, pair = blockIdx.z;
    const int n = pair / a.HV, hv = pair % a.HV, hq = hv / (a.HV / a.H);
    int64_t bos, len;
    if (a.cu_seqlens) {
        bos = a.cu_seqlens[n];
        len = a.cu_seqlens[n + 1] - bos;
    } else {
        bos = (int64_t)n * a.T;
        len = a.T;
    }
    const int NT = (int)((len + kChunk - 1) / kChunk);
    const int c0 = seg * a.seg_chunks;
    if (seg > 0 && c0 >= NT) return;
    const int c1 = min(c0 + a.seg_chunks, NT);
    if (seg == a.n_seg - 1 && c1 < NT && tid == 0 && vt == 0) atomicOr(a.status, kStatusPlan);
    const int col0 = vt * kBV;
    const bool fwd = a.mode == kModeForward;
    const size_t sidx = ((size_t)n * a.HV + hv) * a.n_seg + seg;
    const int V = a.V;
    int cs = c0;
    if (fwd && a.warm_start) {
        cs = a.warm_start[sidx];
        if (cs < 0 || cs > c0) {  // inconsistent plan: fall back to the exact start
            if (tid == 0) atomicOr(a.status, kStatusPlan);
            cs = 0;
        }
    }
    const DT *q = (const DT *)a.q, *k = (const DT *)a.k, *v = (const DT *)a.v;

    // initial state slice
    for (int e = tid; e < K * kBV; e += kThreads) {
        const int d = e / kBV, col = col0 + e % kBV;
        float val = 0.f;
        if (fwd) {
            if (col < V) {
                if (a.seg_init && seg > 0)
                    val = a.seg_init[(sidx * K + d) * V + col];
                else if (cs == 0 && a.h0)
                    val = a.h0[(((size_t)n * a.HV + hv) * K + d) * V + col];
            }
        } else if (col >= V && col - V == d) {
            val = 1.f;  // the transition matrix M starts at the identity
        }
        sS[e] = val;
    }

    for (int c = cs; c < c1; ++c) {
        const bool emit = fwd && c >= c0 && a.o != nullptr;  // (no o: a state dump for the backward pass)
        const int64_t t0 = bos + (int64_t)c * kChunk;
        const int nrow = (int)rows_in_chunk(len, c);
        __syncthreads();  // previous chunk done with every buffer
        if (a.chunk_states) {
            // the state entering chunk c, for the backward pass
            float *dst = a.chunk_states + ((size_t)tile_slot(bos, n, c) * a.HV + hv) * K * V;
            for (int e = tid; e < K * kBV; e += kThreads) {
                const int d = e / kBV, col = col0 + e % kBV;
                if (col < V) dst[(size_t)d * V + col] = sS[e];
            }
        }

        // ---- 1. loads (rows past the sequence end are inert zeros)
        for (int e = tid; e < 64 * K; e += kThreads) {
            const int r = e / K, d = e % K;
            float kv = 0.f, qv = 0.f, gv = 0.f;
            if (r < nrow) {
                const size_t off = ((size_t)(t0 + r) * a.H + hq) * K + d;
                kv = to_f(k[off]);
                if (emit) qv = to_f(q[off]);
                if (CHANNEL) gv = act_gate(a.act, a.g[((size_t)(t0 + r) * a.HV + hv) * K + d], hv, d, K) * kRcpLn2;
            }
            sK[r * KP + d] = kv;
            sQ[r * KP + d] = qv;
            if (CHANNEL) sG[r * KP + d] = gv;
        }
        for (int e = tid; e < 64 * kBV; e += kThreads) {
            const int r = e / kBV, col = col0 + e % kBV;
            float vv = 0.f;
            if (r < nrow && col < V) vv = to_f(v[((size_t)(t0 + r) * a.HV + hv) * V + col]);
            sV[e] = vv;
        }
        if (tid < 64) {
            const bool ok = tid < nrow;
            sB[tid] = ok ? act_beta(a.act, a.beta[(size_t)(t0 + tid) * a.HV + hv]) : 0.f;
            if (!CHANNEL) sG[tid] = ok ? act_gate(a.act, a.g[(size_t)(t0 + tid) * a.HV + hv], hv, -1, K) * kRcpLn2 : 0.f;
        }
        __syncthreads();
        if (a.act.qk_l2norm) {
            // in-kernel L2 norm: every row of k (and of q when the chunk is emitted) to unit length
            if (tid < 128 && (tid < 64 || emit)) {
                float *row = (tid < 64 ? sK : sQ) + (tid & 63) * KP;
                float ss = 0.f;
                for (int d = 0; d < K; ++d) ss = fmaf(row[d], row[d], ss);
                const float rn = 1.f / fmaxf(sqrtf(ss), kNormEps);
                for (int d = 0; d < K; ++d) row[d] *= rn;
            }
            __syncthreads();
        }

        // ---- gate cumsum inside the chunk (inclusive)
        if (CHANNEL) {
            for (int d = tid; d < K; d += kThreads) {
                float acc = 0.f;
                for (int r = 0; r < 64; ++r) {
                    acc += sG[r * KP + d];
                    sG[r * KP + d] = acc;
                }
                sGC[d] = acc;
            }
        } else if (tid < 32) {
            const float x0 = sG[2 * tid], x1 = sG[2 * tid + 1];
            float s = x0 + x1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, s, off);
                if (tid >= off) s += y;
            }
            const float ex = s - (x0 + x1);
            sG[2 * tid] = ex + x0;
            sG[2 * tid + 1] = ex + x0 + x1;
            if (tid == 31) sGC[0] = s;
        }
        __syncthreads();

        // ---- 2. gated K K^T (strictly lower, times beta_i) and Q K^T (lower incl. diagonal)
        {
            const int bi = tid >> 4, bj = tid & 15;
            const int i0 = 4 * bi, j0 = 4 * bj;
            if (bj <= bi) {
                float ak[4][4], aq[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int w = 0; w < 4; ++w) ak[u][w] = aq[u][w] = 0.f;
#pragma unroll 4
                for (int d = 0; d < K; ++d) {
                    float ki[4], qi[4], kj[4];
                    if (CHANNEL) {
                        // reference point j0 keeps both factors bounded:
                        // 2^(G_i - G_j) = 2^(G_i - G_j0) * 2^(G_j0 - G_j)
                        const float gr = sG[j0 * KP + d];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float fi = ex2(sG[(i0 + u) * KP + d] - gr);
                            ki[u] = sK[(i0 + u) * KP + d] * fi;
                            qi[u] = sQ[(i0 + u) * KP + d] * fi;
                            kj[u] = sK[(j0 + u) * KP + d] * ex2(gr - sG[(j0 + u) * KP + d]);
                        }
                    } else {
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            ki[u] = sK[(i0 + u) * KP + d];
                            qi[u] = sQ[(i0 + u) * KP + d];
                            kj[u] = sK[(j0 + u) * KP + d];
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            ak[u][w] = fmaf(ki[u], kj[w], ak[u][w]);
                            aq[u][w] = fmaf(qi[u], kj[w], aq[u][w]);
                        }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int i = i0 + u, j = j0 + w;
                        float lv = 0.f, pv = 0.f;
                        if (j <= i) {
                            const float gf = CHANNEL ? 1.f : ex2(sG[i] - sG[j]);
                            if (j < i) lv = sB[i] * gf * ak[u][w];
                            pv = gf * aq[u][w];
                        }
                        sL[i * kLd + j] = lv;
                        sP[i * kLd + j] = pv;
                    }
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        sL[(i0 + u) * kLd + j0 + w] = 0.f;
                        sP[(i0 + u) * kLd + j0 + w] = 0.f;
                    }
            }
        }
        __syncthreads();

        // ---- per-channel gate: fold the decays into k and q (in place)
        if (CHANNEL) {
            for (int e = tid; e < 64 * K; e += kThreads) {
                const int r = e / K, d = e % K;
                const float G = sG[r * KP + d], kv = sK[r * KP + d];
                sG[r * KP + d] = kv * ex2(sGC[d] - G);  // k * 2^(G_C - G): state write
                sK[r * KP + d] = kv * ex2(G);           // k * 2^G: read-out of the old state
                if (emit) sQ[r * KP + d] *= ex2(G);     // q * 2^G: inter-chunk output
            }
        }

        // ---- 3. X = (I + L)^-1: each column by 4 lanes, forward substitution
        {
            const int col = tid >> 2, r4 = tid & 3;
            for (int j = r4; j < 64; j += 4) sX[j * kLd + col] = (j == col) ? 1.f : 0.f;
            __syncwarp();
            const int first = (tid >> 5) * 8 + 1;  // smallest column of this warp, plus one
            for (int i = first; i < 64; ++i) {
                float part = 0.f;
                if (i > col)
                    for (int j = col + r4; j < i; j += 4) part = fmaf(sL[i * kLd + j], sX[j * kLd + col], part);
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                if (r4 == 0 && i > col) sX[i * kLd + col] = -part;
                __syncwarp();
            }
        }
        __syncthreads();

        const int cc = tid & 31, r0 = (tid >> 5) * 8;
        // ---- 4. beta * R = beta * (V - (K 2^G) S)
        {
            float acc[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[u] = 0.f;
#pragma unroll 4
            for (int d = 0; d < K; ++d) {
                const float s = sS[d * kBV + cc];
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[u] = fmaf(sK[(r0 + u) * KP + d], s, acc[u]);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = r0 + u;
                const float ks = CHANNEL ? acc[u] : ex2(sG[i]) * acc[u];
                sV[i * kBV + cc] = sB[i] * (sV[i * kBV + cc] - ks);
            }
        }
        __syncthreads();

        // ---- 5. V' = X (beta R)
        {
            float acc[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[u] = 0.f;
            for (int j = 0; j < r0 + 8; ++j) {
                const float rv = sV[j * kBV + cc];
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[u] = fmaf(sX[(r0 + u) * kLd + j], rv, acc[u]);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) sVp[(r0 + u) * kBV + cc] = acc[u];
        }
        __syncthreads();

        // ---- 6. O = scale [ (Q 2^G) S + P V' ]   (S is still the state entering the chunk)
        if (emit) {
            float acc[8], acc2[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) acc[u] = acc2[u] = 0.f;
#pragma unroll 4
            for (int d = 0; d < K; ++d) {
                const float s = sS[d * kBV + cc];
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[u] = fmaf(sQ[(r0 + u) * KP + d], s, acc[u]);
            }
            for (int j = 0; j < r0 + 8; ++j) {
                const float vp = sVp[j * kBV + cc];
#pragma unroll
                for (int u = 0; u < 8; ++u) acc2[u] = fmaf(sP[(r0 + u) * kLd + j], vp, acc2[u]);
            }
            const int col = col0 + cc;
            if (col < V) {
                DT *o = (DT *)a.o;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = r0 + u;
                    if (i < nrow) {
                        const float inter = CHANNEL ? acc[u] : ex2(sG[i]) * acc[u];
                        from_f(o + ((size_t)(t0 + i) * a.HV + hv) * V + col, a.scale * (inter + acc2[u]));
                    }
                }
            }
        }
        __syncthreads();

        // ---- 7. S <- Diag(2^G_C) S + (K 2^(G_C - G))^T V'
        {
            constexpr int DPT = K / 8;  // state rows per thread
            const int dr = tid >> 5;
            float acc[DPT];
#pragma unroll
            for (int m = 0; m < DPT; ++m) {
                const int d = dr + 8 * m;
                const float decay = ex2(CHANNEL ? sGC[d] : sGC[0]);
                acc[m] = decay * sS[d * kBV + cc];
            }
            for (int j = 0; j < 64; ++j) {
                const float vp = sVp[j * kBV + cc];
                const float rowf = CHANNEL ? 1.f : ex2(sGC[0] - sG[j]);
#pragma unroll
                for (int m = 0; m < DPT; ++m) {
                    const int d = dr + 8 * m;
                    const float kt = CHANNEL ? sG[j * KP + d] : rowf * sK[j * KP + d];
                    acc[m] = fmaf(kt, vp, acc[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < DPT; ++m) sS[(dr + 8 * m) * kBV + cc] = acc[m];
        }
    }
    __syncthreads();

    // final state of this segment
    if (fwd) {
        if (c1 == NT && a.ht) {
            for (int e = tid; e < K * kBV; e += kThreads) {
                const int d = e / kBV, col = col0 + e % kBV;
                if (col < V) a.ht[(((size_t)n * a.HV + hv) * K + d) * V + col] = sS[e];
            }
        }
    } else {
        const int VE = V + K;
        for (int e = tid; e < K * kBV; e += kThreads) {
            const int d = e / kBV, col = col0 + e % kBV;
            if (col < VE) a.seg_out[(sidx * K + d) * VE + col] = sS[e];
        }
    }
}

// Exact split, step 2.2 of the FlashQLA blog: S_start(j+1) = S*_j + M_j S_start(j),
// serial over the segments of one (sequence, head), one CTA per 32-column tile.
template <int K>
__global__ void __launch_bounds__(kThreads) cp_combine_kernel(const CombineArgs a)
{
    extern __shared__ float smem[];
    float *sS = smem, *sT = smem + K * kBV;
    const int tid = threadIdx.x, pair = blockIdx.y, col0 = blockIdx.x * kBV;
    const int n = pair / a.HV, hv = pair % a.HV;
    const int64_t len = a.cu_seqlens ? a.cu_seqlens[n + 1] - a.cu_seqlens[n] : (int64_t)a.T;
    const int NT = (int)((len + kChunk - 1) / kChunk);
    int nseg = max(1, ceil_div(NT, a.seg_chunks));
    if (nseg > a.n_seg) {  // a sequence longer than the plan's bound: never index past the grid
        if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(a.status, kStatusPlan);
        nseg = a.n_seg;
    }
    const int V = a.V, VE = a.V + K;
    for (int e = tid; e < K * kBV; e += kThreads) {
        const int d = e / kBV, col = col0 + e % kBV;
        sS[e] = (a.h0 && col < V) ? a.h0[(((size_t)n * a.HV + hv) * K + d) * V + col] : 0.f;
    }
    __syncthreads();
    for (int j = 0; j + 1 < nseg; ++j) {
        const float *so = a.seg_out + (((size_t)n * a.HV + hv) * a.n_seg + j) * K * VE;
        for (int e = tid; e < K * kBV; e += kThreads) {
            const int d = e / kBV, cc = e % kBV, col = col0 + cc;
            float acc = col < V ? so[(size_t)d * VE + col] : 0.f;
            const float *Mrow = so + (size_t)d * VE + V;
#pragma unroll 8
            for (int m = 0; m < K; ++m) acc = fmaf(Mrow[m], sS[m * kBV + cc], acc);
            sT[e] = acc;
        }
        __syncthreads();
        float *dst = a.seg_init + (((size_t)n * a.HV + hv) * a.n_seg + j + 1) * K * V;
        for (int e = tid; e < K * kBV; e += kThreads) {
            const int d = e / kBV, col = col0 + e % kBV;
            sS[e] = sT[e];
            if (col < V) dst[(size_t)d * V + col] = sT[e];
        }
        __syncthreads();
    }
}

// Start states of consecutive pieces of one sequence from their summaries (the context-parallel
// exchange across ranks: FlashQLA blog, "Key problems", the S* / M pre-process, applied to the pieces
// held by successive ranks): starts[0] = h0, starts[r + 1] = S*_r + M_r starts[r].  Summaries are
// [ranks][pairs][K][V + K] (S* in the first V columns of each row, M in the last K), starts
// [ranks][pairs][K][V].  One CTA per (32-column value tile, pair), serial over the ranks.
template <int K>
__global__ void __launch_bounds__(kThreads) chain_states_kernel(const ChainArgs a)
{
    extern __shared__ float smem[];
    float *sS = smem, *sT = smem + K * kBV;
    const int tid = threadIdx.x, pair = blockIdx.y, col0 = blockIdx.x * kBV;
    const int V = a.V, VE = a.V + K;
    const size_t pairs = (size_t)a.pairs;
    for (int e = tid; e < K * kBV; e += kThreads) {
        const int d = e / kBV, col = col0 + e % kBV;
        const float x = (a.h0 && col < V) ? a.h0[((size_t)pair * K + d) * V + col] : 0.f;
        sS[e] = x;
        if (col < V) a.starts[((size_t)pair * K + d) * V + col] = x;
    }
    __syncthreads();
    for (int r = 0; r + 1 < a.ranks; ++r) {
        const float *so = a.summaries + ((size_t)r * pairs + pair) * K * VE;
        for (int e = tid; e < K * kBV; e += kThreads) {
            const int d = e / kBV, cc = e % kBV, col = col0 + cc;
            float acc = col < V ? so[(size_t)d * VE + col] : 0.f;
            const float *Mrow = so + (size_t)d * VE + V;
#pragma unroll 8
            for (int m = 0; m < K; ++m) acc = fmaf(Mrow[m], sS[m * kBV + cc], acc);
            sT[e] = acc;
        }
        __syncthreads();
        float *dst = a.starts + ((size_t)(r + 1) * pairs + pair) * K * V;
        for (int e = tid; e < K * kBV; e += kThreads) {
            const int d = e / kBV, col = col0 + e % kBV;
            sS[e] = sT[e];
            if (col < V) dst[(size_t)d * V + col] = sT[e];
        }
        __syncthreads();
    }
}

// Gate statistics for the warmup split (FlashQLA blog, "Further optimisation
// via gate decay": the warmup length of each segment comes from a separate
// gate-statistics kernel).  Per chunk the base-2 log of an upper bound on the
// decay (scalar gate: sum of g; per-channel gate: sum over tokens of the
// largest channel's g), then per segment the walk back from its first chunk
// until the accumulated log-decay is <= log2_eps.
__global__ void __launch_bounds__(kThreads) gate_stats_kernel(const GateStatsArgs a)
{
    extern __shared__ float csum[];  // [max chunks of one sequence]
    const int tid = threadIdx.x, pair = blockIdx.x;
    const int n = pair / a.HV, hv = pair % a.HV;
    int64_t bos, len;
    if (a.cu_seqlens) {
        bos = a.cu_seqlens[n];
        len = a.cu_seqlens[n + 1] - bos;
    } else {
        bos = (int64_t)n * a.T;
        len = a.T;
    }
    const int NT = (int)((len + kChunk - 1) / kChunk);
    const int nseg = max(1, ceil_div(NT, a.seg_chunks));
    const int cap = a.n_seg * a.seg_chunks;  // shared-memory capacity in chunks
    const int warp = tid >> 5, lane = tid & 31, nwarps = blockDim.x >> 5;
    for (int c = warp; c < NT && c < cap; c += nwarps) {
        // one warp per chunk: lane l takes tokens l and l + 32
        const int rows = (int)min((int64_t)kChunk, len - (int64_t)c * kChunk);
        float part = 0.f;
        for (int r = lane; r < rows; r += 32) {
            const size_t t = (size_t)(bos + (int64_t)c * kChunk + r);
            if (a.channel) {
                const float *gt = a.g + (t * a.HV + hv) * a.K;
                float mx = act_gate(a.act, gt[0], hv, 0, a.K);
                for (int d = 1; d < a.K; ++d) mx = fmaxf(mx, act_gate(a.act, gt[d], hv, d, a.K));
                part += mx;
            } else {
                part += act_gate(a.act, a.g[t * a.HV + hv], hv, -1, a.K);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (lane == 0) csum[c] = part * kRcpLn2;
    }
    __syncthreads();
    int *ws = a.warm_start + ((size_t)n * a.HV + hv) * a.n_seg;
    for (int j = tid; j < a.n_seg; j += blockDim.x) {
        int w = 0;
        if (j > 0 && j < nseg) {
            const int c0 = j * a.seg_chunks;
            float acc = 0.f;
            int c = c0;
            w = 0;
            while (c > 0) {
                --c;
                acc += csum[c];
                if (acc <= a.log2_eps) {
                    w = c;
                    break;
                }
                if (c0 - c >= a.max_warm_chunks) {
                    w = 0;
                    break;
                }
            }
        }
        ws[j] = w;
    }
}

template <typename DT, int K, bool CH>
cudaError_t launch_scan_t(const ScanArgs &a, cudaStream_t st)
{
    const size_t smem = sizeof(float) * SimtLayout<K, CH>::total;
    auto kern = simt_scan_kernel<DT, K, CH>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(ceil_div(a.vext, kBV), a.n_seg, a.N * a.HV);
    kern<<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

template <typename DT, bool CH>
cudaError_t launch_scan_k(const ScanArgs &a, cudaStream_t st)
{
    switch (a.K) {
    case 32: return launch_scan_t<DT, 32, CH>(a, st);
    case 64: return launch_scan_t<DT, 64, CH>(a, st);
    case 128: return launch_scan_t<DT, 128, CH>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t simt_smem_bytes(int K, gdn_gate_kind gate)
{
    const bool ch = gate == GDN_GATE_CHANNEL;
    switch (K) {
    case 32: return sizeof(float) * (ch ? SimtLayout<32, true>::total : SimtLayout<32, false>::total);
    case 64: return sizeof(float) * (ch ? SimtLayout<64, true>::total : SimtLayout<64, false>::total);
    case 128: return sizeof(float) * (ch ? SimtLayout<128, true>::total : SimtLayout<128, false>::total);
    default: return 0;
    }
}

cudaError_t launch_simt_scan(const ScanArgs &a, gdn_dtype dt, gdn_gate_kind gate, cudaStream_t st)
{
    if (a.N * a.HV == 0) return cudaSuccess;
    const bool ch = gate == GDN_GATE_CHANNEL;
    if (dt == GDN_F32) return ch ? launch_scan_k<float, true>(a, st) : launch_scan_k<float, false>(a, st);
    return ch ? launch_scan_k<__nv_bfloat16, true>(a, st) : launch_scan_k<__nv_bfloat16, false>(a, st);
}

cudaError_t launch_cp_combine(const CombineArgs &a, cudaStream_t st)
{
    if (a.N * a.HV == 0) return cudaSuccess;
    dim3 grid(ceil_div(a.V, kBV), a.N * a.HV);
    const size_t smem = sizeof(float) * 2 * a.K * kBV;
    switch (a.K) {
    case 32: cp_combine_kernel<32><<<grid, kThreads, smem, st>>>(a); break;
    case 64: cp_combine_kernel<64><<<grid, kThreads, smem, st>>>(a); break;
    case 128: cp_combine_kernel<128><<<grid, kThreads, smem, st>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_chain_states(const ChainArgs &a, cudaStream_t st)
{
    if (a.ranks <= 0 || a.pairs <= 0 || a.V <= 0) return cudaSuccess;
    const dim3 grid(ceil_div(a.V, kBV), a.pairs);
    const size_t smem = 2 * sizeof(float) * (size_t)a.K * kBV;
    switch (a.K) {
    case 32: chain_states_kernel<32><<<grid, kThreads, smem, st>>>(a); break;
    case 64: chain_states_kernel<64><<<grid, kThreads, smem, st>>>(a); break;
    case 128: chain_states_kernel<128><<<grid, kThreads, smem, st>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// Batched fp32 transpose through 32 x 33 shared tiles (coalesced reads and writes).
__global__ void __launch_bounds__(256) transpose_kernel(const float *src, float *dst, int A, int B)
{
    __shared__ float t[32][33];
    const size_t p = blockIdx.z;
    const int a0 = blockIdx.y * 32, b0 = blockIdx.x * 32, tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const float *s = src + p * (size_t)A * B;
    float *d = dst + p * (size_t)A * B;
    for (int i = ty; i < 32; i += 8)
        if (a0 + i < A && b0 + tx < B) t[i][tx] = s[(size_t)(a0 + i) * B + b0 + tx];
    __syncthreads();
    for (int i = ty; i < 32; i += 8)
        if (b0 + i < B && a0 + tx < A) d[(size_t)(b0 + i) * A + a0 + tx] = t[tx][i];
}

cudaError_t launch_transpose(const float *src, float *dst, int P, int A, int B, cudaStream_t st)
{
    if (P == 0 || A == 0 || B == 0) return cudaSuccess;
    if (P > 65535) return cudaErrorInvalidValue;
    transpose_kernel<<<dim3(ceil_div(B, 32), ceil_div(A, 32), P), 256, 0, st>>>(src, dst, A, B);
    return cudaGetLastError();
}

cudaError_t launch_gate_stats(const GateStatsArgs &a, cudaStream_t st)
{
    if (a.N * a.HV == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * (size_t)a.n_seg * a.seg_chunks;
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(gate_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    gate_stats_kernel<<<a.N * a.HV, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn

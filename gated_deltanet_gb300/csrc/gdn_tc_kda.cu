// Chunk preparation for the tensor-core engine with per-key-channel gates (the
// "KDA source walkthrough" chunk form): for every chunk of every (sequence, value
// head), everything of the chunk that does not depend on the state, as bf16 tiles
// the scan loads with TMA.  With G = chunk-local inclusive cumsum of the log-gate
// per channel (base 2), G_C = G of the last row:
//
//   Akk_ij = beta_i sum_d k_id k_jd 2^(G_id - G_jd)   (j < i)     gated K K^T
//   Aqk_ij =        sum_d q_id k_jd 2^(G_id - G_jd)   (j <= i)    gated Q K^T
//   X      = (I + Akk)^-1
//   U      = X diag(beta) V,   W = X diag(beta) (K * 2^G)         WY form: V' = U - W S
//   K^     = K * 2^(G_C - G),  Q~ = scale Q * 2^G,  P = scale Aqk
//   gC_d   = 2^(G_C,d)                                            per-channel state decay
//
// so that the scan computes V' = U - W S, O = Q~ S + P V', S <- diag(gC) S + K^T V'.
// Both gated products take each 2^(G_i - G_j) as 2^(G_i - G_r) 2^(G_r - G_j) with r
// the first row of j's group of four, so no factor overflows.
//
// Tiles: bf16 [slot][HV][9][64][64] (boxes: K^ dk 0-63, Q~ dk 0-63, K^ dk 64-127, Q~ dk 64-127,
// U dv 0-63, U dv 64-127, -W dk 0-63, -W dk 64-127, P), rows of 64 elements; gC fp32
// [slot][HV][128].  One CTA of 256 threads per (slot, value head), two per SM (102 KB of shared
// memory: four buffers that change roles as the chunk's data dies).
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {
using namespace ptx;

constexpr int kThreadsKda = 256;
constexpr int KP = 132;  // fp32 row pitch of G (rows 16-byte aligned)
constexpr int QP = 136;  // bf16 row pitch of q
constexpr int kLdX = 68;  // fp32 row pitch of the L / X tile

struct KdaSmem {
    __nv_bfloat16 k[64 * QP];  // k (bf16 input, exact), then k * 2^G
    __nv_bfloat16 q[64 * QP];    // q until Q~ is written, then v
    float g[64 * KP];            // G (base 2, chunk-local cumsum per channel)
    float lx[64 * kLdX];         // L = beta_i Akk_ij in the lower triangle, then X^T in the upper:
                                 // X(r, j), j < r, at lx[j * kLdX + r]
    __nv_bfloat16 kj[64 * QP];   // k_j 2^(G_r - G_j), r = first row of j's 16-row block
    float beta[64];
    float gc[128];
    float wpart[8];              // warmup split: each warp's share of the chunk's log-decay bound
};
static_assert(64 * KP * sizeof(float) >= 4 * 8192 + 1024, "the U / -W staging boxes fit the G buffer");

__device__ __forceinline__ int rows_in(int64_t len, int c)
{
    const int64_t r = len - (int64_t)c * kChunk;
    return r < kChunk ? (int)r : kChunk;
}

// element (row r, column col) of a 64 x 128 matrix stored as two [64][64] boxes b0, b0 + 1
__device__ __forceinline__ size_t box_index(int b0, int r, int col) { return (size_t)((b0 + (col >> 6)) * 64 + r) * 64 + (col & 63); }

__global__ void __launch_bounds__(kThreadsKda, 2) kda_prep_kernel(const KdaPrepArgs a,
                                                                  const __grid_constant__ CUtensorMap tmap)
{
    extern __shared__ __align__(16) uint8_t kda_raw[];
    KdaSmem &sh = *(KdaSmem *)kda_raw;
    const int tid = threadIdx.x;
    if (a.seq_order && blockIdx.x == 0 && blockIdx.y == 0) {  // the scan's CTA order (G's buffer as scratch)
        order_longest_first(a.cu_seqlens, a.N, a.n_buckets, (int *)sh.g, a.seq_order);
        __syncthreads();
    }
    const int slot = blockIdx.x, hv = blockIdx.y;
    const int HV = a.HV, hq = hv / (HV / a.H);
    auto seq_start = [&](int m) -> int64_t { return a.cu_seqlens ? a.cu_seqlens[m] : (int64_t)m * a.T; };
    // the sequence owning this slot: the last n with tile_slot(bos_n, n, 0) <= slot
    int lo = 0, hi = a.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_slot(seq_start(mid), mid, 0) <= slot) lo = mid; else hi = mid - 1;
    }
    const int n = lo;
    const int64_t bos = seq_start(n), len = seq_start(n + 1) - bos;
    const int c = (int)(slot - tile_slot(bos, n, 0));
    const int NT = (int)((len + kChunk - 1) / kChunk);
    if (c < 0 || c >= NT) return;  // an unused slot
    const int rows = rows_in(len, c);
    const int64_t t0 = bos + (int64_t)c * kChunk;
    const __nv_bfloat16 *qg = (const __nv_bfloat16 *)a.q, *kg = (const __nv_bfloat16 *)a.k;
    const __nv_bfloat16 *vg = (const __nv_bfloat16 *)a.v;
    __nv_bfloat16 *tile = (__nv_bfloat16 *)a.tiles + ((size_t)slot * HV + hv) * 9 * 4096;

    // v is read only after the inverse: start bringing its rows into L2 now
    if (tid < rows) prefetch_l2(vg + ((size_t)(t0 + tid) * HV + hv) * 128, 256);
    // ---- k, q, log-gates (rows past the end of the sequence are inert zeros), beta: 16-byte loads,
    //      all issued before the first store
    {
        uint4 kv[4], qv[4];
        float4 gv[8];
        // a thread's four channels are the same in every row: the activation's per-channel bias and the
        // head's exp(A_log) are taken once
        float ea = 0.f;
        float4 bias = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.act.A_log) {
            ea = expf(a.act.A_log[hv]);
            if (a.act.dt_bias) {
                const float *bp = a.act.dt_bias + (size_t)hv * 128 + (tid & 31) * 4;
                bias = make_float4(bp[0], bp[1], bp[2], bp[3]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = tid + kThreadsKda * i, r = e >> 4, c8 = (e & 15) * 8;
            kv[i] = qv[i] = make_uint4(0, 0, 0, 0);
            if (r < rows) {
                const size_t off = ((size_t)(t0 + r) * a.H + hq) * 128 + c8;
                kv[i] = *(const uint4 *)(kg + off);
                qv[i] = *(const uint4 *)(qg + off);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = tid + kThreadsKda * i, r = e >> 5, c4 = (e & 31) * 4;
            gv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < rows) gv[i] = *(const float4 *)(a.gk + ((size_t)(t0 + r) * HV + hv) * 128 + c4);
        }
        if (a.act.A_log) {
            // raw gate input: the activation, per channel, once every load is issued (rows past the end
            // stay 0)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (((tid + kThreadsKda * i) >> 5) < rows) {
                    gv[i].x = act_gate_pre(a.act, gv[i].x, bias.x, ea);
                    gv[i].y = act_gate_pre(a.act, gv[i].y, bias.y, ea);
                    gv[i].z = act_gate_pre(a.act, gv[i].z, bias.z, ea);
                    gv[i].w = act_gate_pre(a.act, gv[i].w, bias.w, ea);
                }
            }
        }
        if (a.wdec) {
            // warmup split: the chunk's bound on the state's decay, per token the slowest channel's (largest)
            // log-gate summed over the tokens, as the CUDA-core engine's gate statistics take it; warp w holds
            // every channel of rows w + 8 i (rows past the end of the sequence are 0)
            float part = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float m = fmaxf(fmaxf(gv[i].x, gv[i].y), fmaxf(gv[i].z, gv[i].w));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                part += m;
            }
            if ((tid & 31) == 0) sh.wpart[tid >> 5] = part;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = tid + kThreadsKda * i, r = e >> 4, c8 = (e & 15) * 8;
            *(uint4 *)(sh.k + r * QP + c8) = kv[i];  // bf16 as given (exact)
            *(uint4 *)(sh.q + r * QP + c8) = qv[i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = tid + kThreadsKda * i, r = e >> 5, c4 = (e & 31) * 4;
            *(float4 *)(sh.g + r * KP + c4) =
                make_float4(gv[i].x * kRcpLn2, gv[i].y * kRcpLn2, gv[i].z * kRcpLn2, gv[i].w * kRcpLn2);
        }
    }
    if (tid < 64) sh.beta[tid] = tid < rows ? act_beta(a.act, a.beta[(size_t)(t0 + tid) * HV + hv]) : 0.f;
    __syncthreads();
    if (a.wdec && tid == 0) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kThreadsKda / 32; ++w) sum += sh.wpart[w];
        a.wdec[(size_t)slot * HV + hv] = sum * kRcpLn2;
    }
    if (a.check_norm) {
        // the warmup split relies on beta ||k||^2 <= 2 (non-expansive transitions): four threads per row
        const int r = tid >> 2, pc = tid & 3;
        const __nv_bfloat16 *row = sh.k + r * QP + 32 * pc;
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = *(const uint4 *)(row + 8 * j);
            const __nv_bfloat162 *h2 = (const __nv_bfloat162 *)&x;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h2[u]);
                ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
            }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        if (pc == 0 && r < rows && sh.beta[r] * ss > 2.0001f) atomicOr(a.status, kStatusNormBound);
    }
    if (a.act.qk_l2norm) {
        // in-kernel L2 norm: the rows of k and q to unit length (fp32 arithmetic, one bf16 rounding, as
        // every operand of the products below is bf16); two threads per row, eight 16-byte pieces each
        const int rr = tid >> 1, h = tid & 1;
        __nv_bfloat16 *row = (rr < 64 ? sh.k : sh.q) + (rr & 63) * QP + 64 * h;
        uint4 x[8];
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            x[j] = *(const uint4 *)(row + 8 * j);
            const __nv_bfloat162 *b2 = (const __nv_bfloat162 *)&x[j];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(b2[u]);
                ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
            }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        const float rn = 1.f / fmaxf(sqrtf(ss), kNormEps);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            __nv_bfloat162 *b2 = (__nv_bfloat162 *)&x[j];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(b2[u]);
                b2[u] = __floats2bfloat162_rn(f.x * rn, f.y * rn);
            }
            *(uint4 *)(row + 8 * j) = x[j];
        }
        __syncthreads();
    }
    // ---- per-channel inclusive cumsum (one thread per channel)
    if (tid < 128) {
        float acc = 0.f;
        for (int r = 0; r < 64; ++r) {
            acc += sh.g[r * KP + tid];
            sh.g[r * KP + tid] = acc;
        }
        sh.gc[tid] = acc;
    }
    __syncthreads();

    // ---- gated K K^T (times beta_i, strictly lower) and Q K^T (lower with the diagonal).  On the tensor
    //      cores: for the 16-row key block b with reference row r = 16 b, [K; Q]_i 2^(G_i - G_r) times
    //      (k_j 2^(G_r - G_j))^T; the factors stay bounded while the decay inside a block is below 2^100
    float emax = 0.f;
#pragma unroll 2
    for (int e = tid; e < 64 * 32; e += kThreadsKda) {  // four channels per step
        const int j = e >> 5, d = (e & 31) * 4, r = j & ~15;
        const float4 gr = *(const float4 *)(sh.g + r * KP + d), gj = *(const float4 *)(sh.g + j * KP + d);
        const uint2 kk = *(const uint2 *)(sh.k + j * QP + d);
        const float2 k01 = __bfloat1622float2(*(const __nv_bfloat162 *)&kk.x);
        const float2 k23 = __bfloat1622float2(*(const __nv_bfloat162 *)&kk.y);
        const float e0 = gr.x - gj.x, e1 = gr.y - gj.y, e2 = gr.z - gj.z, e3 = gr.w - gj.w;
        emax = fmaxf(emax, fmaxf(fmaxf(e0, e1), fmaxf(e2, e3)));
        *(uint2 *)(sh.kj + j * QP + d) = make_uint2(ptx::pack_bf16(k01.x * ex2(e0), k01.y * ex2(e1)),
                                                    ptx::pack_bf16(k23.x * ex2(e2), k23.y * ex2(e3)));
    }
    // K^ = k 2^(G_C - G) and Q~ = scale q 2^G to the tiles (four channels per step, a warp writes one row);
    // k, q and G are only read here, so this runs beside the gated products
    auto khat_qtilde_out = [&](int first, int stride) {
#pragma unroll 2
        for (int e = first; e < 64 * 32; e += stride) {
            const int r = e >> 5, c4 = (e & 31) * 4;
            const float4 G4 = *(const float4 *)(sh.g + r * KP + c4), gc4 = *(const float4 *)(sh.gc + c4);
            const uint2 kk = *(const uint2 *)(sh.k + r * QP + c4), qq = *(const uint2 *)(sh.q + r * QP + c4);
            const float2 k01 = __bfloat1622float2(*(const __nv_bfloat162 *)&kk.x);
            const float2 k23 = __bfloat1622float2(*(const __nv_bfloat162 *)&kk.y);
            const float2 q01 = __bfloat1622float2(*(const __nv_bfloat162 *)&qq.x);
            const float2 q23 = __bfloat1622float2(*(const __nv_bfloat162 *)&qq.y);
            const uint2 kh = make_uint2(ptx::pack_bf16(k01.x * ex2(gc4.x - G4.x), k01.y * ex2(gc4.y - G4.y)),
                                        ptx::pack_bf16(k23.x * ex2(gc4.z - G4.z), k23.y * ex2(gc4.w - G4.w)));
            const uint2 qt = make_uint2(ptx::pack_bf16(a.scale * q01.x * ex2(G4.x), a.scale * q01.y * ex2(G4.y)),
                                        ptx::pack_bf16(a.scale * q23.x * ex2(G4.z), a.scale * q23.y * ex2(G4.w)));
            *(uint2 *)(tile + box_index(0, r, c4) + (c4 >= 64 ? 64 * 64 : 0)) = kh;  // K^: boxes 0, 2
            *(uint2 *)(tile + box_index(1, r, c4) + (c4 >= 64 ? 64 * 64 : 0)) = qt;  // Q~: boxes 1, 3
        }
    };
    if (!__syncthreads_or(emax > 100.f)) {
        const int warp = tid >> 5, lane = tid & 31, gq = lane >> 2, t = lane & 3;
        // item = (key block b, 16-row tile mt >= b): ten of them over the eight warps
        for (int item = warp; item < 10; item += 8) {
            const int b = item < 4 ? 0 : item < 7 ? 1 : item < 9 ? 2 : 3;
            const int mt = item < 4 ? item : item < 7 ? item - 3 : item < 9 ? item - 5 : 3;
            const int r = 16 * b, i0 = 16 * mt, j0 = 16 * b;
            float ak[2][4], aq[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) ak[nt][c] = aq[nt][c] = 0.f;
#pragma unroll 4
            for (int ks = 0; ks < 8; ++ks) {
                const int d0 = 16 * ks + 2 * t;
                // A fragments (rows i0 + gq (+8), columns d0, d0 + 1 (+8)) with the factor 2^(G_i - G_r)
                uint32_t fk[4], fq[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int i = i0 + gq + 8 * (h & 1), d = d0 + 8 * (h >> 1);
                    const float2 gi = *(const float2 *)(sh.g + i * KP + d), gr = *(const float2 *)(sh.g + r * KP + d);
                    const float f0 = ex2(gi.x - gr.x), f1 = ex2(gi.y - gr.y);
                    const __nv_bfloat162 kk = *(const __nv_bfloat162 *)(sh.k + i * QP + d);
                    const __nv_bfloat162 qq = *(const __nv_bfloat162 *)(sh.q + i * QP + d);
                    fk[h] = ptx::pack_bf16(__low2float(kk) * f0, __high2float(kk) * f1);
                    fq[h] = ptx::pack_bf16(__low2float(qq) * f0, __high2float(qq) * f1);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int j = j0 + 8 * nt + gq;
                    const uint32_t b0 = *(const uint32_t *)(sh.kj + j * QP + d0);
                    const uint32_t b1 = *(const uint32_t *)(sh.kj + j * QP + d0 + 8);
                    ptx::mma_bf16_16816(ak[nt], fk[0], fk[1], fk[2], fk[3], b0, b1);
                    ptx::mma_bf16_16816(aq[nt], fq[0], fq[1], fq[2], fq[3], b0, b1);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {  // rows i0 + gq and i0 + gq + 8; columns j, j + 1
                    const int i = i0 + gq + 8 * hr, j = j0 + 8 * nt + 2 * t;
                    const float b = sh.beta[i];
                    sh.lx[i * kLdX + j] = j < i ? b * ak[nt][2 * hr] : 0.f;
                    sh.lx[i * kLdX + j + 1] = j + 1 < i ? b * ak[nt][2 * hr + 1] : 0.f;
                    *(uint32_t *)(tile + (size_t)(8 * 64 + i) * 64 + j) =
                        ptx::pack_bf16(j <= i ? a.scale * aq[nt][2 * hr] : 0.f, j + 1 <= i ? a.scale * aq[nt][2 * hr + 1] : 0.f);
                }
        }
        // warps 2-7 have one item, warps 0 and 1 two: the others write K^, Q~ and the zero blocks of P
        // (above the diagonal blocks; L there is never read) meanwhile
        if (warp >= 2) {
            khat_qtilde_out(tid - 64, kThreadsKda - 64);
            for (int e = tid - 64; e < 64 * 64; e += kThreadsKda - 64) {
                const int i = e >> 6, j = e & 63;
                if ((j >> 4) > (i >> 4)) tile[(size_t)(8 * 64 + i) * 64 + j] = __float2bfloat16_rn(0.f);
            }
        }
    } else {
        // steep chunk: per-element factors with a reference row per group of four (4 x 4 blocks)
        const int bi = tid >> 4, bj = tid & 15;
        const int i0 = 4 * bi, j0 = 4 * bj;
        if (bj <= bi) {
            float ak[4][4], aq[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int w = 0; w < 4; ++w) ak[u][w] = aq[u][w] = 0.f;
#pragma unroll 4
            for (int dd = 0; dd < 128; ++dd) {
                // reference row j0: 2^(G_i - G_j) = 2^(G_i - G_j0) 2^(G_j0 - G_j), both factors bounded.
                // Each thread starts at its own channel so that the sixteen j0 of a warp read distinct banks.
                const int d = (dd + bj) & 127;
                const float gr = sh.g[j0 * KP + d];
                float ki[4], qi[4], kj[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float fi = ex2(sh.g[(i0 + u) * KP + d] - gr);
                    ki[u] = __bfloat162float(sh.k[(i0 + u) * QP + d]) * fi;
                    qi[u] = __bfloat162float(sh.q[(i0 + u) * QP + d]) * fi;
                    kj[u] = __bfloat162float(sh.k[(j0 + u) * QP + d]) * ex2(gr - sh.g[(j0 + u) * KP + d]);
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
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u;
                float pv[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int j = j0 + w;
                    sh.lx[i * kLdX + j] = j < i ? sh.beta[i] * ak[u][w] : 0.f;
                    pv[w] = j <= i ? a.scale * aq[u][w] : 0.f;
                }
                // P = scale Aqk -> box 8, four columns per 8-byte store
                *(uint2 *)(tile + (size_t)(8 * 64 + i) * 64 + j0) =
                    make_uint2(ptx::pack_bf16(pv[0], pv[1]), ptx::pack_bf16(pv[2], pv[3]));
            }
        } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
#pragma unroll
                for (int w = 0; w < 4; ++w) sh.lx[(i0 + u) * kLdX + j0 + w] = 0.f;
                *(uint2 *)(tile + (size_t)(8 * 64 + i0 + u) * 64 + j0) = make_uint2(0u, 0u);
            }
        }
        khat_qtilde_out(tid, kThreadsKda);
    }
    __syncthreads();  // q is dead: its buffer takes v

    // ---- X = (I + L)^-1 by blocks (FLA page, sec. 4): 8 x 8 forward substitution, exact merges 8 -> 16
    //      (FMA), 16 -> 32 and 32 -> 64 (tf32 m16n8k8) on warps 0-3; warps 4-7 load v, scale k by 2^G and
    //      write g_C meanwhile
    if (tid < 128) {
        const int warp = tid >> 5, lane = tid & 31;
        float *lx = sh.lx;
        auto Lx = [&](int r, int j) -> float { return lx[r * kLdX + j]; };
        auto Xt = [&](int r, int j) -> float { return lx[j * kLdX + r]; };  // X(r, j), j < r
        auto Xm = [&](int r, int j) -> float { return r > j ? lx[j * kLdX + r] : (r == j ? 1.f : 0.f); };
        const int pw = warp;  // 0..3
        // ---- A: the eight 8 x 8 diagonal blocks by forward substitution; 2 threads per (block, column)
        {
            const int task = tid >> 1, hh = tid & 1;
            const int base = 8 * (task >> 3), cc = task & 7;
            float x[8];
    #pragma unroll
            for (int r = 0; r < 8; ++r) x[r] = (r == cc) ? 1.f : 0.f;
    #pragma unroll
            for (int r = 1; r < 8; ++r) {
                float part = 0.f;
    #pragma unroll
                for (int j = 0; j < r; ++j)
                    if ((j & 1) == hh) part = fmaf(Lx(base + r, base + j), x[j], part);
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                if (r > cc) x[r] = -part;
            }
            if (hh == 0) {
    #pragma unroll
                for (int r = 1; r < 8; ++r)
                    if (r > cc) lx[(base + cc) * kLdX + base + r] = x[r];
            }
        }
        bar_sync(1, 128);
        // ---- B: 8 -> 16, one warp per merge:  X(B, A) = -X(B, B) (L(B, A) X(A, A))
        {
            const int A = 16 * pw, Bb = A + 8;
            const int r = lane >> 2, cp = (lane & 3) * 2;
            float t0v = 0.f, t1v = 0.f;
    #pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float l = Lx(Bb + r, A + k);
                const float x0 = k > cp ? Xt(A + k, A + cp) : (k == cp ? 1.f : 0.f);
                const float x1 = k > cp + 1 ? Xt(A + k, A + cp + 1) : (k == cp + 1 ? 1.f : 0.f);
                t0v = fmaf(l, x0, t0v);
                t1v = fmaf(l, x1, t1v);
            }
            float a0 = 0.f, a1 = 0.f;
    #pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float tk0 = __shfl_sync(0xffffffffu, t0v, 4 * k + (lane & 3));
                const float tk1 = __shfl_sync(0xffffffffu, t1v, 4 * k + (lane & 3));
                const float xb = k < r ? Xt(Bb + r, Bb + k) : (k == r ? 1.f : 0.f);
                a0 = fmaf(xb, tk0, a0);
                a1 = fmaf(xb, tk1, a1);
            }
            lx[(A + cp) * kLdX + Bb + r] = -a0;
            lx[(A + cp + 1) * kLdX + Bb + r] = -a1;
        }
        bar_sync(1, 128);
        // ---- C: 16 -> 32 (tf32 m16n8k8); warp = (merge, 8-column tile):
        //      T = L(B, A) X(A, A)[:, tile] (kept transposed where the result goes), then
        //      X(B, A)[:, tile] = -X(B, B) T
        {
            const int g = lane >> 2, t = lane & 3;
            const int A = 32 * (pw >> 1), Bb = A + 16, n0 = 8 * (pw & 1);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
    #pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int k0 = 8 * ks;
                mma_tf32(d, Lx(Bb + g, A + k0 + t), Lx(Bb + g + 8, A + k0 + t), Lx(Bb + g, A + k0 + t + 4),
                         Lx(Bb + g + 8, A + k0 + t + 4), Xm(A + k0 + t, A + n0 + g), Xm(A + k0 + t + 4, A + n0 + g));
            }
            // T^T into this warp's own part of the upper triangle (where X(B, A)[:, tile]^T goes): no other
            // warp reads there, and the B fragments below read it without bank conflicts
            lx[(A + n0 + 2 * t) * kLdX + Bb + g] = d[0];
            lx[(A + n0 + 2 * t + 1) * kLdX + Bb + g] = d[1];
            lx[(A + n0 + 2 * t) * kLdX + Bb + g + 8] = d[2];
            lx[(A + n0 + 2 * t + 1) * kLdX + Bb + g + 8] = d[3];
            __syncwarp();
            float u[4] = {0.f, 0.f, 0.f, 0.f};
    #pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int k0 = 8 * ks;
                mma_tf32(u, Xm(Bb + g, Bb + k0 + t), Xm(Bb + g + 8, Bb + k0 + t), Xm(Bb + g, Bb + k0 + t + 4),
                         Xm(Bb + g + 8, Bb + k0 + t + 4), lx[(A + n0 + g) * kLdX + Bb + k0 + t],
                         lx[(A + n0 + g) * kLdX + Bb + k0 + t + 4]);
            }
            __syncwarp();  // every lane has read T^T
            lx[(A + n0 + 2 * t) * kLdX + Bb + g] = -u[0];
            lx[(A + n0 + 2 * t + 1) * kLdX + Bb + g] = -u[1];
            lx[(A + n0 + 2 * t) * kLdX + Bb + g + 8] = -u[2];
            lx[(A + n0 + 2 * t + 1) * kLdX + Bb + g + 8] = -u[3];
        }
        bar_sync(1, 128);
        // ---- D: 32 -> 64; warp = 8-column tile of the lower-left 32 x 32 block:
        //      T = L(32:64, 0:32) X(0:32, tile) (kept transposed where the result goes), then
        //      X(32:64, tile) = -X(32:64, 32:64) T
        {
            const int g = lane >> 2, t = lane & 3, n0 = 8 * pw;
            float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    #pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                if (ks < pw) continue;  // X(k, n) = 0 for k < n
                const int k0 = 8 * ks;
                const float b0 = Xm(k0 + t, n0 + g), b1 = Xm(k0 + t + 4, n0 + g);
    #pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int m0 = 32 + 16 * mt;
                    mma_tf32(d[mt], Lx(m0 + g, k0 + t), Lx(m0 + g + 8, k0 + t), Lx(m0 + g, k0 + t + 4),
                             Lx(m0 + g + 8, k0 + t + 4), b0, b1);
                }
            }
            // T^T into this warp's own rows of the upper-right block (where X(32:64, tile)^T goes): no other
            // warp reads there, and the B fragments below read it without bank conflicts
    #pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int m0 = 32 + 16 * mt;
                lx[(n0 + 2 * t) * kLdX + m0 + g] = d[mt][0];
                lx[(n0 + 2 * t + 1) * kLdX + m0 + g] = d[mt][1];
                lx[(n0 + 2 * t) * kLdX + m0 + g + 8] = d[mt][2];
                lx[(n0 + 2 * t + 1) * kLdX + m0 + g + 8] = d[mt][3];
            }
            __syncwarp();
            float u[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    #pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const int k0 = 8 * ks;
                const float b0 = lx[(n0 + g) * kLdX + 32 + k0 + t], b1 = lx[(n0 + g) * kLdX + 32 + k0 + t + 4];  // T(k, n)
    #pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    if (k0 > 16 * mt + 15) continue;  // X(32 + m, 32 + k) = 0 for k > m
                    const int m0 = 32 + 16 * mt;
                    mma_tf32(u[mt], Xm(m0 + g, 32 + k0 + t), Xm(m0 + g + 8, 32 + k0 + t), Xm(m0 + g, 32 + k0 + t + 4),
                             Xm(m0 + g + 8, 32 + k0 + t + 4), b0, b1);
                }
            }
            __syncwarp();  // every lane has read T^T
    #pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const int m0 = 32 + 16 * mt;
                lx[(n0 + 2 * t) * kLdX + m0 + g] = -u[mt][0];
                lx[(n0 + 2 * t + 1) * kLdX + m0 + g] = -u[mt][1];
                lx[(n0 + 2 * t) * kLdX + m0 + g + 8] = -u[mt][2];
                lx[(n0 + 2 * t + 1) * kLdX + m0 + g + 8] = -u[mt][3];
            }
        }
    } else {
        // v (bf16) into the q buffer: 16-byte loads, all issued first; meanwhile k -> k 2^G in place (the
        // last use of k and G) and the per-channel chunk decay
        uint4 vv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = tid - 128 + 128 * i, r = e >> 4, c8 = (e & 15) * 8;
            vv[i] = make_uint4(0, 0, 0, 0);
            if (r < rows) vv[i] = *(const uint4 *)(vg + ((size_t)(t0 + r) * HV + hv) * 128 + c8);
        }
        a.gc[((size_t)slot * HV + hv) * 128 + tid - 128] = ex2(sh.gc[tid - 128]);
#pragma unroll 4
        for (int e = tid - 128; e < 64 * 32; e += 128) {
            const int r = e >> 5, c4 = (e & 31) * 4;
            const float4 G4 = *(const float4 *)(sh.g + r * KP + c4);
            const uint2 kk = *(const uint2 *)(sh.k + r * QP + c4);
            const float2 k01 = __bfloat1622float2(*(const __nv_bfloat162 *)&kk.x);
            const float2 k23 = __bfloat1622float2(*(const __nv_bfloat162 *)&kk.y);
            *(uint2 *)(sh.k + r * QP + c4) = make_uint2(ptx::pack_bf16(k01.x * ex2(G4.x), k01.y * ex2(G4.y)),
                                                        ptx::pack_bf16(k23.x * ex2(G4.z), k23.y * ex2(G4.w)));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = tid - 128 + 128 * i, r = e >> 4, c8 = (e & 15) * 8;
            *(uint4 *)(sh.q + r * QP + c8) = vv[i];
        }
    }
    __syncthreads();

    // ---- U = (X diag(beta)) V and -W = -(X diag(beta)) (k 2^G) on the tensor cores (tf32 m16n8k8; the bf16
    //      operands are exact in tf32, X beta is rounded to it): warp = (U or W, 32 output columns) over all
    //      64 rows, so every warp does the same work; a 16-row tile stops at its diagonal (X is lower
    //      triangular)
    // the four output boxes of U and -W are staged in the G buffer (dead now), rounded up to the 1024-byte
    // alignment of the 128-byte swizzle; the buffer has the 1 KB of slack that takes
    uint8_t *stage = (uint8_t *)sh.g + ((1024u - (smem_u32(sh.g) & 1023u)) & 1023u);
    {
        const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
        const int which = warp >> 2, n0 = (warp & 3) * 32;
        const __nv_bfloat16 *src = which ? sh.k : sh.q;  // k 2^G or v, bf16 rows of pitch QP
        auto bf = [](__nv_bfloat16 h) { return __uint_as_float((uint32_t)__bfloat16_as_ushort(h) << 16); };
        auto xb = [&](int r, int j, float be) {  // X(r, j) beta_j, rounded to the nearest tf32
            const float x = j < r ? sh.lx[j * kLdX + r] : (j == r ? 1.f : 0.f);
            return __uint_as_float((__float_as_uint(x * be) + 0x1000u) & 0xffffe000u);
        };
        float acc[4][4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[mt][nt][c] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const int k0 = 8 * ks;
            float b[4][2];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                b[nt][0] = bf(src[(k0 + t) * QP + n0 + 8 * nt + g]);
                b[nt][1] = bf(src[(k0 + t + 4) * QP + n0 + 8 * nt + g]);
            }
            const float be0 = sh.beta[k0 + t], be1 = sh.beta[k0 + t + 4];
#pragma unroll
            for (int mt = ks >> 1; mt < 4; ++mt) {
                const int r = 16 * mt + g;
                const float a0 = xb(r, k0 + t, be0), a1 = xb(r + 8, k0 + t, be0);
                const float a2 = xb(r, k0 + t + 4, be1), a3 = xb(r + 8, k0 + t + 4, be1);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) mma_tf32(acc[mt][nt], a0, a1, a2, a3, b[nt][0], b[nt][1]);
            }
        }
        // into four 128-byte-swizzled staging boxes (U dv 0-63, U dv 64-127, -W dk 0-63, -W dk 64-127) in
        // the dead G buffer: a fragment store's eight rows hit eight different 16-byte columns (no conflicts)
        const float sgn = which ? -1.f : 1.f;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int r = 16 * mt + g, col = n0 + 8 * nt + 2 * t;
                uint8_t *bx = stage + (2 * which + (col >> 6)) * 8192 + (col & 7) * 2;
                const uint32_t sw = (uint32_t)((((col & 63) >> 3) ^ (r & 7)) << 4);  // (r + 8) & 7 == r & 7
                *(uint32_t *)(bx + r * 128 + sw) = ptx::pack_bf16(sgn * acc[mt][nt][0], sgn * acc[mt][nt][1]);
                *(uint32_t *)(bx + (r + 8) * 128 + sw) = ptx::pack_bf16(sgn * acc[mt][nt][2], sgn * acc[mt][nt][3]);
            }
    }
    fence_proxy_async();  // the boxes leave through TMA stores
    __syncthreads();
    if (tid == 0) {
        const int row0 = (int)((((size_t)slot * HV + hv) * 9 + 4) * 64);
#pragma unroll
        for (int b = 0; b < 4; ++b) tma_store_2d(&tmap, stage + b * 8192, 0, row0 + 64 * b);
        tma_store_commit();
        tma_store_wait_read0();  // the boxes stay valid until the copies have read them
    }
}

}  // namespace

size_t kda_prep_smem_bytes() { return sizeof(KdaSmem); }

cudaError_t launch_kda_prep(const KdaPrepArgs &a, cudaStream_t st)
{
    if (a.N * a.HV == 0 || a.slots == 0) return cudaSuccess;
    const int smem = (int)sizeof(KdaSmem);
    cudaError_t e = cudaFuncSetAttribute(kda_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // two CTAs per SM need the largest shared-memory carveout
    e = cudaFuncSetAttribute(kda_prep_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    dim3 grid(a.slots, a.HV);
    // U and -W leave through TMA stores (2-D map over the tiles, 64-row boxes)
    alignas(64) CUtensorMap tmap;
    if (!encode_tiles_map(&tmap, a.tiles, (int64_t)a.slots * a.HV * 576, 64)) return cudaErrorInvalidValue;
    kda_prep_kernel<<<grid, kThreadsKda, smem, st>>>(a, tmap);
    return cudaGetLastError();
}

}  // namespace gdn

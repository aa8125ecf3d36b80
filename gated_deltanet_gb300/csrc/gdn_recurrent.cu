// Token-by-token (recurrent) engine of the gated delta rule, for decode and
// short continuations: the "Flash Linear Attention" page, sec. 8
// (fused_recurrent, the C = 1 form that the layer selects for short queries),
// with the delta-rule update of the FlashQLA blog ("Further optimisation via
// gate decay", the recurrence):
//
//   S <- Diag(alpha_t) S                      alpha_t = exp(g_t) (scalar) or exp(gk_t) per key channel
//   u <- S^T k_t                              read-out of the decayed state
//   S <- S + k_t (beta_t (v_t - u))^T         delta-rule write
//   o_t = scale * S^T q_t                     output of the updated state
//
// No chunking, no intermediate state in memory: the state tile is loaded once,
// updated for every token of the sequence and written back once (in place is
// allowed: every CTA reads its whole tile before it writes it).  Bound by the
// state's traffic (8 K V bytes per (sequence, head)) for short sequences.
//
// One CTA (128 threads) per (sequence, value head, 32-column value tile).
// Lane = value column, warp w = key rows [w K/4, (w+1) K/4): the state rows
// are read and written as 128-byte coalesced segments, the two contractions
// over the key dimension per token are a per-thread sum plus a four-way
// reduction through shared memory.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRecThreads = 128;
constexpr int kRecBV = 32;

template <typename T>
__device__ __forceinline__ float ldf(const T *p) { return (float)*p; }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void stf(T *p, float x) { *p = x; }
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

template <typename T, int KD, bool CHANNEL>
__global__ void __launch_bounds__(kRecThreads) recurrent_kernel(const RecArgs a)
{
    constexpr int RPW = KD / 4;  // key rows per warp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int HV = a.HV, V = a.V, nvt = (V + kRecBV - 1) / kRecBV;
    // one-dimensional grid (no 65535 limit on the sequence count): x = (n HV + hv) nvt + vt
    const int vt = (int)(blockIdx.x % nvt), hv = (int)((blockIdx.x / nvt) % HV), n = (int)(blockIdx.x / ((unsigned)nvt * HV));
    const int hq = hv / (HV / a.H);
    const int v = vt * kRecBV + lane;
    const bool vok = v < V;
    int64_t bos, len;
    if (a.cu_seqlens) {
        bos = a.cu_seqlens[n];
        len = a.cu_seqlens[n + 1] - bos;
    } else {
        bos = (int64_t)n * a.T;
        len = a.T;
    }
    __shared__ float s_kq[2][2][KD];     // [token parity][k, scale q][key dim]
    __shared__ float s_gk[2][CHANNEL ? KD : 1];
    __shared__ float s_red[2][4][kRecBV];  // [u, o][warp][column]
    __shared__ float s_gb[2][2];           // [token parity][alpha, beta]
    __shared__ float s_nrm[2][2][4];       // [token parity][k, q][warp]: partial sums of squares

    const size_t sbase = ((size_t)n * HV + hv) * KD * V;
    float s[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) s[i] = (a.h0 && vok) ? a.h0[sbase + (size_t)(warp * RPW + i) * V + v] : 0.f;

    const T *q = (const T *)a.q, *k = (const T *)a.k, *vv = (const T *)a.v;
    T *o = (T *)a.o;
    // stage token t's k, scale * q and gates into buffer t & 1
    auto stage = [&](int64_t t) {
        const int b = (int)(t & 1);
        const size_t tok = (size_t)(bos + t);
        // KD <= kRecThreads: at most one key-dimension element per thread
        float kx = 0.f, qx = 0.f;
        if (threadIdx.x < KD) {
            const int i = threadIdx.x;
            kx = ldf(k + (tok * a.H + hq) * KD + i);
            qx = ldf(q + (tok * a.H + hq) * KD + i);
            s_kq[b][0][i] = kx;
            s_kq[b][1][i] = a.scale * qx;
            if constexpr (CHANNEL) s_gk[b][i] = expf(act_gate(a.act, a.g[(tok * HV + hv) * KD + i], hv, i, KD));
        }
        if (a.act.qk_l2norm) {
            // in-kernel L2 norm: per-warp sums of squares, combined by the readers
            float sk = kx * kx, sq = qx * qx;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
            }
            if (lane == 0) {
                s_nrm[b][0][warp] = sk;
                s_nrm[b][1][warp] = sq;
            }
        }
        if (threadIdx.x == 0) {
            if constexpr (!CHANNEL) s_gb[b][0] = expf(act_gate(a.act, a.g[tok * HV + hv], hv, -1, KD));
            s_gb[b][1] = act_beta(a.act, a.beta[tok * HV + hv]);
        }
    };
    if (len > 0) stage(0);
    for (int64_t t = 0; t < len; ++t) {
        const int b = (int)(t & 1);
        const size_t tok = (size_t)(bos + t);
        const float vval = vok ? ldf(vv + (tok * HV + hv) * V + v) : 0.f;
        __syncthreads();  // token t staged; the reductions of token t - 1 are read
        // 1 / ||k_t||, 1 / ||q_t|| of the in-kernel L2 norm (1 otherwise)
        float rk = 1.f, rq = 1.f;
        if (a.act.qk_l2norm) {
            rk = 1.f / fmaxf(sqrtf(s_nrm[b][0][0] + s_nrm[b][0][1] + s_nrm[b][0][2] + s_nrm[b][0][3]), kNormEps);
            rq = 1.f / fmaxf(sqrtf(s_nrm[b][1][0] + s_nrm[b][1][1] + s_nrm[b][1][2] + s_nrm[b][1][3]), kNormEps);
        }
        if (t + 1 < len) stage(t + 1);
        // decay, then the read-out of the decayed state
        float u = 0.f;
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const int r = warp * RPW + i;
            s[i] *= CHANNEL ? s_gk[b][r] : s_gb[b][0];
            u = fmaf(s_kq[b][0][r], s[i], u);
        }
        s_red[0][warp][lane] = u;
        __syncthreads();
        u = rk * (s_red[0][0][lane] + s_red[0][1][lane] + s_red[0][2][lane] + s_red[0][3][lane]);
        const float delta = rk * s_gb[b][1] * (vval - u);  // the write uses k / ||k|| too
        float ov = 0.f;
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const int r = warp * RPW + i;
            s[i] = fmaf(s_kq[b][0][r], delta, s[i]);
            ov = fmaf(s_kq[b][1][r], s[i], ov);
        }
        s_red[1][warp][lane] = ov;
        __syncthreads();
        if (warp == 0 && vok)
            stf(o + (tok * HV + hv) * V + v,
                rq * (s_red[1][0][lane] + s_red[1][1][lane] + s_red[1][2][lane] + s_red[1][3][lane]));
    }
    if (a.ht && vok) {
#pragma unroll
        for (int i = 0; i < RPW; ++i) a.ht[sbase + (size_t)(warp * RPW + i) * V + v] = s[i];
    }
}

template <typename T, int KD>
cudaError_t launch_k(const RecArgs &a, bool channel, cudaStream_t st)
{
    const unsigned long long ctas = (unsigned long long)((a.V + kRecBV - 1) / kRecBV) * a.HV * a.N;
    if (ctas >= (1ull << 31)) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)ctas);
    if (channel) recurrent_kernel<T, KD, true><<<grid, kRecThreads, 0, st>>>(a);
    else recurrent_kernel<T, KD, false><<<grid, kRecThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const RecArgs &a, bool channel, cudaStream_t st)
{
    switch (a.K) {
    case 32: return launch_k<T, 32>(a, channel, st);
    case 64: return launch_k<T, 64>(a, channel, st);
    case 128: return launch_k<T, 128>(a, channel, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_recurrent(const RecArgs &a, gdn_dtype dt, gdn_gate_kind gate, cudaStream_t st)
{
    if (a.N == 0 || a.HV == 0 || a.V == 0) return cudaSuccess;
    const bool channel = gate == GDN_GATE_CHANNEL;
    return dt == GDN_BF16 ? launch_t<__nv_bfloat16>(a, channel, st) : launch_t<float>(a, channel, st);
}

}  // namespace gdn

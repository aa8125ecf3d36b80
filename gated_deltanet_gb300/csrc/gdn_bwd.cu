// Backward pass of the chunked gated delta rule (scalar gates): the gradients of o and of the final
// state with respect to q, k, v, beta, g and h0.  The method is the chunked backward of the GDN-in-FLA
// notes (backward, Steps 1-7) with the state gradient scanned in reverse time ("Flash Linear
// Attention" page, sec. 7).  With G the chunk-local inclusive log-gate cumsum, gam = exp(G),
// Gam_ij = exp(G_i - G_j), L = StrictLower(diag(beta) Gam * K K^T), A = (I + L)^-1,
// P = scale Lower(Gam) * Q K^T and S0 the state entering the chunk:
//
//   R   = V - diag(gam) K S0,   B = diag(beta) R,   D = A B            (D: the chunk's v_new)
//   dD  = P^T dO + diag(gam_C / gam) K dS                                             (Steps 3-4)
//   dS0 = gam_C dS + scale Q^T diag(gam) dO - K^T diag(gam) dR,   dR = diag(beta) A^T dD  (Step 4)
//   dq  = scale diag(gam) dO S0^T + F K,  F = scale Lower(Gam) * (dO D^T)                 (Step 5)
//   dk  = F^T Q + diag(gam_C / gam) D dS^T - diag(gam) dR S0^T + E K + E^T K,           (Steps 5-6)
//         E = StrictLower(diag(beta) Gam * dL),  dL = -A^T (dD B^T) A^T
//   dv  = dR,  dbeta = rowsum((A^T dD) * R) + rowsum(dL * Gam * K K^T)                  (Step 6)
//   dG  = the derivative with respect to each G_i of every factor exp(G) above         (Steps 5-6)
//   dg  = the suffix sum of dG within each chunk (Step 7); dh0 = the last dS.
//
// Kernels, after the chunk states are recomputed by a forward pass with a state dump (Step 2):
//   bwd_prep_kernel     one CTA per chunk and value head: A and P (Step 1: nothing in them depends on
//                       the state; A by forward substitution per column), fp32 into the workspace;
//   chunk_bwd_kernel    one CTA per (sequence, value head, 32-column value tile), chunks newest first
//                       with its tile of dS in shared memory: everything that needs S0 or dS, and the
//                       tile's parts of dO D^T and dD B^T (sums over the value columns) to the workspace;
//   bwd_finish_kernel   one CTA per chunk and value head: the tiles' parts summed, F, dL, E and their
//                       products with K and Q, the gate and beta terms of P and L;
//   gate_suffix_kernel  Step 7.
// dq, dk, dbeta and dG are sums over value tiles and kernels (and dq, dk over a GVA group's value
// heads): fp32 atomic adds into buffers the host zeroes.  The shared-memory products run on the tensor
// cores in split tf32 (about fp32 accuracy; the remainder terms of bf16 inputs, exact in tf32, left out), and
// so do the row tiles of dq and dk, kept in accumulator fragments; the rest runs on CUDA cores in fp32.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kBThreads = 256;  // the A and P kernel (two CTAs per SM)
constexpr int kRThreads = 512;  // the reverse scan and the finish (sixteen warps: a product block per warp)
constexpr int kBC = 64;      // chunk
constexpr int kBV = 32;      // value columns per CTA
constexpr int kCP = kBC + 4;  // pitches (4 mod 32: the tensor-core fragments' strided reads hit at most
constexpr int kVP = kBV + 4;  // two lanes per bank)

template <int K>
struct BwdLayout {  // the reverse kernel
    static constexpr int KP = K + 4;
    static constexpr int oK = 0, oQ = oK + kBC * KP, oS0 = oQ + kBC * KP, odS = oS0 + K * kVP,
                         oV = odS + K * kVP, odO = oV + kBC * kVP, oR = odO + kBC * kVP, oD = oR + kBC * kVP,
                         odD = oD + kBC * kVP, oY = odD + kBC * kVP, oA = oY + kBC * kVP, oP = oA + kBC * kCP,
                         oM2 = oP + kBC * kCP, oG = oM2 + kBC * kCP, oGam = oG + kBC, oBeta = oGam + kBC,
                         odG = oBeta + kBC, odB = odG + kBC, oRed = odB + kBC, total = oRed + 12 * kBC;
};
template <int K>
struct PrepLayout {  // A and P of a chunk (two CTAs per SM at K = 128)
    static constexpr int KP = K + 4;
    static constexpr int oK = 0, oQ = oK + kBC * KP, oA = oQ + kBC * KP, oP = oA + kBC * kCP, oG = oP + kBC * kCP,
                         oBeta = oG + kBC, oRed = oBeta + kBC, total = oRed + 4 * kBC;
};
template <int K>
struct ChunkLayout {  // the finish
    static constexpr int KP = K + 4;
    static constexpr int oK = 0, oQ = oK + kBC * KP, oA = oQ + kBC * KP, oP = oA + kBC * kCP, odP = oP + kBC * kCP,
                         odA = odP + kBC * kCP, oT = odA + kBC * kCP, oG = oT + kBC * kCP, oBeta = oG + kBC,
                         oRed = oBeta + kBC, total = oRed + 4 * kBC;
};

template <typename T>
__device__ __forceinline__ float ldf(const T *p) { return (float)*p; }
// eight consecutive elements as fp32 (one 16-byte load for bf16, two for fp32; p 16-byte aligned), and
// eight fp32 into shared memory (p 16-byte aligned)
__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float (&f)[8])
{
    const uint4 u = __ldg((const uint4 *)p);
    const __nv_bfloat162 *h = (const __nv_bfloat162 *)&u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 x = __bfloat1622float2(h[q]);
        f[2 * q] = x.x;
        f[2 * q + 1] = x.y;
    }
}
__device__ __forceinline__ void ld8(const float *p, float (&f)[8])
{
    const float4 x = __ldg((const float4 *)p), y = __ldg((const float4 *)p + 1);
    f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
    f[4] = y.x; f[5] = y.y; f[6] = y.z; f[7] = y.w;
}
__device__ __forceinline__ void st8(float *p, const float (&f)[8])
{
    *(float4 *)p = make_float4(f[0], f[1], f[2], f[3]);
    *(float4 *)(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}
// bf16 inputs (k, q, v, dO) are exact in tf32: their products need no remainder term
template <typename T>
constexpr bool kExactOf = false;
template <>
constexpr bool kExactOf<__nv_bfloat16> = true;
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// Shared-memory products: out[m][n] = alpha * sum_x A(m, x) xs[x] B(x, n) (+ out when acc), with
// A(m, x) = a[x lda + m] if TA else a[m lda + x], B(x, n) = b[n ldb + x] if TB else b[x ldb + n], xs optional.
__device__ __forceinline__ uint32_t tf32_of(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32x(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// On the tensor cores (mma.sync m16n8k8, tf32): each operand is split into a tf32
// part and the tf32 rounding of its remainder, and hi*hi + hi*lo + lo*hi keeps the product to about fp32
// accuracy.  An operand that is exact in tf32 (EA, EB: bf16 inputs, unscaled) has no remainder, and its
// term is left out.  A warp takes 16 x (8 NB) output blocks, NB tiles side by side sharing the A fragment
// (NB independent accumulations in flight); M a multiple of 16, N of 8 NB, X of 8.  xs scales the
// contraction index on A's side, or on B's with XB (so that the other operand stays exact).
template <bool TA, bool TB, int NB, bool EA = false, bool EB = false, bool XB = false, int NTH = kBThreads>
__device__ void tmm(float *out, int ldo, const float *a, int lda, const float *b, int ldb, int M, int N, int X,
                    float alpha, bool acc, const float *xs = nullptr)
{
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
    const int bn = N / (8 * NB), blocks = (M / 16) * bn;
    for (int blk = w; blk < blocks; blk += NTH / 32) {
        const int m0 = (blk / bn) * 16, n0 = (blk % bn) * 8 * NB;
        float d[NB][4];
#pragma unroll
        for (int j = 0; j < NB; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
#pragma unroll 2
        for (int x0 = 0; x0 < X; x0 += 8) {
            const int xa = x0 + t, xb = x0 + t + 4;
            const float sa = xs ? xs[xa] : 1.f, sb = xs ? xs[xb] : 1.f;
            const float fa = XB ? 1.f : sa, fb = XB ? 1.f : sb, ga = XB ? sa : 1.f, gb = XB ? sb : 1.f;
            const float av[4] = {
                fa * (TA ? a[xa * lda + m0 + g] : a[(m0 + g) * lda + xa]),
                fa * (TA ? a[xa * lda + m0 + g + 8] : a[(m0 + g + 8) * lda + xa]),
                fb * (TA ? a[xb * lda + m0 + g] : a[(m0 + g) * lda + xb]),
                fb * (TA ? a[xb * lda + m0 + g + 8] : a[(m0 + g + 8) * lda + xb])};
            uint32_t ah[4], al[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ah[i] = tf32_of(av[i]);
                al[i] = EA ? 0u : tf32_of(av[i] - __uint_as_float(ah[i]));
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                const int nn = n0 + 8 * j + g;
                const float bv0 = ga * (TB ? b[nn * ldb + xa] : b[xa * ldb + nn]);
                const float bv1 = gb * (TB ? b[nn * ldb + xb] : b[xb * ldb + nn]);
                const uint32_t bh0 = tf32_of(bv0), bh1 = tf32_of(bv1);
                if (!EA) mma_tf32x(d[j], al, bh0, bh1);
                if (!EB) {
                    const uint32_t bl0 = tf32_of(bv0 - __uint_as_float(bh0)), bl1 = tf32_of(bv1 - __uint_as_float(bh1));
                    mma_tf32x(d[j], ah, bl0, bl1);
                }
                mma_tf32x(d[j], ah, bh0, bh1);
            }
        }
#pragma unroll
        for (int j = 0; j < NB; ++j) {
            float *o0 = out + (m0 + g) * ldo + n0 + 8 * j + 2 * t, *o1 = o0 + 8 * ldo;
            if (acc) {
                o0[0] = fmaf(alpha, d[j][0], o0[0]);
                o0[1] = fmaf(alpha, d[j][1], o0[1]);
                o1[0] = fmaf(alpha, d[j][2], o1[0]);
                o1[1] = fmaf(alpha, d[j][3], o1[1]);
            } else {
                o0[0] = alpha * d[j][0];
                o0[1] = alpha * d[j][1];
                o1[0] = alpha * d[j][2];
                o1[1] = alpha * d[j][3];
            }
        }
    }
}

// A [kBC x K] tile in tensor-core accumulator fragments over NTH threads: the warps form 4 row groups x
// NTH / 128 column parts; warp w holds rows 16 (w & 3) .. + 15 and the K / parts columns of part w >> 2
// as NT = K * 16 / NTH blocks of m16n8; thread (g = lane / 4, t = lane % 4) holds, in block j, rows
// r = 16 (w & 3) + g and r + 8 at columns c = (part start) + 8 j + 2 t and c + 1.
// facc: acc[m][n] += alpha * rs[m] * sum_x A(m, x) B(x, n) (rs optional), split tf32 as in tmm, X a
// multiple of 8.
template <int K, int NTH>
constexpr int kFragNT = K * 16 / NTH;
template <int K, bool TA, bool TB, bool EA = false, bool EB = false, int NTH = kBThreads>
__device__ void facc(float (&acc)[kFragNT<K, NTH>][4], const float *a, int lda, const float *b, int ldb, int X,
                     float alpha = 1.f, const float *rs = nullptr)
{
    constexpr int NT = kFragNT<K, NTH>;
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
    const int m0 = 16 * (w & 3), n0 = 8 * NT * (w >> 2);
    float d[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
#pragma unroll 2
    for (int x0 = 0; x0 < X; x0 += 8) {
        const int xa = x0 + t, xb = x0 + t + 4;
        const float av[4] = {TA ? a[xa * lda + m0 + g] : a[(m0 + g) * lda + xa],
                             TA ? a[xa * lda + m0 + g + 8] : a[(m0 + g + 8) * lda + xa],
                             TA ? a[xb * lda + m0 + g] : a[(m0 + g) * lda + xb],
                             TA ? a[xb * lda + m0 + g + 8] : a[(m0 + g + 8) * lda + xb]};
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ah[i] = tf32_of(av[i]);
            al[i] = EA ? 0u : tf32_of(av[i] - __uint_as_float(ah[i]));
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int nn = n0 + 8 * j + g;
            const float bv0 = TB ? b[nn * ldb + xa] : b[xa * ldb + nn];
            const float bv1 = TB ? b[nn * ldb + xb] : b[xb * ldb + nn];
            const uint32_t bh0 = tf32_of(bv0), bh1 = tf32_of(bv1);
            if (!EA) mma_tf32x(d[j], al, bh0, bh1);
            if (!EB) {
                const uint32_t bl0 = tf32_of(bv0 - __uint_as_float(bh0)), bl1 = tf32_of(bv1 - __uint_as_float(bh1));
                mma_tf32x(d[j], ah, bl0, bl1);
            }
            mma_tf32x(d[j], ah, bh0, bh1);
        }
    }
    const float f0 = alpha * (rs ? rs[m0 + g] : 1.f), f1 = alpha * (rs ? rs[m0 + g + 8] : 1.f);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        acc[j][0] = fmaf(f0, d[j][0], acc[j][0]);
        acc[j][1] = fmaf(f0, d[j][1], acc[j][1]);
        acc[j][2] = fmaf(f1, d[j][2], acc[j][2]);
        acc[j][3] = fmaf(f1, d[j][3], acc[j][3]);
    }
}

// the warp's part of the row dot products of a fragment tile with a [kBC x K] shared-memory matrix (pitch
// ld) over its columns: out[0] for row 16 (w & 3) + g, out[1] for that + 8, on every lane of the quad
template <int K, int NTH = kBThreads>
__device__ void frdot(const float (&acc)[kFragNT<K, NTH>][4], const float *m, int ld, float (&out)[2])
{
    constexpr int NT = kFragNT<K, NTH>;
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
    const int r0 = 16 * (w & 3) + g, n0 = 8 * NT * (w >> 2);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int c = n0 + 8 * j + 2 * t;
        s0 = fmaf(acc[j][0], m[r0 * ld + c], fmaf(acc[j][1], m[r0 * ld + c + 1], s0));
        s1 = fmaf(acc[j][2], m[(r0 + 8) * ld + c], fmaf(acc[j][3], m[(r0 + 8) * ld + c + 1], s1));
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    out[0] = s0;
    out[1] = s1;
}

// fragment tiles dq, dk into the fp32 sums of rows t0 + r (r < rows) of [T, H, K] tensors (head hq): four
// columns by one 16-byte atomic add
template <int K, int NTH = kBThreads>
__device__ void fatomic_rows(const float (&dq)[kFragNT<K, NTH>][4], const float (&dk)[kFragNT<K, NTH>][4],
                             float *gq, float *gk, int64_t t0, int rows, int H, int hq)
{
    constexpr int NT = kFragNT<K, NTH>;
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, g = l >> 2, t = l & 3;
    const int n0 = 8 * NT * (w >> 2);
    // lanes t and t ^ 1 trade halves: the even one gathers four columns of row r0 = 16 (w & 3) + g, the odd
    // one four columns of r0 + 8, and each adds them by one 16-byte atomic
    const bool odd = t & 1;
    const int i = 16 * (w & 3) + g + (odd ? 8 : 0);
    const bool live = i < rows;
    float *pq = gq + ((size_t)(t0 + i) * H + hq) * K, *pk = gk + ((size_t)(t0 + i) * H + hq) * K;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const float q0 = __shfl_xor_sync(0xffffffffu, odd ? dq[j][0] : dq[j][2], 1);
        const float q1 = __shfl_xor_sync(0xffffffffu, odd ? dq[j][1] : dq[j][3], 1);
        const float k0 = __shfl_xor_sync(0xffffffffu, odd ? dk[j][0] : dk[j][2], 1);
        const float k1 = __shfl_xor_sync(0xffffffffu, odd ? dk[j][1] : dk[j][3], 1);
        const int c = n0 + 8 * j + 4 * (t >> 1);
        if (live) {
            atomicAdd((float4 *)(pq + c), odd ? make_float4(q0, q1, dq[j][2], dq[j][3]) : make_float4(dq[j][0], dq[j][1], q0, q1));
            atomicAdd((float4 *)(pk + c), odd ? make_float4(k0, k1, dk[j][2], dk[j][3]) : make_float4(dk[j][0], dk[j][1], k0, k1));
        }
    }
}

// The chunk (sequence n, value head hv, chunk c): k, q rows (zero past the sequence end), the
// inclusive log-gate cumsum G and beta.  Every thread of the CTA takes part; returns the rows.
template <typename DT, int K, int NTH = kBThreads>
__device__ int load_chunk(const BwdArgs &a, int64_t bos, int64_t len, int c, int hv, float *sK, float *sQ,
                          float *sG, float *sGam, float *sBeta)
{
    constexpr int KP = K + 4;
    const int HV = a.HV, hq = hv / (HV / a.H);
    const int64_t t0 = bos + (int64_t)c * kBC;
    const int rows = (int)min((int64_t)kBC, len - (int64_t)c * kBC);
    const DT *q = (const DT *)a.q, *k = (const DT *)a.k;
    constexpr int P8 = K / 8;  // eight-element pieces of a row (rows are K * sizeof(DT) >= 64 bytes)
#pragma unroll 4
    for (int e = threadIdx.x; e < kBC * P8; e += NTH) {
        const int i = e / P8, d8 = (e - i * P8) * 8;
        float kv[8], qv[8];
        if (i < rows) {
            const size_t off = ((size_t)(t0 + i) * a.H + hq) * K + d8;
            ld8(k + off, kv);
            ld8(q + off, qv);
        } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) kv[u] = qv[u] = 0.f;
        }
        st8(sK + i * KP + d8, kv);
        st8(sQ + i * KP + d8, qv);
    }
    if (threadIdx.x < 32) {
        const int l = threadIdx.x, r0 = 2 * l, r1 = r0 + 1;
        const float g0 = r0 < rows ? a.g[(size_t)(t0 + r0) * HV + hv] : 0.f;
        const float g1 = r1 < rows ? a.g[(size_t)(t0 + r1) * HV + hv] : 0.f;
        float sp = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, sp, off);
            if (l >= off) sp += y;
        }
        sG[r0] = sp - g1;
        sG[r1] = sp;
        if (sGam) {
            sGam[r0] = __expf(sp - g1);
            sGam[r1] = __expf(sp);
        }
        sBeta[r0] = r0 < rows ? a.beta[(size_t)(t0 + r0) * HV + hv] : 0.f;
        sBeta[r1] = r1 < rows ? a.beta[(size_t)(t0 + r1) * HV + hv] : 0.f;
    }
    return rows;
}

// One reverse step's inputs with every global load issued before the first shared-memory store (one
// memory round trip): the chunk's k, q rows and gates, the value tile's v and dO columns and state rows,
// A and P.  V a multiple of 8.  Returns the rows.
template <typename DT, int K>
__device__ int load_step(const BwdArgs &a, int64_t bos, int64_t len, int c, int hv, int col0, size_t cidx,
                         float *sK, float *sQ, float *sG, float *sGam, float *sBeta, float *sV, float *sdO,
                         float *sS0, float *sA, float *sP)
{
    constexpr int KP = K + 4, P8 = K / 8, NTH = kRThreads;
    constexpr int KQI = (kBC * P8 + NTH - 1) / NTH, VI = (kBC * (kBV / 8) + NTH - 1) / NTH,
                  SI = (K * (kBV / 4) + NTH - 1) / NTH, AI = (kBC * kBC / 4 + NTH - 1) / NTH;
    const int tid = threadIdx.x, HV = a.HV, V = a.V, hq = hv / (HV / a.H);
    const int64_t t0 = bos + (int64_t)c * kBC;
    const int rows = (int)min((int64_t)kBC, len - (int64_t)c * kBC);
    const DT *q = (const DT *)a.q, *k = (const DT *)a.k, *v = (const DT *)a.v, *dout = (const DT *)a.dout;
    float kv[KQI][8], qv[KQI][8], vv[VI][8], dv[VI][8];
    float4 s4[SI], a4[AI], p4[AI];
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < KQI; ++u) {
        const int e = tid + u * NTH, i = e / P8, d8 = (e % P8) * 8;
        if (e < kBC * P8 && i < rows) {
            const size_t off = ((size_t)(t0 + i) * a.H + hq) * K + d8;
            ld8(k + off, kv[u]);
            ld8(q + off, qv[u]);
        } else {
#pragma unroll
            for (int x = 0; x < 8; ++x) kv[u][x] = qv[u][x] = 0.f;
        }
    }
#pragma unroll
    for (int u = 0; u < VI; ++u) {
        const int e = tid + u * NTH, i = e / (kBV / 8), j = (e % (kBV / 8)) * 8, col = col0 + j;
        if (e < kBC * (kBV / 8) && i < rows && col < V) {
            const size_t off = ((size_t)(t0 + i) * HV + hv) * V + col;
            ld8(v + off, vv[u]);
            ld8(dout + off, dv[u]);
        } else {
#pragma unroll
            for (int x = 0; x < 8; ++x) vv[u][x] = dv[u][x] = 0.f;
        }
    }
    const float *src = a.chunk_states + cidx * K * V;
#pragma unroll
    for (int u = 0; u < SI; ++u) {
        const int e = tid + u * NTH, d = e / (kBV / 4), j = (e % (kBV / 4)) * 4, col = col0 + j;
        s4[u] = (e < K * (kBV / 4) && col < V) ? __ldg((const float4 *)(src + (size_t)d * V + col)) : z4;
    }
    const float4 *ga = (const float4 *)(a.Abuf + cidx * kBC * kBC), *gp = (const float4 *)(a.Pbuf + cidx * kBC * kBC);
#pragma unroll
    for (int u = 0; u < AI; ++u) {
        const int e = tid + u * NTH;
        a4[u] = e < kBC * kBC / 4 ? __ldg(ga + e) : z4;
        p4[u] = e < kBC * kBC / 4 ? __ldg(gp + e) : z4;
    }
    float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
    const int l = tid & 31, r0 = 2 * l, r1 = r0 + 1;
    if (tid < 32) {
        if (r0 < rows) {
            g0 = a.g[(size_t)(t0 + r0) * HV + hv];
            b0 = a.beta[(size_t)(t0 + r0) * HV + hv];
        }
        if (r1 < rows) {
            g1 = a.g[(size_t)(t0 + r1) * HV + hv];
            b1 = a.beta[(size_t)(t0 + r1) * HV + hv];
        }
    }
    // ---- stores
#pragma unroll
    for (int u = 0; u < KQI; ++u) {
        const int e = tid + u * NTH, i = e / P8, d8 = (e % P8) * 8;
        if (e < kBC * P8) {
            st8(sK + i * KP + d8, kv[u]);
            st8(sQ + i * KP + d8, qv[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < VI; ++u) {
        const int e = tid + u * NTH, i = e / (kBV / 8), j = (e % (kBV / 8)) * 8;
        if (e < kBC * (kBV / 8)) {
            st8(sV + i * kVP + j, vv[u]);
            st8(sdO + i * kVP + j, dv[u]);
        }
    }
#pragma unroll
    for (int u = 0; u < SI; ++u) {
        const int e = tid + u * NTH, d = e / (kBV / 4), j = (e % (kBV / 4)) * 4;
        if (e < K * (kBV / 4)) *(float4 *)(sS0 + d * kVP + j) = s4[u];
    }
#pragma unroll
    for (int u = 0; u < AI; ++u) {
        const int e = tid + u * NTH, i = e / (kBC / 4), j = (e % (kBC / 4)) * 4;
        if (e < kBC * kBC / 4) {
            *(float4 *)(sA + i * kCP + j) = a4[u];
            *(float4 *)(sP + i * kCP + j) = p4[u];
        }
    }
    if (tid < 32) {
        float sp = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, sp, off);
            if (l >= off) sp += y;
        }
        sG[r0] = sp - g1;
        sG[r1] = sp;
        sGam[r0] = __expf(sp - g1);
        sGam[r1] = __expf(sp);
        sBeta[r0] = b0;
        sBeta[r1] = b1;
    }
    return rows;
}

// A = (I + L)^-1 in place (sA holds L below the diagonal, zero elsewhere) by forward substitution per
// column: column j solves x_i = [i == j] - sum_{k < i} L_ik x_k.  Four threads share a column, thread p
// keeping x_k for k = p mod 4 and summing those terms; the four partial sums meet by shuffles, so no
// barrier runs between rows.
__device__ void unit_lower_inverse(float *sA)
{
    const int tid = threadIdx.x, j = tid >> 2, p = tid & 3;
    float xq[kBC / 4];  // x_{4 q + p}
#pragma unroll
    for (int q = 0; q < kBC / 4; ++q) xq[q] = 0.f;
#pragma unroll
    for (int i = 0; i < kBC; ++i) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int q = 0; q < kBC / 4; ++q) {
            if (4 * q + 3 < i || 4 * q + p < i) {  // (the first test is constant: the full groups)
                const float v = sA[i * kCP + 4 * q + p] * xq[q];
                if (q & 1) s1 += v; else s0 += v;
            }
        }
        float sum = s0 + s1;
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (p == (i & 3)) xq[i >> 2] = (i == j ? 1.f : 0.f) - sum;
    }
    __syncthreads();  // every thread has read L
#pragma unroll
    for (int q = 0; q < kBC / 4; ++q) sA[(4 * q + p) * kCP + j] = xq[q];
    __syncthreads();
}

// (sequence, value head, chunk) of a per-chunk CTA: blockIdx.x = chunk, blockIdx.y = pair
__device__ bool chunk_of_block(const BwdArgs &a, int &n, int &hv, int &c, int64_t &bos, int64_t &len)
{
    c = blockIdx.x;
    const int pair = blockIdx.y;
    n = pair / a.HV;
    hv = pair % a.HV;
    bos = a.cu_seqlens ? a.cu_seqlens[n] : (int64_t)n * a.T;
    len = a.cu_seqlens ? a.cu_seqlens[n + 1] - bos : a.T;
    return (int64_t)c * kBC < len;
}

// ---- Step 1: A and P of every chunk
template <typename DT, int K>
__global__ void __launch_bounds__(kBThreads, 2) bwd_prep_kernel(const BwdArgs a)
{
    using Lay = PrepLayout<K>;
    constexpr int KP = Lay::KP;
    extern __shared__ float smem[];
    float *sK = smem + Lay::oK, *sQ = smem + Lay::oQ, *sA = smem + Lay::oA, *sP = smem + Lay::oP;
    float *sG = smem + Lay::oG, *sBeta = smem + Lay::oBeta, *sRed = smem + Lay::oRed;
    int n, hv, c;
    int64_t bos, len;
    if (!chunk_of_block(a, n, hv, c, bos, len)) return;
    load_chunk<DT, K>(a, bos, len, c, hv, sK, sQ, sG, nullptr, sBeta);
    __syncthreads();
    constexpr bool EX = kExactOf<DT>;
    tmm<false, true, 4, EX, EX>(sA, kCP, sK, KP, sK, KP, kBC, kBC, K, 1.f, false);
    tmm<false, true, 4, EX, EX>(sP, kCP, sQ, KP, sK, KP, kBC, kBC, K, 1.f, false);
    __syncthreads();
    for (int e = threadIdx.x; e < kBC * kBC; e += kBThreads) {
        const int i = e / kBC, j = e - i * kBC;
        const float gm = i >= j ? __expf(sG[i] - sG[j]) : 0.f;
        sA[i * kCP + j] = i > j ? sBeta[i] * gm * sA[i * kCP + j] : 0.f;  // L
        sP[i * kCP + j] = a.scale * gm * sP[i * kCP + j];
    }
    __syncthreads();
    unit_lower_inverse(sA);
    const size_t base = ((size_t)tile_slot(bos, n, c) * a.HV + hv) * kBC * kBC;
    for (int e4 = threadIdx.x; e4 < kBC * kBC / 4; e4 += kBThreads) {
        const int i = e4 / (kBC / 4), j = (e4 % (kBC / 4)) * 4;
        *(float4 *)(a.Abuf + base + 4 * e4) = *(const float4 *)(sA + i * kCP + j);
        *(float4 *)(a.Pbuf + base + 4 * e4) = *(const float4 *)(sP + i * kCP + j);
    }
}

// ---- Steps 3-6, the state-dependent part: one CTA per (sequence, value head, value tile), newest chunk first
template <typename DT, int K>
__global__ void __launch_bounds__(kRThreads, 1) chunk_bwd_kernel(const BwdArgs a)
{
    using Lay = BwdLayout<K>;
    constexpr int KP = Lay::KP;
    constexpr bool EX = kExactOf<DT>;
    extern __shared__ float smem[];
    float *sK = smem + Lay::oK, *sQ = smem + Lay::oQ, *sS0 = smem + Lay::oS0, *sdS = smem + Lay::odS;
    float *sV = smem + Lay::oV, *sdO = smem + Lay::odO, *sR = smem + Lay::oR, *sD = smem + Lay::oD;
    float *sdD = smem + Lay::odD, *sY = smem + Lay::oY, *sA = smem + Lay::oA, *sP = smem + Lay::oP;
    float *sM2 = smem + Lay::oM2, *sG = smem + Lay::oG, *sGam = smem + Lay::oGam;
    float *sBeta = smem + Lay::oBeta, *sdG = smem + Lay::odG, *sdB = smem + Lay::odB, *sRed = smem + Lay::oRed;

    const int tid = threadIdx.x, w = tid >> 5, l = tid & 31;
    const int vt = blockIdx.x, pair = blockIdx.y;
    const int HV = a.HV, V = a.V, n = pair / HV, hv = pair % HV, hq = hv / (HV / a.H);
    const int64_t bos = a.cu_seqlens ? a.cu_seqlens[n] : (int64_t)n * a.T;
    const int64_t len = a.cu_seqlens ? a.cu_seqlens[n + 1] - bos : a.T;
    const int NT = (int)((len + kBC - 1) / kBC);
    const int col0 = vt * kBV;
    const float scale = a.scale;
    const DT *v = (const DT *)a.v, *dout = (const DT *)a.dout;
    const size_t pbase = ((size_t)n * HV + hv) * K * V;

    // dS: the gradient with respect to the state after the last chunk (dht)
    for (int e = tid; e < K * kBV; e += kRThreads) {
        const int d = e / kBV, j = e - d * kBV, col = col0 + j;
        sdS[d * kVP + j] = (a.dht && col < V) ? a.dht[pbase + (size_t)d * V + col] : 0.f;
    }

    for (int c = NT - 1; c >= 0; --c) {
        const int64_t t0 = bos + (int64_t)c * kBC;
        const size_t cidx = (size_t)tile_slot(bos, n, c) * HV + hv;
        __syncthreads();
        // ---- loads (rows past the sequence end are inert zeros)
        int rows;
        if (V % 8 == 0) {
            rows = load_step<DT, K>(a, bos, len, c, hv, col0, cidx, sK, sQ, sG, sGam, sBeta, sV, sdO, sS0, sA, sP);
        } else {
            rows = load_chunk<DT, K, kRThreads>(a, bos, len, c, hv, sK, sQ, sG, sGam, sBeta);
            const float *src = a.chunk_states + cidx * K * V;
            for (int e = tid; e < kBC * kBV; e += kRThreads) {
                const int i = e / kBV, j = e - i * kBV, col = col0 + j;
                float vv = 0.f, dv = 0.f;
                if (i < rows && col < V) {
                    const size_t off = ((size_t)(t0 + i) * HV + hv) * V + col;
                    vv = ldf(v + off);
                    dv = ldf(dout + off);
                }
                sV[i * kVP + j] = vv;
                sdO[i * kVP + j] = dv;
            }
            for (int e = tid; e < K * kBV; e += kRThreads) {
                const int d = e / kBV, j = e - d * kBV, col = col0 + j;
                sS0[d * kVP + j] = col < V ? src[(size_t)d * V + col] : 0.f;
            }
            const float *ga = a.Abuf + cidx * kBC * kBC, *gp = a.Pbuf + cidx * kBC * kBC;
            for (int e4 = tid; e4 < kBC * kBC / 4; e4 += kRThreads) {
                const int i = e4 / (kBC / 4), j = (e4 % (kBC / 4)) * 4;
                *(float4 *)(sA + i * kCP + j) = __ldg((const float4 *)ga + e4);
                *(float4 *)(sP + i * kCP + j) = __ldg((const float4 *)gp + e4);
            }
        }
        if (tid < kBC) sdG[tid] = sdB[tid] = 0.f;
        __syncthreads();
        const float GC = sG[kBC - 1], gamC = sGam[kBC - 1];
        if (tid < kBC) sRed[tid] = __expf(GC - sG[tid]);  // gam_C / gam

        // Phases between barriers (each line one phase; the products inside a phase are independent):
        //   K S0, P^T dO, K dS | R, B = diag(beta) R, dD | D = A B, Y = A^T dD | dO D^T, row sums, dR |
        //   dD B^T, the state terms of dq and dk | the gate terms, the dS update | the sums, dS
        // ---- K S0 (-> R), P^T dO (-> dD), K dS (scratch)
        tmm<false, false, 1, EX, false, false, kRThreads>(sR, kVP, sK, KP, sS0, kVP, kBC, kBV, K, 1.f, false);
        tmm<true, false, 1, false, EX, false, kRThreads>(sdD, kVP, sP, kCP, sdO, kVP, kBC, kBV, kBC, 1.f, false);
        tmm<false, false, 1, EX, false, false, kRThreads>(sM2, kVP, sK, KP, sdS, kVP, kBC, kBV, K, 1.f, false);
        __syncthreads();
        // ---- R = V - diag(gam) K S0, B = diag(beta) R (-> Y), dD = P^T dO + diag(gam_C / gam) K dS
        for (int e = tid; e < kBC * kBV; e += kRThreads) {
            const int i = e / kBV, j = e - i * kBV;
            const float r = sV[i * kVP + j] - sGam[i] * sR[i * kVP + j];
            sR[i * kVP + j] = r;
            sY[i * kVP + j] = sBeta[i] * r;
            sdD[i * kVP + j] = fmaf(sRed[i], sM2[i * kVP + j], sdD[i * kVP + j]);
        }
        __syncthreads();
        // ---- D = A B; Y2 = A^T dD (-> the scratch)
        tmm<false, false, 1, false, false, false, kRThreads>(sD, kVP, sA, kCP, sY, kVP, kBC, kBV, kBC, 1.f, false);
        tmm<true, false, 1, false, false, false, kRThreads>(sM2, kVP, sA, kCP, sdD, kVP, kBC, kBV, kBC, 1.f, false);
        __syncthreads();
        // ---- this tile's part of dP = dO D^T (-> P's buffer: P is read); dbeta_i += sum_v Y2 R,
        //      dG_i += beta_i sum_v Y2 (R - V); dR = diag(beta) Y2 (= dv, -> Y: B is read)
        tmm<false, true, 2, EX, false, false, kRThreads>(sP, kCP, sdO, kVP, sD, kVP, kBC, kBC, kBV, 1.f, false);
        {
            // kRThreads / 64 threads per row, columns p, p + that, ..., reduced over the group
            constexpr int TR = kRThreads / kBC;
            const int i = tid / TR, p = tid % TR;
            float sb = 0.f, sg = 0.f;
#pragma unroll
            for (int jj = 0; jj < kBV / TR; ++jj) {
                const int j = p + TR * jj;
                const float y = sM2[i * kVP + j], r = sR[i * kVP + j];
                sb = fmaf(y, r, sb);
                sg = fmaf(y, r - sV[i * kVP + j], sg);
            }
#pragma unroll
            for (int off = 1; off < TR; off <<= 1) {
                sb += __shfl_xor_sync(0xffffffffu, sb, off);
                sg += __shfl_xor_sync(0xffffffffu, sg, off);
            }
            if (p == 0) {
                sdB[i] += sb;
                sdG[i] += sBeta[i] * sg;
            }
        }
        for (int e = tid; e < kBC * kBV; e += kRThreads) {
            const int i = e / kBV, j = e - i * kBV;
            const float dr = sBeta[i] * sM2[i * kVP + j];
            sY[i * kVP + j] = dr;
            const int col = col0 + j;
            if (i < rows && col < V) a.dv[((size_t)(t0 + i) * HV + hv) * V + col] = dr;
        }
        __syncthreads();
        {
            float *dst = a.dPbuf + ((size_t)vt * a.chunk_heads + cidx) * kBC * kBC;
            for (int e4 = tid; e4 < kBC * kBC / 4; e4 += kRThreads)
                *(float4 *)(dst + 4 * e4) = *(const float4 *)(sP + (e4 / (kBC / 4)) * kCP + (e4 % (kBC / 4)) * 4);
        }
        // ---- this tile's part of dA = dD B^T (B = diag(beta) R: a column scale; -> the scratch, Y2 is read)
        tmm<false, true, 2, false, false, false, kRThreads>(sM2, kCP, sdD, kVP, sR, kVP, kBC, kBC, kBV, 1.f, false);

        // ---- state terms: dq += scale diag(gam) dO S0^T (dG_i += q_i . that), dk += diag(gam_C / gam) D dS^T
        //      (dG_C += k_j . that, dG_j -= k_j . that), dk -= diag(gam) dR S0^T, dG_C += gam_C <dS, S0>
        // (row dots: column part p of a row lands at kBC + 3 kBC p for q, at 2 kBC + 3 kBC p for k)
        constexpr int FNT = kFragNT<K, kRThreads>, NP = kRThreads / 128;
        float dq[FNT][4], dk[FNT][4], rd[2];
#pragma unroll
        for (int j = 0; j < FNT; ++j) dq[j][0] = dq[j][1] = dq[j][2] = dq[j][3] = dk[j][0] = dk[j][1] = dk[j][2] = dk[j][3] = 0.f;
        const int fr = 16 * (w & 3) + (l >> 2), fh = 3 * kBC * (w >> 2);
        facc<K, false, true, EX, false, kRThreads>(dq, sdO, kVP, sS0, kVP, kBV, scale, sGam);
        frdot<K, kRThreads>(dq, sQ, KP, rd);
        if ((l & 3) == 0) {
            sRed[kBC + fh + fr] = rd[0];
            sRed[kBC + fh + fr + 8] = rd[1];
        }
        facc<K, false, true, false, false, kRThreads>(dk, sD, kVP, sdS, kVP, kBV, 1.f, sRed);
        frdot<K, kRThreads>(dk, sK, KP, rd);
        if ((l & 3) == 0) {
            sRed[2 * kBC + fh + fr] = rd[0];
            sRed[2 * kBC + fh + fr + 8] = rd[1];
        }
        facc<K, false, true, false, false, kRThreads>(dk, sY, kVP, sS0, kVP, kBV, -1.f, sGam);
        {
            float sum = 0.f;
            for (int e = tid; e < K * kBV; e += kRThreads) {
                const int d = e / kBV, j = e - d * kBV;
                sum = fmaf(sdS[d * kVP + j], sS0[d * kVP + j], sum);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (l == 0) sRed[3 * kBC + w] = sum;
        }
        // this chunk's dq, dk into the sums over value tiles (and a GVA group's value heads)
        fatomic_rows<K, kRThreads>(dq, dk, a.dq, a.dk, t0, rows, a.H, hq);
        __syncthreads();  // S0 is read for the last time; the row terms are in sRed; dA's part is complete
        {
            float *dst = a.dAbuf + ((size_t)vt * a.chunk_heads + cidx) * kBC * kBC;
            for (int e4 = tid; e4 < kBC * kBC / 4; e4 += kRThreads) {
                const int i = e4 / (kBC / 4), j = (e4 % (kBC / 4)) * 4;
                const float4 m = *(const float4 *)(sM2 + i * kCP + j), b = *(const float4 *)(sBeta + j);
                *(float4 *)(dst + 4 * e4) = make_float4(m.x * b.x, m.y * b.y, m.z * b.z, m.w * b.w);
            }
        }
        if (w == 0) {
            // gate terms of the state products (lane: rows l, l + 32); G_C is the last row's G (rows past the
            // end carry g = 0), so its gradient belongs to the last row of the sequence
            float gcsum = l < kRThreads / 32 ? gamC * sRed[3 * kBC + l] : 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = l + 32 * h;
                float qd = 0.f, kd = 0.f;
#pragma unroll
                for (int pp = 0; pp < NP; ++pp) {
                    qd += sRed[kBC + 3 * kBC * pp + i];
                    kd += sRed[2 * kBC + 3 * kBC * pp + i];
                }
                sdG[i] += qd - kd;
                gcsum += kd;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) gcsum += __shfl_xor_sync(0xffffffffu, gcsum, off);
            __syncwarp();
            if (l == 0) sdG[kBC - 1] += gcsum;
            __syncwarp();
            float tail = (l >= rows ? sdG[l] : 0.f) + (l + 32 >= rows ? sdG[l + 32] : 0.f);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tail += __shfl_xor_sync(0xffffffffu, tail, off);
            if (l == 0) sdG[rows - 1] += tail;
        }
        // ---- Step 4: dS <- gam_C dS + scale Q^T diag(gam) dO - K^T diag(gam) dR (into S0's buffer)
        tmm<true, false, 2, EX, false, true, kRThreads>(sS0, kVP, sQ, KP, sdO, kVP, K, kBV, kBC, scale, false, sGam);
        tmm<true, false, 2, EX, false, true, kRThreads>(sS0, kVP, sK, KP, sY, kVP, K, kBV, kBC, -1.f, true, sGam);
        __syncthreads();
        for (int i = tid; i < rows; i += kRThreads) {
            atomicAdd(&a.dbeta[(size_t)(t0 + i) * HV + hv], sdB[i]);
            atomicAdd(&a.dG[(size_t)(t0 + i) * HV + hv], sdG[i]);
        }
        for (int e = tid; e < K * kBV; e += kRThreads) {
            const int d = e / kBV, j = e - d * kBV;
            sS0[d * kVP + j] = fmaf(gamC, sdS[d * kVP + j], sS0[d * kVP + j]);
        }
        float *tmp = sS0;
        sS0 = sdS;
        sdS = tmp;
    }
    __syncthreads();
    if (a.dh0) {
        for (int e = tid; e < K * kBV; e += kRThreads) {
            const int d = e / kBV, j = e - d * kBV, col = col0 + j;
            if (col < V) a.dh0[pbase + (size_t)d * V + col] = sdS[d * kVP + j];
        }
    }
}

// ---- Steps 5-6, the state-independent part: one CTA per chunk and value head, after the reverse scan
template <typename DT, int K>
__global__ void __launch_bounds__(kRThreads, 1) bwd_finish_kernel(const BwdArgs a)
{
    using Lay = ChunkLayout<K>;
    constexpr int KP = Lay::KP;
    constexpr bool EX = kExactOf<DT>;
    extern __shared__ float smem[];
    float *sK = smem + Lay::oK, *sQ = smem + Lay::oQ, *sA = smem + Lay::oA, *sP = smem + Lay::oP;
    float *sdP = smem + Lay::odP, *sdA = smem + Lay::odA, *sT = smem + Lay::oT, *sG = smem + Lay::oG;
    float *sBeta = smem + Lay::oBeta, *sRed = smem + Lay::oRed;
    const int tid = threadIdx.x;
    int n, hv, c;
    int64_t bos, len;
    if (!chunk_of_block(a, n, hv, c, bos, len)) return;
    const int HV = a.HV, hq = hv / (HV / a.H);
    const int64_t t0 = bos + (int64_t)c * kBC;
    const size_t cidx = (size_t)tile_slot(bos, n, c) * HV + hv;
    const int rows = load_chunk<DT, K, kRThreads>(a, bos, len, c, hv, sK, sQ, sG, nullptr, sBeta);
    const int tiles = (a.V + kBV - 1) / kBV;
    // the value tiles' parts of dP and dA summed (16-byte loads, all of a thread's issued together)
#pragma unroll 4
    for (int e4 = tid; e4 < kBC * kBC / 4; e4 += kRThreads) {
        const int i = e4 / (kBC / 4), j = (e4 % (kBC / 4)) * 4;
        float4 dp = make_float4(0.f, 0.f, 0.f, 0.f), da = dp;
#pragma unroll 4
        for (int t = 0; t < tiles; ++t) {
            const float4 x = __ldg((const float4 *)(a.dPbuf + ((size_t)t * a.chunk_heads + cidx) * kBC * kBC) + e4);
            const float4 y = __ldg((const float4 *)(a.dAbuf + ((size_t)t * a.chunk_heads + cidx) * kBC * kBC) + e4);
            dp.x += x.x; dp.y += x.y; dp.z += x.z; dp.w += x.w;
            da.x += y.x; da.y += y.y; da.z += y.z; da.w += y.w;
        }
        *(float4 *)(sdP + i * kCP + j) = dp;
        *(float4 *)(sdA + i * kCP + j) = da;
        *(float4 *)(sA + i * kCP + j) = __ldg((const float4 *)(a.Abuf + cidx * kBC * kBC) + e4);
        *(float4 *)(sP + i * kCP + j) = __ldg((const float4 *)(a.Pbuf + cidx * kBC * kBC) + e4);
    }
    __syncthreads();
    // P = scale Gam * Q K^T (i >= j): dG_i += rowsum(P dP), dG_j -= colsum(P dP); F = scale Gam * dP
    if (tid < 2 * kBC) {
        const int x = tid & (kBC - 1);
        float sum = 0.f;
        if (tid < kBC)
            for (int j = 0; j < kBC; ++j) sum = fmaf(sP[x * kCP + j], sdP[x * kCP + j], sum);
        else
            for (int i = 0; i < kBC; ++i) sum = fmaf(sP[i * kCP + x], sdP[i * kCP + x], sum);
        sRed[tid] = sum;  // [0, 64): rows, [64, 128): columns
    }
    __syncthreads();
    for (int e = tid; e < kBC * kBC; e += kRThreads) {
        const int i = e / kBC, j = e - i * kBC;
        sdP[i * kCP + j] = i >= j ? a.scale * __expf(sG[i] - sG[j]) * sdP[i * kCP + j] : 0.f;  // F
    }
    // dL = -A^T (dA A^T)
    tmm<false, true, 2, false, false, false, kRThreads>(sT, kCP, sdA, kCP, sA, kCP, kBC, kBC, kBC, 1.f, false);
    __syncthreads();
    tmm<true, false, 2, false, false, false, kRThreads>(sdA, kCP, sA, kCP, sT, kCP, kBC, kBC, kBC, -1.f, false);
    // K K^T -> Lraw = Gam * K K^T below the diagonal (into A's buffer: A is no longer read)
    __syncthreads();
    tmm<false, true, 2, EX, EX, false, kRThreads>(sA, kCP, sK, KP, sK, KP, kBC, kBC, K, 1.f, false);
    __syncthreads();
    for (int e = tid; e < kBC * kBC; e += kRThreads) {
        const int i = e / kBC, j = e - i * kBC;
        const float gm = i > j ? __expf(sG[i] - sG[j]) : 0.f;
        const float lraw = gm * sA[i * kCP + j];
        const float dl = i > j ? sdA[i * kCP + j] : 0.f;
        sT[i * kCP + j] = dl * lraw;                    // dL * Lraw (dbeta; times beta_i: the gate terms of L)
        sdA[i * kCP + j] = sBeta[i] * gm * dl;          // E = d(K K^T)
    }
    __syncthreads();
    // dbeta_i += rowsum(dL Lraw); dG_i += beta_i rowsum(dL Lraw) - beta_j colsum(dL Lraw) ... (L_ij = beta_i Lraw_ij)
    if (tid < 2 * kBC) {
        const int x = tid & (kBC - 1);
        float sum = 0.f;
        if (tid < kBC) {
            for (int j = 0; j < kBC; ++j) sum += sT[x * kCP + j];
        } else {
            for (int i = 0; i < kBC; ++i) sum = fmaf(sBeta[i], sT[i * kCP + x], sum);
        }
        sRed[2 * kBC + tid] = sum;  // [128, 192): dL Lraw row sums, [192, 256): beta-weighted column sums
    }
    // dq += F K, dk += F^T Q + E K + E^T K
    constexpr int FNT = kFragNT<K, kRThreads>;
    float dq[FNT][4], dk[FNT][4];
#pragma unroll
    for (int j = 0; j < FNT; ++j) dq[j][0] = dq[j][1] = dq[j][2] = dq[j][3] = dk[j][0] = dk[j][1] = dk[j][2] = dk[j][3] = 0.f;
    facc<K, false, false, false, EX, kRThreads>(dq, sdP, kCP, sK, KP, kBC);
    facc<K, true, false, false, EX, kRThreads>(dk, sdP, kCP, sQ, KP, kBC);
    facc<K, false, false, false, EX, kRThreads>(dk, sdA, kCP, sK, KP, kBC);
    facc<K, true, false, false, EX, kRThreads>(dk, sdA, kCP, sK, KP, kBC);
    fatomic_rows<K, kRThreads>(dq, dk, a.dq, a.dk, t0, rows, a.H, hq);
    __syncthreads();
    if (tid < rows) {
        const int i = tid;
        const float db = sRed[2 * kBC + i];
        const float dgv = sRed[i] - sRed[kBC + i] + sBeta[i] * db - sRed[3 * kBC + i];
        atomicAdd(&a.dbeta[(size_t)(t0 + i) * HV + hv], db);
        atomicAdd(&a.dG[(size_t)(t0 + i) * HV + hv], dgv);
    }
}

// dg = the suffix sum of dG within each chunk (one warp per (sequence, value head, chunk))
__global__ void gate_suffix_kernel(const BwdArgs a)
{
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int pair = (int)(item / a.max_nt), c = (int)(item % a.max_nt);
    if (pair >= a.N * a.HV) return;
    const int n = pair / a.HV, hv = pair % a.HV;
    const int64_t bos = a.cu_seqlens ? a.cu_seqlens[n] : (int64_t)n * a.T;
    const int64_t len = a.cu_seqlens ? a.cu_seqlens[n + 1] - bos : a.T;
    if ((int64_t)c * kBC >= len) return;
    const int rows = (int)min((int64_t)kBC, len - (int64_t)c * kBC);
    const int64_t t0 = bos + (int64_t)c * kBC;
    // lane l holds rows 2l, 2l + 1; a reverse inclusive scan
    const int r0 = 2 * lane, r1 = r0 + 1;
    const float x0 = r0 < rows ? a.dG[(size_t)(t0 + r0) * a.HV + hv] : 0.f;
    const float x1 = r1 < rows ? a.dG[(size_t)(t0 + r1) * a.HV + hv] : 0.f;
    float sp = x0 + x1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, sp, off);
        if (lane + off < 32) sp += y;
    }
    if (r0 < rows) a.dg[(size_t)(t0 + r0) * a.HV + hv] = sp;
    if (r1 < rows) a.dg[(size_t)(t0 + r1) * a.HV + hv] = sp - x0;
}

template <typename DT, int K>
cudaError_t launch_bwd_k(const BwdArgs &a, cudaStream_t st)
{
    auto prep = bwd_prep_kernel<DT, K>;
    auto scan = chunk_bwd_kernel<DT, K>;
    auto fin = bwd_finish_kernel<DT, K>;
    const size_t sp = sizeof(float) * PrepLayout<K>::total, sc = sizeof(float) * ChunkLayout<K>::total,
                 ss = sizeof(float) * BwdLayout<K>::total;
    cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fin, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc);
    if (e != cudaSuccess) return e;
    const dim3 gc(a.max_nt, a.N * a.HV);
    prep<<<gc, kBThreads, sp, st>>>(a);
    scan<<<dim3(ceil_div(a.V, kBV), a.N * a.HV), kRThreads, ss, st>>>(a);
    fin<<<gc, kRThreads, sc, st>>>(a);
    return cudaGetLastError();
}

template <typename DT>
cudaError_t launch_bwd_t(const BwdArgs &a, cudaStream_t st)
{
    switch (a.K) {
    case 32: return launch_bwd_k<DT, 32>(a, st);
    case 64: return launch_bwd_k<DT, 64>(a, st);
    case 128: return launch_bwd_k<DT, 128>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_chunk_bwd(const BwdArgs &a, gdn_dtype dt, cudaStream_t st)
{
    static_assert(sizeof(float) * BwdLayout<128>::total <= 227 * 1024 &&
                      sizeof(float) * ChunkLayout<128>::total <= 227 * 1024 &&
                      2 * (sizeof(float) * PrepLayout<128>::total + 1024) <= 228 * 1024,
                  "shared memory budget");
    if (a.N * a.HV == 0 || a.max_nt == 0) return cudaSuccess;
    cudaError_t e = dt == GDN_BF16 ? launch_bwd_t<__nv_bfloat16>(a, st) : launch_bwd_t<float>(a, st);
    if (e != cudaSuccess) return e;
    const int64_t items = (int64_t)a.N * a.HV * a.max_nt;
    gate_suffix_kernel<<<(unsigned)((items + 7) / 8), 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn

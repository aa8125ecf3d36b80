// Chunk preparation for the tensor-core engine: for every chunk of every
// (sequence, value head), the two bf16 operand tiles of the WY form
//
//   L    = diag(beta) StrictLower(K K^T)                    (FlashQLA blog, step 1)
//   X    = (I + L)^-1                                      (FLA page, sec. 4: exact blocked inverse)
//   A_g  = Gam * X,   Gam_ij = 2^(G_i - G_j)               (gated inverse, FlashQLA blog)
//   T_U  = A_g diag(beta),   T_W = A_g diag(beta gam) = diag(gam) X diag(beta)
//
// (G = chunk-local inclusive cumsum of the log-gate in base 2, gam = 2^G).  None of
// this depends on the state, so all chunks are prepared at once, one CTA per chunk,
// several CTAs per SM; the scan kernel loads the tiles with TMA (U = T_U V and
// W = T_W K are then single tensor-core products on its side).
//
// Tiles: bf16 [slot][HV][2][64][64] row-major (T_U then T_W), slot = tile_slot(bos, n, c).
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

namespace gdn {
namespace {
using namespace ptx;

constexpr int kThreadsPrep = 128;
constexpr int kLdX = 68;   // fp32 row pitch of the L / X tile
constexpr uint32_t kTmemCols = 64;  // the K K^T accumulator; eight CTAs per SM fill the 512 columns
constexpr float kFactorFloor = -100.f;  // G_C >= this: Gam_ij = gam_i * 2^-G_j without overflow

struct PrepSmem {
    // bytes 0-16383: the chunk's K rows, 128-byte swizzled boxes of 64 rows x 64 dk (dk 0-63, then
    // 64-127), until K K^T is formed (the 128-row operand of the product reads one box past the second:
    // bytes 16384-24575, where the in-kernel L2 norm puts q's first box, dk 0-63).  Then bytes 0-8191:
    // q's second box (L2 norm only) until the last merge, then the T_W and T_U tiles, 128-byte swizzled,
    // for their TMA stores; from byte 8192 the fp32 L / X tile: L in the lower triangle, X^T in the upper
    // (X(r, j), j < r, at lx[j * kLdX + r]).
    __align__(1024) uint8_t buf[8192 + 64 * kLdX * 4];
    __align__(16) float G[64], beta[64], gam[64], br[64];  // br = beta / gam
    __align__(16) float bw[64], rk[64];  // beta / ||k|| (T_W's column factor), 1 / ||k|| (in-kernel L2 norm)
    uint64_t bar, kbar, qbar;  // the product's completion; the K boxes' arrival; the second Q box's (L2 norm)
    uint32_t tslot;
};

__device__ __forceinline__ int rows_in(int64_t len, int c)
{
    const int64_t r = len - (int64_t)c * kChunk;
    return r < kChunk ? (int)r : kChunk;
}

template <bool ACT>
__global__ void __launch_bounds__(kThreadsPrep, 8) tc_prep_kernel(const PrepArgs a, const __grid_constant__ CUtensorMap tmap,
                                                                   const __grid_constant__ CUtensorMap kmap,
                                                                   const __grid_constant__ CUtensorMap qmap)
{
    // ACT: the in-kernel input activations (raw gate input, sigmoid(beta), L2 norm of k and q); a
    // separate instance, so that the plain one carries none of their code
    __shared__ __align__(1024) PrepSmem sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (a.seq_order && blockIdx.x == 0 && blockIdx.y == 0) {  // the scan's CTA order (K's buffer as scratch)
        order_longest_first(a.cu_seqlens, a.N, a.n_buckets, (int *)sh.buf, a.seq_order);
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
    float *lx = (float *)(sh.buf + 8192);

    if (warp == 0) tmem_alloc(&sh.tslot, kTmemCols);
    if (tid == 32) {
        // the chunk's K rows by two TMA boxes (dk 0-63, 64-127) straight into the swizzled operand layout
        mbar_init(&sh.bar, 1);
        mbar_init(&sh.kbar, 1);
        mbar_init(&sh.qbar, 1);
        fence_mbar_init();
        fence_proxy_async();  // (block (0, 0) used the buffer as scratch above)
        const bool qn = ACT && a.rq;  // in-kernel L2 norm of q: its first box (dk 0-63) beside K's, where L goes later
        mbar_arrive_expect_tx(&sh.kbar, qn ? 24576u : 16384u);
        tma_load_3d(sh.buf, &kmap, 0, hq, (int)t0, &sh.kbar);
        tma_load_3d(sh.buf + 8192, &kmap, 64, hq, (int)t0, &sh.kbar);
        if (qn) tma_load_3d(sh.buf + 16384, &qmap, 0, hq, (int)t0, &sh.kbar);
    }
    __syncthreads();  // the barriers are initialised before any thread waits on them
    // ---- gates (warp 0; issued while the K boxes are in flight), then the K boxes' tail rows
    const int r0 = 2 * lane, r1 = r0 + 1;
    float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
    if (warp == 0) {
        // every load first (the head's activation parameters with them), then the activations
        float ea = 0.f, bias = 0.f;
        if (ACT && a.act.A_log) {
            ea = a.act.A_log[hv];
            if (a.act.dt_bias) bias = a.act.dt_bias[hv];
        }
        if (r0 < rows) {
            g0 = a.g[(size_t)(t0 + r0) * HV + hv];
            b0 = a.beta[(size_t)(t0 + r0) * HV + hv];
        }
        if (r1 < rows) {
            g1 = a.g[(size_t)(t0 + r1) * HV + hv];
            b1 = a.beta[(size_t)(t0 + r1) * HV + hv];
        }
        if constexpr (ACT) {
            if (a.act.A_log) {
                ea = expf(ea);
                if (r0 < rows) g0 = act_gate_pre(a.act, g0, bias, ea);
                if (r1 < rows) g1 = act_gate_pre(a.act, g1, bias, ea);
            }
            if (r0 < rows) b0 = act_beta(a.act, b0);
            if (r1 < rows) b1 = act_beta(a.act, b1);
        }
        g0 *= kRcpLn2;
        g1 *= kRcpLn2;
    }
    {
        // the K boxes have landed; rows past the end of the sequence (the next one's, or zero fill past the
        // tensor) become zeros (a wait that runs out leaves the status flag and a wrong chunk, never a hang)
        mbar_wait(&sh.kbar, 0, a.status, kStatusTimeout, a.wait_ns);
        for (int e = tid; e < (kChunk - rows) * 16; e += kThreadsPrep) {
            const int r = rows + (e >> 4), piece = e & 15;
            *(uint4 *)(sh.buf + (piece >> 3) * 8192 + r * 128 + (piece & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();  // the tensor core reads them
    }
    // in-kernel L2 norm of q, first half: row qr's sum of squares over dk 0-63 (two threads per row, four of its
    // eight 16-byte pieces each: the swizzle only permutes a row's pieces; each row takes its pieces in an
    // order rotated by the row, so that the eight lanes of a quarter warp read eight different bank groups)
    const int qr = tid >> 1, qh = tid & 1;
    float qss = 0.f;
    auto q_sumsq = [&](const uint8_t *box) {
        const uint8_t *src = box + qr * 128 + qh * 64;
        uint4 x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = *(const uint4 *)(src + ((j + qr) & 3) * 16);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 *h2 = (const __nv_bfloat162 *)&x[j];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 f = __bfloat1622float2(h2[u]);
                qss = fmaf(f.x, f.x, fmaf(f.y, f.y, qss));
            }
        }
    };
    if (ACT && a.rq) q_sumsq(sh.buf + 16384);
    if (warp == 0) {
        float sp = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, sp, off);
            if (lane >= off) sp += y;
        }
        const float G0 = sp - g1, G1 = sp;
        sh.G[r0] = G0;
        sh.G[r1] = G1;
        sh.beta[r0] = b0;
        sh.beta[r1] = b1;
        sh.gam[r0] = ex2(G0);
        sh.gam[r1] = ex2(G1);
        sh.br[r0] = b0 * ex2(-G0);  // used only when G_C >= kFactorFloor
        sh.br[r1] = b1 * ex2(-G1);
    }
    // one barrier publishes the K boxes, the gates and the tensor-memory allocation
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- K K^T on the tensor core: one M = 128 product ([K; next box] K^T, lanes 0-63 hold K K^T);
    //      L row r = beta_r (K K^T)[r, :] straight from tensor memory (the upper triangle is
    //      overwritten by X^T later and never read before)
    const uint32_t tb = sh.tslot;
    if (warp == 0) {
        const uint32_t kb = smem_u32(sh.buf);
        const uint32_t idKK = idesc_bf16_f32(128, 64, 0, 0);
        if (elect_one_sync()) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t d = sdesc_sw128(kb + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
                mma_ss(tb, d, d, idKK, ks > 0 ? 1u : 0u);
            }
            mma_commit(&sh.bar);
        }
        __syncwarp();
    }
    if (warp < 2) {
        const bool ok = mbar_wait(&sh.bar, 0, a.status, kStatusTimeout, a.wait_ns);
        const bool all_ok = __all_sync(0xffffffffu, ok);
        if (ACT && a.rq && tid == 0 && ok) {
            // the product has read K's first box: q's second box (dk 64-127) lands there for the norm
            mbar_arrive_expect_tx(&sh.qbar, 8192u);
            tma_load_3d(sh.buf, &qmap, 64, hq, (int)t0, &sh.qbar);
        }
        const int r = 32 * warp + lane;
        // in-kernel L2 norm: ||k_r||^2 is the diagonal of K K^T (column r, in this warp's half); every
        // entry of L takes beta_r / (||k_r|| ||k_j||) and T_W's columns 1 / ||k_j|| (W = T_W K^, K^ = diag(rk) K)
        float rr = 1.f;
        if (ACT && a.act.qk_l2norm) {
            float dg = 0.f;
            if (all_ok) {
                uint32_t d[32];
                tc_fence_after();
                tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + 32 * warp, d);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j == lane) dg = __uint_as_float(d[j]);
            }
            rr = r < rows ? 1.f / fmaxf(sqrtf(fmaxf(dg, 0.f)), kNormEps) : 0.f;
            if (a.rk) a.rk[((size_t)slot * HV + hv) * 64 + r] = rr;
        }
        if constexpr (ACT) {
            sh.rk[r] = rr;
            sh.bw[r] = sh.beta[r] * rr;
            bar_sync(1, 64);  // both warps' 1 / ||k||
        }
        if (all_ok) {
            tc_fence_after();
            const float br_ = sh.beta[r] * rr;
            float *lr = lx + r * kLdX;
            float diag = 0.f;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t d[32];
                tmem_ld32(tb + ((uint32_t)(32 * warp) << 16) + 32 * h, d);
                tmem_ld_wait();
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 c = ACT ? *(const float4 *)(sh.rk + 32 * h + 4 * j4) : make_float4(1.f, 1.f, 1.f, 1.f);
                    float4 v;
                    v.x = br_ * c.x * __uint_as_float(d[4 * j4]);
                    v.y = br_ * c.y * __uint_as_float(d[4 * j4 + 1]);
                    v.z = br_ * c.z * __uint_as_float(d[4 * j4 + 2]);
                    v.w = br_ * c.w * __uint_as_float(d[4 * j4 + 3]);
                    if (32 * h + 4 * j4 == (r & ~3))
                        diag = (r & 3) == 0 ? v.x : (r & 3) == 1 ? v.y : (r & 3) == 2 ? v.z : v.w;
                    *(float4 *)(lr + 32 * h + 4 * j4) = v;
                }
            }
            // beta ||k||^2 <= 2 keeps every transition non-expansive (warmup split)
            if (a.check_norm && diag > 2.0001f) atomicOr(a.status, kStatusNormBound);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, kTmemCols);
    }

    auto Lx = [&](int r, int j) -> float { return lx[r * kLdX + j]; };
    auto Xt = [&](int r, int j) -> float { return lx[j * kLdX + r]; };  // X(r, j), j < r
    auto Xm = [&](int r, int j) -> float { return r > j ? lx[j * kLdX + r] : (r == j ? 1.f : 0.f); };
    const int pw = warp;
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
    __syncthreads();
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
    __syncthreads();
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
    __syncthreads();
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
    if (ACT && a.rq) {
        // in-kernel L2 norm of q, second half, and 1 / ||q_r|| for the scan's row factors (rows past the end
        // of the sequence 0); the box is read before the barrier after which the tiles are staged there
        if (mbar_wait(&sh.qbar, 0, a.status, kStatusTimeout, a.wait_ns)) q_sumsq(sh.buf);
        qss += __shfl_xor_sync(0xffffffffu, qss, 1);
        if (qh == 0) a.rq[((size_t)slot * HV + hv) * 64 + qr] = qr < rows ? 1.f / fmaxf(sqrtf(qss), kNormEps) : 0.f;
    }
    __syncthreads();

    // ---- operand tiles, each staged in the dead K box (128-byte swizzle) and written by one TMA store:
    //      T_W, then T_U once the first copy has read the box.  Warp w takes the 8-column piece w of each
    //      of the three nonzero quadrants (rows 0-31 x columns 0-31 and rows 32-63 x columns 32-63: diagonal
    //      blocks; rows 32-63 x columns 0-31: all below the diagonal, no masks), lane = row within the
    //      quadrant, one 16-byte piece per quadrant: consecutive rows of X^T (no conflicts), equal work per
    //      warp.  The all-zero quadrant (rows 0-31, columns 32-63) is written once, piece 4 + w by warp w,
    //      and both tiles share it
    {
        const bool factored = sh.G[63] >= kFactorFloor;
        const int row0 = (int)(((size_t)slot * HV + hv) * 2 * 64);  // T_U rows; T_W follows
        const float ga = sh.gam[lane], gb = sh.gam[32 + lane], Ga = sh.G[lane], Gb = sh.G[32 + lane];
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {  // 0: T_W, 1: T_U
            if (pass == 1) {
                if (tid == 0) tma_store_wait_read0();
                __syncthreads();
            } else {
                *(uint4 *)(sh.buf + lane * 128 + (((4 + warp) ^ (lane & 7)) << 4)) = make_uint4(0, 0, 0, 0);
            }
            const float *bsrc = pass == 0 ? (ACT ? sh.bw : sh.beta) : !factored ? sh.beta : sh.br;
            const bool plain = pass == 0 || factored;  // T_W, or T_U with the factored form: gam_r X beta'_j
#pragma unroll
            for (int qd = 0; qd < 3; ++qd) {  // 0: upper diagonal block, 1: below the diagonal, 2: lower one
                const int r = qd == 0 ? lane : 32 + lane;
                const int j0 = (qd == 2 ? 32 : 0) + 8 * warp;
                const float gr = qd == 0 ? ga : gb, Gr = qd == 0 ? Ga : Gb;
                const float4 b0 = *(const float4 *)(bsrc + j0), b1 = *(const float4 *)(bsrc + j0 + 4);
                const float bj[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int jj = j0 + u;
                    // T_W = gam_r X beta_j; T_U = gam_r X beta_j / gam_j (factored: br = beta / gam; else the
                    // power 2^(G_r - G_j) per element)
                    const float xv = qd == 1 ? lx[jj * kLdX + r] : (jj < r ? lx[jj * kLdX + r] : (jj == r ? 1.f : 0.f));
                    v[u] = plain ? gr * bj[u] * xv : (qd == 1 || jj <= r ? ex2(Gr - sh.G[jj]) * bj[u] * xv : 0.f);
                }
                *(uint4 *)(sh.buf + r * 128 + (((j0 >> 3) ^ (r & 7)) << 4)) = pack8(v);
            }
            fence_proxy_async();  // the tensor-memory-access unit reads the staging box
            __syncthreads();
            if (tid == 0) {
                tma_store_2d(&tmap, sh.buf, 0, row0 + (pass == 0 ? 64 : 0));
                tma_store_commit();
            }
        }
        if (tid == 0) tma_store_wait_read0();  // the box stays valid until the copy has read it
    }
}

}  // namespace

cudaError_t launch_tc_prep(const PrepArgs &a, cudaStream_t st)
{
    if (a.N * a.HV == 0 || a.slots == 0) return cudaSuccess;
    // eight CTAs per SM need the largest shared-memory carveout
    cudaError_t e = cudaFuncSetAttribute(tc_prep_kernel<false>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(tc_prep_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    // T_W leaves through a TMA store: the same tile map as the scan reads it with
    alignas(64) CUtensorMap tmap;
    if (!encode_tiles_map(&tmap, a.tiles, (int64_t)a.slots * a.HV * 128, 64)) return cudaErrorInvalidValue;
    // the chunks' K rows arrive by TMA: the map the scan reads K with
    alignas(64) CUtensorMap kmap;
    if (!encode_rows_map(&kmap, a.k, a.H, a.cu_seqlens ? (int64_t)a.T : (int64_t)a.N * a.T)) return cudaErrorInvalidValue;
    // and, for the in-kernel L2 norm of q, its rows (the K map again when there is none: never read)
    alignas(64) CUtensorMap qmap = kmap;
    if (a.rq && !encode_rows_map(&qmap, a.q, a.H, a.cu_seqlens ? (int64_t)a.T : (int64_t)a.N * a.T))
        return cudaErrorInvalidValue;
    dim3 grid(a.slots, a.HV);
    if (a.act.A_log || a.act.beta_logits || a.act.qk_l2norm) tc_prep_kernel<true><<<grid, kThreadsPrep, 0, st>>>(a, tmap, kmap, qmap);
    else tc_prep_kernel<false><<<grid, kThreadsPrep, 0, st>>>(a, tmap, kmap, qmap);
    return cudaGetLastError();
}

}  // namespace gdn

// Tensor-core engine (sm_103a: tcgen05 + TMEM + TMA) of the chunked gated
// delta rule for bf16 q/k/v, dk = dv = 128, scalar gate, C = 64.
//
// One CTA owns one (sequence, value head, segment) and walks its chunks
// serially.  The state is kept transposed, S^T [dv x dk] fp32, in tensor
// memory (lane = dv), so every product of the chunk step is an M = 128
// tcgen05 MMA with dv as M.  The chunk step is the FlashQLA restructured form
// (FlashQLA blog, "A balanced solution", step 3), with A0 from step 1:
//
//   A0    = (I + StrictLower(diag(beta) K K^T))^-1        (prep warps, CUDA cores)
//   A_g   = Gam * A0,  P_g = scale Lower(Gam) * (Q K^T)    (prep warps)
//   X^T   = S^T K^T                                        (MMA, A = S^T bf16 in TMEM)
//   Y^T   = (V^T - X^T diag(gam)) diag(beta)               (chain warps)
//   V'^T  = Y^T A_g^T                                      (MMA)
//   O^T   = scale (S^T Q^T) diag(gam) + V'^T P_g^T         (MMA x2, epilogue warps)
//   S^T  <- gC S^T + (V'^T diag(gC / gam)) K               (MMA, B = K MN-major)
//
// with G the chunk-local inclusive cumsum of the log-gate (kept in base 2),
// gam = 2^G, Gam_ij = 2^(G_i - G_j), gC = gam of the last valid row.
//
// Warp roles (16 warps): 0 TMA producer (+ gate cumsum), 1 MMA issuer,
// 2 TMEM allocator, 4-7 chain (state / Y / V'), 8-11 prep (K K^T -> inverse
// -> A_g, Q K^T -> P_g), 12-15 output epilogue.  All waits are bounded in
// wall time; a wait that runs out records a timeout in the status word and
// every role leaves its loop, so the kernel always ends and frees TMEM.
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace gdn {
namespace {
using namespace ptx;

constexpr int kThreadsTC = 512;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait, then give up

// ---- shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t kStageBytes = 49152;  // K0 | Q0 | K1 | Q1 | V0 | V1, 8 KB each
constexpr uint32_t sK0 = 0, sQ0 = 8192, sK1 = 16384, sQ1 = 24576, sV0 = 32768, sV1 = 40960;
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_A = OFF_STAGE + 2 * kStageBytes;  // A_g  [64 x 64] bf16 SW128, x2
constexpr uint32_t OFF_P = OFF_A + 2 * 8192;             // P_g  [64 x 64] bf16 SW128, x2
constexpr uint32_t OFF_VP = OFF_P + 2 * 8192;            // V'^T [128 x 64] bf16 SW128
constexpr uint32_t OFF_O = OFF_VP + 16384;               // O staging, 2 boxes [64 x 64] bf16
constexpr uint32_t OFF_L = OFF_O + 16384;                // L  fp32 [64][65]
constexpr uint32_t OFF_X = OFF_L + 64 * 65 * 4;          // X  fp32 [64][65]
constexpr uint32_t OFF_GATE = OFF_X + 64 * 65 * 4;       // per stage: G, beta, gam, rdec [64] f32
constexpr uint32_t OFF_PG = OFF_GATE + 2 * 1024;         // prep copy of G [64]
constexpr uint32_t OFF_EG = OFF_PG + 256;                // epilogue: scale * gam, per warp [4][64]
constexpr uint32_t OFF_BAR = OFF_EG + 1024;
constexpr uint32_t kSmemTC = OFF_BAR + 256 + 1024;       // + slack for the 1024-byte alignment

// ---- tensor memory columns
constexpr uint32_t TM_S = 0, TM_XV = 128, TM_O1 = 192, TM_O2 = 256, TM_KQ = 320, TM_SBF = 384,
                   TM_YBF = 448, TM_VTB = 480;

enum Bar {
    B_FULL = 0, B_EMPTY = 2, B_TMA = 4, B_KQF = 6, B_KQE, B_AF, B_AE = 10, B_SBF = 12, B_XF, B_YF, B_VPF,
    B_VTF, B_SF, B_OF, B_OE, B_COUNT
};

struct TcMaps {
    CUtensorMap q, k, v, o;
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

__device__ __forceinline__ bool bar_and(int id, int count, bool pred)
{
    uint32_t r;
    asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "r"(id), "r"(count)
                 : "memory");
    return r != 0;
}

__device__ __forceinline__ int rows_in(int64_t len, int c)
{
    const int64_t r = len - (int64_t)c * kChunk;
    return r < kChunk ? (int)r : kChunk;
}

__device__ __forceinline__ uint64_t kmaj(uint32_t addr) { return sdesc_sw128(addr, 16, 1024); }

__global__ void __launch_bounds__(kThreadsTC, 1) tc_scan_kernel(const ScanArgs a, const __grid_constant__ TcMaps m)
{
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    uint64_t *bars = (uint64_t *)(sm + OFF_BAR);
    uint32_t *tslot = (uint32_t *)(sm + OFF_BAR + 8 * B_COUNT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int vt = blockIdx.x, seg = blockIdx.y, pair = blockIdx.z;
    const int HV = a.HV, V = a.V;
    const int n = pair / HV, hv = pair % HV, hq = hv / (HV / a.H);
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
    const bool fwd = a.mode == kModeForward;
    const size_t sidx = ((size_t)n * HV + hv) * a.n_seg + seg;
    int cs = c0;
    if (fwd && a.warm_start) {
        cs = a.warm_start[sidx];
        if (cs < 0 || cs > c0) cs = 0;
    }
    const int nch = c1 - cs;
    const bool zero_values = !fwd && vt == 1;   // prepass: the M columns carry no values
    const bool check_norm = fwd && a.warm_start != nullptr;

    if (tid == 0) {
        if (seg == a.n_seg - 1 && c1 < NT) atomicOr(a.status, kStatusPlan);
        if (fwd && a.warm_start && (a.warm_start[sidx] < 0 || a.warm_start[sidx] > c0))
            atomicOr(a.status, kStatusPlan);
        mbar_init(&bars[B_FULL], 1);
        mbar_init(&bars[B_FULL + 1], 1);
        mbar_init(&bars[B_EMPTY], 9);
        mbar_init(&bars[B_EMPTY + 1], 9);
        mbar_init(&bars[B_TMA], 1);
        mbar_init(&bars[B_TMA + 1], 1);
        mbar_init(&bars[B_KQF], 1);
        mbar_init(&bars[B_KQE], 4);
        mbar_init(&bars[B_AF], 4);
        mbar_init(&bars[B_AF + 1], 4);
        mbar_init(&bars[B_AE], 1);
        mbar_init(&bars[B_AE + 1], 1);
        mbar_init(&bars[B_SBF], 4);
        mbar_init(&bars[B_XF], 1);
        mbar_init(&bars[B_YF], 4);
        mbar_init(&bars[B_VPF], 1);
        mbar_init(&bars[B_VTF], 4);
        mbar_init(&bars[B_SF], 1);
        mbar_init(&bars[B_OF], 1);
        mbar_init(&bars[B_OE], 4);
        fence_mbar_init();
    }
    if (warp == 2) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tslot;
    unsigned *status = a.status;

    if (warp == 0) {
        // ================================================================ producer
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
            const int c = cs + i, s = i & 1;
            if (i >= 2) ok = mbar_wait(&bars[B_EMPTY + s], ((i >> 1) - 1) & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const int64_t t0 = bos + (int64_t)c * kChunk;
            const int rows = rows_in(len, c);
            const bool emit = fwd && c >= c0;
            uint8_t *st = sm + OFF_STAGE + s * kStageBytes;
            // gates: lane holds rows 2l, 2l+1; base-2 inclusive cumsum across the warp
            const int r0 = 2 * lane, r1 = r0 + 1;
            float g0 = 0.f, g1 = 0.f, b0 = 0.f, b1 = 0.f;
            if (r0 < rows) {
                g0 = a.g[(size_t)(t0 + r0) * HV + hv] * kRcpLn2;
                b0 = a.beta[(size_t)(t0 + r0) * HV + hv];
            }
            if (r1 < rows) {
                g1 = a.g[(size_t)(t0 + r1) * HV + hv] * kRcpLn2;
                b1 = a.beta[(size_t)(t0 + r1) * HV + hv];
            }
            float sp = g0 + g1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, sp, off);
                if (lane >= off) sp += y;
            }
            const float G0 = sp - g1, G1 = sp;
            const float GC = __shfl_sync(0xffffffffu, sp, 31);
            float *gt = (float *)(sm + OFF_GATE + s * 1024);
            gt[r0] = G0;
            gt[r1] = G1;
            gt[64 + r0] = b0;
            gt[64 + r1] = b1;
            gt[128 + r0] = exp2f(G0);
            gt[128 + r1] = exp2f(G1);
            gt[192 + r0] = exp2f(GC - G0);
            gt[192 + r1] = exp2f(GC - G1);
            if (lane == 0) {
                const uint32_t bytes = 16384u + (emit ? 16384u : 0u) + (zero_values ? 0u : 16384u);
                mbar_arrive_expect_tx(&bars[B_TMA + s], bytes);
                const int tt = (int)t0;
                tma_load_3d(st + sK0, &m.k, 0, hq, tt, &bars[B_TMA + s]);
                tma_load_3d(st + sK1, &m.k, 64, hq, tt, &bars[B_TMA + s]);
                if (emit) {
                    tma_load_3d(st + sQ0, &m.q, 0, hq, tt, &bars[B_TMA + s]);
                    tma_load_3d(st + sQ1, &m.q, 64, hq, tt, &bars[B_TMA + s]);
                }
                if (!zero_values) {
                    tma_load_3d(st + sV0, &m.v, 0, hv, tt, &bars[B_TMA + s]);
                    tma_load_3d(st + sV1, &m.v, 64, hv, tt, &bars[B_TMA + s]);
                }
            }
            ok = mbar_wait(&bars[B_TMA + s], (i >> 1) & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (rows < kChunk) {
                // rows past the end of the sequence belong to the next one: make them inert zeros
                const uint4 z = make_uint4(0, 0, 0, 0);
                const int nz = (kChunk - rows) * 8;  // 16-byte pieces per box
#pragma unroll
                for (int bx = 0; bx < 6; ++bx) {
                    if ((bx == 2 || bx == 3) && !emit) continue;
                    if (bx >= 4 && zero_values) continue;
                    const uint32_t boff = bx == 0 ? sK0 : bx == 1 ? sK1 : bx == 2 ? sQ0 : bx == 3 ? sQ1 : bx == 4 ? sV0 : sV1;
                    uint4 *p = (uint4 *)(st + boff + rows * 128);
                    for (int e = lane; e < nz; e += 32) p[e] = z;
                }
                fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_FULL + s]);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0 && nch > 0) {
            const uint32_t idN64 = idesc_bf16_f32(128, 64, 0, 0);
            const uint32_t idN128MN = idesc_bf16_f32(128, 128, 0, 1);
            bool ok = mbar_wait(&bars[B_FULL], 0, status, kStatusTimeout, kWaitNs);
            auto issue_kq = [&](int j) {
                const uint32_t st = sbase + OFF_STAGE + (j & 1) * kStageBytes;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_ss(tb + TM_KQ, kmaj(st + off), kmaj(st + off), idN64, ks > 0);
                }
                mma_commit(&bars[B_KQF]);
            };
            if (ok) {
                tc_fence_after();
                issue_kq(0);
            }
            int e = 0;
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i & 1, b = i & 1, c = cs + i;
                const bool emit = fwd && c >= c0;
                const uint32_t st = sbase + OFF_STAGE + s * kStageBytes;
                ok = mbar_wait(&bars[B_SBF], i & 1, status, kStatusTimeout, kWaitNs);
                if (ok && emit && e > 0) ok = mbar_wait(&bars[B_OE], (e - 1) & 1, status, kStatusTimeout, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                // X^T = S^T K^T ; O1^T = S^T Q^T
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_ts(tb + TM_XV, tb + TM_SBF + ks * 8, kmaj(st + sK0 + off), idN64, ks > 0);
                }
                if (emit) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_ts(tb + TM_O1, tb + TM_SBF + ks * 8, kmaj(st + sQ0 + off), idN64, ks > 0);
                    }
                }
                mma_commit(&bars[B_XF]);
                ok = mbar_wait(&bars[B_YF], i & 1, status, kStatusTimeout, kWaitNs) &&
                     mbar_wait(&bars[B_AF + b], (i >> 1) & 1, status, kStatusTimeout, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                // V'^T = Y^T A_g^T
                const uint32_t abuf = sbase + OFF_A + b * 8192;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ts(tb + TM_XV, tb + TM_YBF + ks * 8, kmaj(abuf + ks * 32), idN64, ks > 0);
                mma_commit(&bars[B_VPF]);
                ok = mbar_wait(&bars[B_VTF], i & 1, status, kStatusTimeout, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                // S^T += (V'^T diag(gC/gam)) K   (B = K, MN-major: dk atoms 16 KB apart)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ts(tb + TM_S, tb + TM_VTB + ks * 8, sdesc_sw128(st + sK0 + ks * 2048, 16384, 1024),
                           idN128MN, 1);
                mma_commit(&bars[B_SF]);
                if (emit) {
                    // O2^T = V'^T P_g^T
                    const uint32_t pbuf = sbase + OFF_P + b * 8192, vp = sbase + OFF_VP;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tb + TM_O2, kmaj(vp + ks * 32), kmaj(pbuf + ks * 32), idN64, ks > 0);
                    mma_commit(&bars[B_OF]);
                    ++e;
                }
                mma_commit(&bars[B_EMPTY + s]);
                mma_commit(&bars[B_AE + b]);
                if (i + 1 < nch) {
                    ok = mbar_wait(&bars[B_FULL + ((i + 1) & 1)], ((i + 1) >> 1) & 1, status, kStatusTimeout, kWaitNs) &&
                         mbar_wait(&bars[B_KQE], i & 1, status, kStatusTimeout, kWaitNs);
                    if (!ok) break;
                    tc_fence_after();
                    issue_kq(i + 1);
                }
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ================================================================ chain (lane = dv)
        const int dv = tid - 128;
        const uint32_t tl = tb + ((uint32_t)((warp & 3) * 32) << 16);
        const float *init = nullptr;
        size_t init_stride = V;
        bool identity = false;
        if (fwd) {
            if (a.seg_init && seg > 0)
                init = a.seg_init + sidx * 128 * V;
            else if (cs == 0 && a.h0)
                init = a.h0 + ((size_t)n * HV + hv) * 128 * V;
        } else if (vt == 1) {
            identity = true;
        }
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
            const int s = i & 1, c = cs + i;
            const bool emit = fwd && c >= c0;
            ok = mbar_wait(&bars[B_FULL + s], (i >> 1) & 1, status, kStatusTimeout, kWaitNs);
            if (ok && i > 0) ok = mbar_wait(&bars[B_SF], (i - 1) & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const float *gt = (const float *)(sm + OFF_GATE + s * 1024);
            const float dec = gt[128 + 63];  // gC = 2^G_C
            // ---- S_i -> bf16 copy (MMA operand) and gC * S_i (accumulator of this chunk's update)
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t r[32], p[16];
                if (i == 0) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int d = 32 * q4 + j;
                        float x = 0.f;
                        if (init) x = init[(size_t)d * init_stride + dv];
                        else if (identity) x = (d == dv) ? 1.f : 0.f;
                        r[j] = f2u(x);
                    }
                } else {
                    tmem_ld32(tl + TM_S + 32 * q4, r);
                    tmem_ld_wait();
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) p[j] = pack_bf16(u2f(r[2 * j]), u2f(r[2 * j + 1]));
                tmem_st16(tl + TM_SBF + 16 * q4, p);
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = f2u(u2f(r[j]) * dec);
                tmem_st32(tl + TM_S + 32 * q4, r);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_SBF]);

            // ---- Y^T = beta (V^T - gam X^T)
            ok = mbar_wait(&bars[B_XF], i & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            {
                const uint8_t *vbox = sm + OFF_STAGE + s * kStageBytes + (dv < 64 ? sV0 : sV1);
                const int dl = dv & 63;
                uint32_t y[32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32];
                    tmem_ld32(tl + TM_XV + 32 * h, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const int cc = 32 * h + j;
                        float v0 = 0.f, v1 = 0.f;
                        if (!zero_values) {
                            v0 = __bfloat162float(*(const __nv_bfloat16 *)(vbox + sw128(cc, dl)));
                            v1 = __bfloat162float(*(const __nv_bfloat16 *)(vbox + sw128(cc + 1, dl)));
                        }
                        const float y0 = gt[64 + cc] * (v0 - gt[128 + cc] * u2f(r[j]));
                        const float y1 = gt[64 + cc + 1] * (v1 - gt[128 + cc + 1] * u2f(r[j + 1]));
                        y[16 * h + j / 2] = pack_bf16(y0, y1);
                    }
                }
                tmem_st32(tl + TM_YBF, y);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_YF]);

            // ---- V'^T -> bf16 (output operand, smem) and V'^T diag(gC/gam) (state operand, TMEM)
            ok = mbar_wait(&bars[B_VPF], i & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            {
                uint32_t vtl[32];
                uint8_t *vprow = sm + OFF_VP;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32];
                    tmem_ld32(tl + TM_XV + 32 * h, r);
                    tmem_ld_wait();
                    if (emit) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 pk;
                            pk.x = pack_bf16(u2f(r[8 * q + 0]), u2f(r[8 * q + 1]));
                            pk.y = pack_bf16(u2f(r[8 * q + 2]), u2f(r[8 * q + 3]));
                            pk.z = pack_bf16(u2f(r[8 * q + 4]), u2f(r[8 * q + 5]));
                            pk.w = pack_bf16(u2f(r[8 * q + 6]), u2f(r[8 * q + 7]));
                            *(uint4 *)(vprow + sw128(dv, 32 * h + 8 * q)) = pk;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const int cc = 32 * h + j;
                        vtl[16 * h + j / 2] = pack_bf16(u2f(r[j]) * gt[192 + cc], u2f(r[j + 1]) * gt[192 + cc + 1]);
                    }
                }
                tmem_st32(tl + TM_VTB, vtl);
                if (emit) fence_proxy_async();
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_VTF]);
                mbar_arrive(&bars[B_EMPTY + s]);  // done with this stage's V and gates
            }
        }
        // ---- final state of the segment
        const bool write_ht = fwd && c1 == NT && a.ht != nullptr;
        const bool write_seg = !fwd;
        if (write_ht || write_seg) {
            float *dst;
            size_t dstride;
            if (write_ht) {
                dst = a.ht + ((size_t)n * HV + hv) * 128 * V + dv;
                dstride = V;
            } else {
                dst = a.seg_out + sidx * 128 * (size_t)(V + 128) + vt * 128 + dv;
                dstride = V + 128;
            }
            if (nch == 0) {
                for (int d = 0; d < 128; ++d) {
                    float x = 0.f;
                    if (init) x = init[(size_t)d * init_stride + dv];
                    else if (identity) x = (d == dv) ? 1.f : 0.f;
                    dst[(size_t)d * dstride] = x;
                }
            } else if (ok) {
                ok = mbar_wait(&bars[B_SF], (nch - 1) & 1, status, kStatusTimeout, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) {
                    tc_fence_after();
#pragma unroll 1
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t r[32];
                        tmem_ld32(tl + TM_S + 32 * q4, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) dst[(size_t)(32 * q4 + j) * dstride] = u2f(r[j]);
                    }
                }
            }
        }
    } else if (warp >= 8 && warp < 12) {
        // ================================================================ prep (lane = row of [K;Q])
        const int pt = tid - 256;
        const uint32_t tl = tb + ((uint32_t)((warp & 3) * 32) << 16);
        float *sL = (float *)(sm + OFF_L);
        float *sX = (float *)(sm + OFF_X);
        float *pG = (float *)(sm + OFF_PG);
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
            const int s = i & 1, b = i & 1, c = cs + i;
            const bool emit = fwd && c >= c0;
            ok = mbar_wait(&bars[B_FULL + s], (i >> 1) & 1, status, kStatusTimeout, kWaitNs);
            if (ok && i >= 2) ok = mbar_wait(&bars[B_AE + b], ((i >> 1) - 1) & 1, status, kStatusTimeout, kWaitNs);
            if (ok) ok = mbar_wait(&bars[B_KQF], i & 1, status, kStatusTimeout, kWaitNs);
            ok = bar_and(1, 128, ok);
            if (!ok) break;
            tc_fence_after();
            const float *gt = (const float *)(sm + OFF_GATE + s * 1024);
            uint32_t kq[64];
            tmem_ld32(tl + TM_KQ, kq);
            tmem_ld32(tl + TM_KQ + 32, kq + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_KQE]);
            if (pt < 64) {
                const int r = pt;
                const float br = gt[64 + r];
                pG[r] = gt[r];
                float diag = 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    sL[r * 65 + j] = (j < r) ? br * u2f(kq[j]) : 0.f;
                    if (j == r) diag = u2f(kq[j]);
                }
                if (check_norm && br * diag > 2.0001f) atomicOr(status, kStatusNormBound);
            } else if (emit) {
                const int r = pt - 64;
                const float Gr = gt[r];
                uint8_t *prow = sm + OFF_P + b * 8192;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = 8 * q + u;
                        v[u] = (j <= r) ? a.scale * exp2f(Gr - gt[j]) * u2f(kq[j]) : 0.f;
                    }
                    uint4 pk;
                    pk.x = pack_bf16(v[0], v[1]);
                    pk.y = pack_bf16(v[2], v[3]);
                    pk.z = pack_bf16(v[4], v[5]);
                    pk.w = pack_bf16(v[6], v[7]);
                    *(uint4 *)(prow + sw128(r, 8 * q)) = pk;
                }
                fence_proxy_async();
            }
            bar_sync(1, 128);
            if (lane == 0) mbar_arrive(&bars[B_EMPTY + s]);  // gates copied; stage no longer read here

            // ---- inverse of the 16 x 16 diagonal blocks: 2 threads per (block, column)
            {
                const int task = pt >> 1, hh = pt & 1;
                const int bb = task >> 4, cc = task & 15;
                const int base = 16 * bb;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
                for (int r = 1; r < 16; ++r) {
                    float part = 0.f;
#pragma unroll
                    for (int j = hh; j < r; j += 2) part = fmaf(sL[(base + r) * 65 + base + j], x[j], part);
                    part += __shfl_xor_sync(0xffffffffu, part, 1);
                    if (r > cc) x[r] = -part;
                }
                if (hh == 0) {
#pragma unroll
                    for (int r = 0; r < 16; ++r) sX[(base + r) * 65 + base + cc] = x[r];
                }
            }
            bar_sync(1, 128);
            // ---- off-diagonal blocks, by distance from the diagonal:
            //      X_ab = -X_aa * sum_{m=b}^{a-1} L_am X_mb   (T kept in the unused upper blocks of L)
#pragma unroll 1
            for (int dist = 1; dist < 4; ++dist) {
                const int nblk = 4 - dist;
                for (int e = pt; e < nblk * 256; e += 128) {
                    const int blk = e >> 8, w = e & 255, r = w >> 4, cc = w & 15;
                    const int bcol = blk, arow = blk + dist;
                    float acc = 0.f;
                    for (int mb = bcol; mb < arow; ++mb)
#pragma unroll
                        for (int mm = 0; mm < 16; ++mm)
                            acc = fmaf(sL[(16 * arow + r) * 65 + 16 * mb + mm], sX[(16 * mb + mm) * 65 + 16 * bcol + cc], acc);
                    sL[(16 * bcol + r) * 65 + 16 * arow + cc] = acc;   // T stored at block (b, a)
                }
                bar_sync(1, 128);
                for (int e = pt; e < nblk * 256; e += 128) {
                    const int blk = e >> 8, w = e & 255, r = w >> 4, cc = w & 15;
                    const int bcol = blk, arow = blk + dist;
                    float acc = 0.f;
#pragma unroll
                    for (int mm = 0; mm < 16; ++mm)
                        acc = fmaf(sX[(16 * arow + r) * 65 + 16 * arow + mm], sL[(16 * bcol + mm) * 65 + 16 * arow + cc], acc);
                    sX[(16 * arow + r) * 65 + 16 * bcol + cc] = -acc;
                }
                bar_sync(1, 128);
            }
            // ---- A_g = Gam * X (lower incl. diagonal) -> bf16, 128-byte swizzled rows
            {
                const int r = pt >> 1, h = pt & 1;
                const float Gr = pG[r];
                uint8_t *arow = sm + OFF_A + b * 8192;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = 32 * h + 8 * q + u;
                        v[u] = (j <= r) ? exp2f(Gr - pG[j]) * sX[r * 65 + j] : 0.f;
                    }
                    uint4 pk;
                    pk.x = pack_bf16(v[0], v[1]);
                    pk.y = pack_bf16(v[2], v[3]);
                    pk.z = pack_bf16(v[4], v[5]);
                    pk.w = pack_bf16(v[6], v[7]);
                    *(uint4 *)(arow + sw128(r, 32 * h + 8 * q)) = pk;
                }
                fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_AF + b]);
            bar_sync(1, 128);  // sL / sX / pG are reused by the next chunk
        }
    } else if (warp >= 12) {
        // ================================================================ epilogue (lane = dv)
        const int et = tid - 384, dv = et;
        const int ew = warp - 12;
        const uint32_t tl = tb + ((uint32_t)((warp & 3) * 32) << 16);
        float *eg = (float *)(sm + OFF_EG) + ew * 64;
        uint8_t *ostage = sm + OFF_O;
        bool ok = true;
        int e = 0;
        for (int i = 0; i < nch && ok; ++i) {
            const int c = cs + i;
            if (!(fwd && c >= c0)) continue;
            const int64_t t0 = bos + (int64_t)c * kChunk;
            const int rows = rows_in(len, c);
            // scale * 2^G for this chunk, from the raw gates (independent of the stage ring)
            {
                const int r0 = 2 * lane, r1 = r0 + 1;
                const float g0 = r0 < rows ? a.g[(size_t)(t0 + r0) * HV + hv] * kRcpLn2 : 0.f;
                const float g1 = r1 < rows ? a.g[(size_t)(t0 + r1) * HV + hv] * kRcpLn2 : 0.f;
                float sp = g0 + g1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, sp, off);
                    if (lane >= off) sp += y;
                }
                eg[r0] = a.scale * exp2f(sp - g1);
                eg[r1] = a.scale * exp2f(sp);
                __syncwarp();
            }
            ok = mbar_wait(&bars[B_OF], e & 1, status, kStatusTimeout, kWaitNs);
            ok = bar_and(3, 128, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t ov[32];  // 64 bf16 of O^T row dv (packed pairs along the chunk)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r1[32], r2[32];
                tmem_ld32(tl + TM_O1 + 32 * h, r1);
                tmem_ld32(tl + TM_O2 + 32 * h, r2);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const int cc = 32 * h + j;
                    ov[16 * h + j / 2] = pack_bf16(eg[cc] * u2f(r1[j]) + u2f(r2[j]),
                                                   eg[cc + 1] * u2f(r1[j + 1]) + u2f(r2[j + 1]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_OE]);
            if (rows == kChunk) {
                if (et == 0) tma_store_wait_read0();
                bar_sync(3, 128);
                uint8_t *box = ostage + (dv >> 6) * 8192 + (dv & 63) * 2;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    *(uint16_t *)(box + (2 * j) * 128) = (uint16_t)(ov[j] & 0xFFFFu);
                    *(uint16_t *)(box + (2 * j + 1) * 128) = (uint16_t)(ov[j] >> 16);
                }
                fence_proxy_async();
                bar_sync(3, 128);
                if (et == 0) {
                    tma_store_3d(&m.o, ostage, 0, hv, (int)t0);
                    tma_store_3d(&m.o, ostage + 8192, 64, hv, (int)t0);
                    tma_store_commit();
                }
            } else {
                uint16_t *o = (uint16_t *)a.o;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    if (2 * jj < rows) o[((size_t)(t0 + 2 * jj) * HV + hv) * V + dv] = (uint16_t)(ov[jj] & 0xFFFFu);
                    if (2 * jj + 1 < rows) o[((size_t)(t0 + 2 * jj + 1) * HV + hv) * V + dv] = (uint16_t)(ov[jj] >> 16);
                }
            }
            ++e;
            __syncwarp();
        }
        if (et == 0) tma_store_wait0();
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    });
    return fn;
}

// 3-D map over a [rows, heads, 128] bf16 tensor, box = 64 elements x 1 head x 64 rows.
bool make_map(CUtensorMap *map, const void *base, int heads, int64_t rows, bool swizzle)
{
    auto enc = get_encoder();
    if (!enc || !base) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

size_t tc_smem_bytes() { return kSmemTC; }

bool tc_shape_ok(const gdn_shape *s)
{
    return s->qkv_dtype == GDN_BF16 && s->gate_kind == GDN_GATE_SCALAR && s->K == 128 && s->V == 128 &&
           (size_t)s->B * s->T < (1ull << 31);
}

bool tc_supported(const gdn_shape *s, const void *q, const void *k, const void *v, const void *o)
{
    if (!tc_shape_ok(s)) return false;
    auto al = [](const void *p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; };
    return al(q) && al(k) && al(v) && al(o) && get_encoder() != nullptr;
}

cudaError_t launch_tc_scan(const ScanArgs &a, int value_tiles, cudaStream_t st)
{
    if (a.N * a.HV == 0) return cudaSuccess;
    TcMaps maps;
    memset(&maps, 0, sizeof(maps));
    const int64_t rows = (int64_t)a.B * a.T;
    if (rows > 0) {
        if (!make_map(&maps.q, a.q, a.H, rows, true) || !make_map(&maps.k, a.k, a.H, rows, true) ||
            !make_map(&maps.v, a.v, a.HV, rows, true))
            return cudaErrorInvalidValue;
        if (a.mode == kModeForward && !make_map(&maps.o, a.o, a.HV, rows, false)) return cudaErrorInvalidValue;
    }
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(tc_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTC);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(value_tiles, a.n_seg, a.N * a.HV);
    tc_scan_kernel<<<grid, kThreadsTC, kSmemTC, st>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace gdn

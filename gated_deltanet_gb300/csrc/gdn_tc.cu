// Tensor-core engine (sm_103a: tcgen05 + TMEM + TMA) of the chunked gated
// delta rule for bf16 q/k/v, dk = dv = 128, scalar gate, C = 64.
//
// One CTA owns one (sequence, value head, segment) and walks its chunks
// serially.  The state is kept transposed, S^T [dv x dk] fp32, in tensor
// memory (lane = dv), so every product of the chunk step is an M = 128
// tcgen05 MMA with dv as M.  The chunk step is the FlashQLA restructured form
// (FlashQLA blog, "A balanced solution", step 3), with A0 from step 1:
//
//   A0    = (I + StrictLower(diag(beta) K K^T))^-1        (prep warps)
//   A_g   = Gam * A0,  P_g = scale Lower(Gam) * (Q K^T)    (prep / aux warps)
//   D^T   = S^T K^T - (V diag(1/gam))^T                    (MMA; the second term
//                                                            through a resident -I)
//   Y^T   = -D^T diag(beta gam) = (V^T - X^T diag(gam)) diag(beta)
//   V'^T  = Y^T A_g^T                                      (MMA)
//   O^T   = scale (S^T Q^T) diag(gam) + V'^T P_g^T         (MMA x2, output warps)
//   S^T  <- gC S^T + (V'^T diag(gC / gam)) K               (MMA, B = K MN-major)
//
// with G the chunk-local inclusive cumsum of the log-gate (kept in base 2),
// gam = 2^G, Gam_ij = 2^(G_i - G_j), gC = gam of the last valid row.  When a
// chunk decays by more than 2^-100 the 1/gam scaling is skipped and Y is
// formed from V directly.
//
// Warp roles (16 warps): 0 TMA producer (+ gate statistics), 1 MMA issuer,
// 2-3 aux (TMEM allocation, V / gam in place, P_g), 4-7 chain (state, Y,
// V'), 8-11 prep (K K^T -> L -> blockwise inverse), 12-15 output (A_g of
// the next chunk, then O of the previous one).
// All waits are bounded in wall time; a wait that runs out records a timeout
// in the status word and every role leaves its loop, so the kernel always
// ends and frees its tensor memory.
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
constexpr uint32_t OFF_NEGI = OFF_STAGE + 2 * kStageBytes;  // -I [128 x 128] bf16 SW128 (2 boxes of 16 KB)
constexpr uint32_t OFF_A = OFF_NEGI + 32768;                // A_g  [64 x 64] bf16 SW128, x2
constexpr uint32_t OFF_P = OFF_A + 2 * 8192;                // P_g  [64 x 64] bf16 SW128, x2
constexpr uint32_t OFF_VP = OFF_P + 2 * 8192;               // V'^T [128 x 64] bf16 SW128
constexpr int kLdX = 68;                                    // row pitch (floats) of the 64 x 64 fp32 tiles
constexpr uint32_t OFF_L = OFF_VP + 16384;                  // L  fp32 [64][68]
constexpr uint32_t OFF_X = OFF_L + 64 * kLdX * 4;           // X  fp32 [64][68]
constexpr uint32_t kGateBytes = 1536;  // per stage: G, beta, gam, 2^(G_C-G), 2^-G, -beta*gam  [64] f32 each
constexpr uint32_t OFF_GATE = OFF_X + 64 * kLdX * 4;
constexpr uint32_t OFF_PG = OFF_GATE + 2 * kGateBytes;      // prep copy: gam, rgam, G [3][64], flag
constexpr uint32_t OFF_SCR = OFF_PG + 1024;                 // prep per-warp scratch [4][256] f32
constexpr uint32_t OFF_EG = OFF_SCR + 4096;                 // scale * gam per chunk, ring of 8 [8][64]
constexpr uint32_t OFF_BAR = OFF_EG + 2048;
constexpr uint32_t kSmemTC = OFF_BAR + 256 + 1024;          // + slack for the 1024-byte alignment

// gate arrays inside a stage's gate block
constexpr int GT_G = 0, GT_BETA = 64, GT_GAM = 128, GT_RDEC = 192, GT_RGAM = 256, GT_NBG = 320;
constexpr float kFactorFloor = -100.f;  // chunks with G_C below this skip the 1/gam factorisations

// ---- tensor memory columns
constexpr uint32_t TM_S = 0, TM_XV = 128, TM_O1 = 192, TM_O2 = 256, TM_KQ = 320, TM_SBF = 384,
                   TM_YBF = 448, TM_VTB = 480;

enum Bar {
    B_FULL = 0, B_EMPTY = 2, B_TMA = 4, B_VH = 6, B_AF = 8, B_AE = 10, B_KQF = 12, B_KQE, B_SBF, B_XF, B_YF,
    B_VPF, B_VTF, B_SF, B_OF, B_OE, B_XR, B_XFREE, B_COUNT
};
constexpr uint32_t kEmptyArrivals = 1 + 4 + 4 + 2;  // MMA commit, chain, prep, aux warps
constexpr uint32_t kKqArrivals = 4 + 2;             // prep + aux warps read the K K^T / Q K^T tile
constexpr uint32_t kAfArrivals = 4 + 2;             // output warps write A_g, aux writes P_g

struct TcMaps {
    CUtensorMap q, k, v;
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

__device__ __forceinline__ uint32_t tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// d += A(16x8, row) * B(8x8, col) in tf32 with fp32 accumulation (one warp)
__device__ __forceinline__ void mma_tf32(float *d, float a0, float a1, float a2, float a3, float b0, float b1)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(tf32(a0)), "r"(tf32(a1)), "r"(tf32(a2)), "r"(tf32(a3)), "r"(tf32(b0)), "r"(tf32(b1)));
}

__device__ __forceinline__ uint64_t kmaj(uint32_t addr) { return sdesc_sw128(addr, 16, 1024); }

__device__ __forceinline__ uint4 pack8(const float *v)
{
    uint4 pk;
    pk.x = pack_bf16(v[0], v[1]);
    pk.y = pack_bf16(v[2], v[3]);
    pk.z = pack_bf16(v[4], v[5]);
    pk.w = pack_bf16(v[6], v[7]);
    return pk;
}

__global__ void __launch_bounds__(kThreadsTC, 1) tc_scan_kernel(const ScanArgs a, const __grid_constant__ TcMaps m)
{
    extern __shared__ __align__(1024) uint8_t smraw[];
    // 1024-byte aligned base (128-byte swizzle atoms); pointer arithmetic on the
    // __shared__ array keeps every derived access in the shared state space
    uint8_t *sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
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
    const bool zero_values = !fwd && vt == 1;   // pre-pass: the M columns carry no values
    const bool check_norm = fwd && a.warm_start != nullptr;

    if (tid == 0) {
        if (seg == a.n_seg - 1 && c1 < NT) atomicOr(a.status, kStatusPlan);
        if (fwd && a.warm_start && (a.warm_start[sidx] < 0 || a.warm_start[sidx] > c0))
            atomicOr(a.status, kStatusPlan);
        for (int j = 0; j < 2; ++j) {
            mbar_init(&bars[B_FULL + j], 1);
            mbar_init(&bars[B_EMPTY + j], kEmptyArrivals);
            mbar_init(&bars[B_TMA + j], 1);
            mbar_init(&bars[B_VH + j], 2);
            mbar_init(&bars[B_AF + j], kAfArrivals);
            mbar_init(&bars[B_AE + j], 1);
        }
        mbar_init(&bars[B_KQF], 1);
        mbar_init(&bars[B_KQE], kKqArrivals);
        mbar_init(&bars[B_SBF], 4);
        mbar_init(&bars[B_XF], 1);
        mbar_init(&bars[B_YF], 4);
        mbar_init(&bars[B_VPF], 1);
        mbar_init(&bars[B_VTF], 4);
        mbar_init(&bars[B_SF], 1);
        mbar_init(&bars[B_OF], 1);
        mbar_init(&bars[B_OE], 4);
        mbar_init(&bars[B_XR], 4);
        mbar_init(&bars[B_XFREE], 4);
        fence_mbar_init();
    }
    // the resident -I operand (K-major, 128-byte swizzle; two 64-column boxes)
    for (int e = tid; e < 128 * 16; e += kThreadsTC) {
        const int r = e >> 4, ch = e & 15, bx = ch >> 3, cl = ch & 7;
        uint4 z = make_uint4(0, 0, 0, 0);
        if ((r >> 6) == bx && ((r & 63) >> 3) == cl) {
            const uint32_t neg1 = 0xBF80u;  // bf16 -1.0
            const int w = (r & 7) >> 1;
            const uint32_t word = (r & 1) ? (neg1 << 16) : neg1;
            if (w == 0) z.x = word; else if (w == 1) z.y = word; else if (w == 2) z.z = word; else z.w = word;
        }
        *(uint4 *)(sm + OFF_NEGI + bx * 16384 + sw128(r, 8 * cl)) = z;
    }
    fence_proxy_async();
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
            // gate statistics while the tiles land: lane holds rows 2l, 2l+1; base-2 inclusive cumsum
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
            float *gt = (float *)(sm + OFF_GATE + s * kGateBytes);
            const float gm0 = exp2f(G0), gm1 = exp2f(G1);
            gt[GT_G + r0] = G0;
            gt[GT_G + r1] = G1;
            gt[GT_BETA + r0] = b0;
            gt[GT_BETA + r1] = b1;
            gt[GT_GAM + r0] = gm0;
            gt[GT_GAM + r1] = gm1;
            gt[GT_RDEC + r0] = exp2f(GC - G0);
            gt[GT_RDEC + r1] = exp2f(GC - G1);
            gt[GT_RGAM + r0] = exp2f(-G0);
            gt[GT_RGAM + r1] = exp2f(-G1);
            gt[GT_NBG + r0] = -b0 * gm0;
            gt[GT_NBG + r1] = -b1 * gm1;
            // output scales of this chunk; read by the output warps after x_ready of the chunk,
            // which the prep warps release after acquiring this stage (so the writes are visible)
            float *osc = (float *)(sm + OFF_EG) + (i & 7) * 64;
            osc[r0] = a.scale * gm0;
            osc[r1] = a.scale * gm1;
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
            const uint32_t negi = sbase + OFF_NEGI;
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
            // -(V diag(1/gam))^T of chunk j into the D region: needs no state, so it is issued
            // as soon as the previous chunk's V' has been read out of that region
            auto vhat_of = [&](int j) {
                const float *gt = (const float *)(sm + OFF_GATE + (j & 1) * kGateBytes);
                return !zero_values && gt[GT_G + 63] >= kFactorFloor;
            };
            auto issue_negv = [&](int j) -> bool {
                if (!vhat_of(j)) return true;
                if (!mbar_wait(&bars[B_VH + (j & 1)], (j >> 1) & 1, status, kStatusTimeout, kWaitNs)) return false;
                tc_fence_after();
                const uint32_t st = sbase + OFF_STAGE + (j & 1) * kStageBytes;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    const uint32_t voff = (ks >> 2) * 8192 + (ks & 3) * 32;
                    mma_ss(tb + TM_XV, kmaj(negi + off), kmaj(st + sV0 + voff), idN64, ks > 0);
                }
                return true;
            };
            if (ok) {
                tc_fence_after();
                issue_kq(0);
                ok = issue_negv(0);
            }
            int e = 0;
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i & 1, b = i & 1, c = cs + i;
                const bool emit = fwd && c >= c0;
                const uint32_t st = sbase + OFF_STAGE + s * kStageBytes;
                const bool vhat = vhat_of(i);
                ok = mbar_spin(&bars[B_SBF], i & 1, status, kStatusTimeout, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                // D^T (+)= S^T K^T
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_ts(tb + TM_XV, tb + TM_SBF + ks * 8, kmaj(st + sK0 + off), idN64, vhat || ks > 0);
                }
                mma_commit(&bars[B_XF]);
                // K K^T / Q K^T of the next chunk, so its preparation overlaps this chunk's chain
                if (i + 1 < nch) {
                    ok = mbar_wait(&bars[B_FULL + ((i + 1) & 1)], ((i + 1) >> 1) & 1, status, kStatusTimeout, kWaitNs) &&
                         mbar_wait(&bars[B_KQE], i & 1, status, kStatusTimeout, kWaitNs);
                    if (!ok) break;
                    tc_fence_after();
                    issue_kq(i + 1);
                }
                ok = mbar_spin(&bars[B_YF], i & 1, status, kStatusTimeout, kWaitNs) &&
                     mbar_spin(&bars[B_AF + b], (i >> 1) & 1, status, kStatusTimeout, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                // V'^T = Y^T A_g^T
                const uint32_t abuf = sbase + OFF_A + b * 8192;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ts(tb + TM_XV, tb + TM_YBF + ks * 8, kmaj(abuf + ks * 32), idN64, ks > 0);
                mma_commit(&bars[B_VPF]);
                if (emit) {
                    // O1^T = S^T Q^T, in the window where the chain converts V'
                    if (e > 0) ok = mbar_wait(&bars[B_OE], (e - 1) & 1, status, kStatusTimeout, kWaitNs);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                        mma_ts(tb + TM_O1, tb + TM_SBF + ks * 8, kmaj(st + sQ0 + off), idN64, ks > 0);
                    }
                }
                ok = mbar_spin(&bars[B_VTF], i & 1, status, kStatusTimeout, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                // S^T += (V'^T diag(gC/gam)) K   (B = K, MN-major: dk atoms 16 KB apart)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ts(tb + TM_S, tb + TM_VTB + ks * 8, sdesc_sw128(st + sK0 + ks * 2048, 16384, 1024),
                           idN128MN, 1);
                mma_commit(&bars[B_SF]);
                // the next chunk's -(V / gam)^T (its stage was waited for before K K^T above)
                if (i + 1 < nch && !issue_negv(i + 1)) {
                    ok = false;
                    break;
                }
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
            }
        }
    } else if (warp == 2 || warp == 3) {
        // ================================================================ aux: V / gam in place, P_g
        const int at = tid - 64;  // 0..63; TMEM lanes 64..127 = Q K^T rows
        const uint32_t tl = tb + ((uint32_t)((warp & 3) * 32) << 16);
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
            const int s = i & 1, b = i & 1, c = cs + i;
            const bool emit = fwd && c >= c0;
            ok = mbar_wait(&bars[B_FULL + s], (i >> 1) & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const float *gt = (const float *)(sm + OFF_GATE + s * kGateBytes);
            const bool factored = gt[GT_G + 63] >= kFactorFloor;
            if (!zero_values && factored) {
                // V <- V diag(2^-G): 16-byte pieces (8 values of one row c)
                uint8_t *st = sm + OFF_STAGE + s * kStageBytes;
#pragma unroll 4
                for (int p = at; p < 1024; p += 64) {
                    const int bx = p >> 9, w = p & 511, r = w >> 3;
                    uint4 *ptr = (uint4 *)(st + sV0 + bx * 8192 + w * 16);
                    uint4 x = *ptr;
                    const float f = gt[GT_RGAM + r];
                    __nv_bfloat162 *h2 = (__nv_bfloat162 *)&x;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float2 fv = __bfloat1622float2(h2[u]);
                        h2[u] = __floats2bfloat162_rn(fv.x * f, fv.y * f);
                    }
                    *ptr = x;
                }
                fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_VH + s]);  // every chunk, so the phases follow the stage uses
            // P_g row r = scale * Gam[r, j <= r] * (Q K^T)[r, j] -> bf16, 128-byte swizzled
            if (i >= 2) ok = mbar_wait(&bars[B_AE + b], ((i >> 1) - 1) & 1, status, kStatusTimeout, kWaitNs);
            if (ok) ok = mbar_wait(&bars[B_KQF], i & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            if (emit) {
                const int r = at;
                const float Gr = gt[GT_G + r], fr = a.scale * gt[GT_GAM + r];
                uint8_t *prow = sm + OFF_P + b * 8192;
#pragma unroll 1
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t kq[32];
                    tmem_ld32(tl + TM_KQ + 32 * hf, kq);
                    tmem_ld_wait();
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const int j0 = 32 * hf + 8 * qq;
                        const float4 rg0 = *(const float4 *)(gt + GT_RGAM + j0);
                        const float4 rg1 = *(const float4 *)(gt + GT_RGAM + j0 + 4);
                        const float rgv[8] = {rg0.x, rg0.y, rg0.z, rg0.w, rg1.x, rg1.y, rg1.z, rg1.w};
                        float v[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int j = j0 + u;
                            const float gij = factored ? fr * rgv[u] : a.scale * exp2f(Gr - gt[GT_G + j]);
                            v[u] = (j <= r) ? gij * u2f(kq[8 * qq + u]) : 0.f;
                        }
                        *(uint4 *)(prow + sw128(r, j0)) = pack8(v);
                    }
                }
                fence_proxy_async();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_KQE]);
                mbar_arrive(&bars[B_AF + b]);
                mbar_arrive(&bars[B_EMPTY + s]);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ================================================================ chain (lane = dv)
        const int dv = tid - 128;
        const uint32_t tl = tb + ((uint32_t)((warp & 3) * 32) << 16);
        const float *init = nullptr;
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
            if (ok && i > 0) ok = mbar_spin(&bars[B_SF], (i - 1) & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const float *gt = (const float *)(sm + OFF_GATE + s * kGateBytes);
            const float dec = gt[GT_GAM + 63];  // gC = 2^G_C
            const bool vhat = !zero_values && gt[GT_G + 63] >= kFactorFloor;
            // ---- S_i -> bf16 copy (MMA operand) and gC * S_i (accumulator of this chunk's update)
#pragma unroll 1
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t r[32], p[16];
                if (i == 0) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int d = 32 * q4 + j;
                        float x = 0.f;
                        if (init) x = init[(size_t)d * V + dv];
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
            ok = mbar_spin(&bars[B_XF], i & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            {
                const uint8_t *vbox = sm + OFF_STAGE + s * kStageBytes + (dv < 64 ? sV0 : sV1);
                const int dl = dv & 63;
                uint32_t rr[2][32];
                tmem_ld32(tl + TM_XV, rr[0]);
                tmem_ld32(tl + TM_XV + 32, rr[1]);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t *r = rr[h];
                    uint32_t y[16];
                    if (vhat) {
                        // the tensor core already formed X^T - (V diag(1/gam))^T: Y = -beta gam (that)
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const float4 nb = *(const float4 *)(gt + GT_NBG + 32 * h + 4 * j4);
                            y[2 * j4] = pack_bf16(nb.x * u2f(r[4 * j4 + 0]), nb.y * u2f(r[4 * j4 + 1]));
                            y[2 * j4 + 1] = pack_bf16(nb.z * u2f(r[4 * j4 + 2]), nb.w * u2f(r[4 * j4 + 3]));
                        }
                    } else {
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const int cc = 32 * h + 4 * j4;
                            const float4 bt = *(const float4 *)(gt + GT_BETA + cc);
                            const float4 gm = *(const float4 *)(gt + GT_GAM + cc);
                            float v[4] = {0.f, 0.f, 0.f, 0.f};
                            if (!zero_values) {
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    v[u] = __bfloat162float(*(const __nv_bfloat16 *)(vbox + sw128(cc + u, dl)));
                            }
                            y[2 * j4] = pack_bf16(bt.x * (v[0] - gm.x * u2f(r[4 * j4 + 0])),
                                                  bt.y * (v[1] - gm.y * u2f(r[4 * j4 + 1])));
                            y[2 * j4 + 1] = pack_bf16(bt.z * (v[2] - gm.z * u2f(r[4 * j4 + 2])),
                                                      bt.w * (v[3] - gm.w * u2f(r[4 * j4 + 3])));
                        }
                    }
                    tmem_st16(tl + TM_YBF + 16 * h, y);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_YF]);

            // ---- V'^T -> bf16 (output operand, smem) and V'^T diag(gC/gam) (state operand, TMEM)
            ok = mbar_spin(&bars[B_VPF], i & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            {
                uint8_t *vprow = sm + OFF_VP;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    uint32_t r[32], vtl[16];
                    tmem_ld32(tl + TM_XV + 32 * h, r);
                    tmem_ld_wait();
                    float4 rd[8];
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) rd[j4] = *(const float4 *)(gt + GT_RDEC + 32 * h + 4 * j4);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        vtl[2 * j4] = pack_bf16(u2f(r[4 * j4 + 0]) * rd[j4].x, u2f(r[4 * j4 + 1]) * rd[j4].y);
                        vtl[2 * j4 + 1] = pack_bf16(u2f(r[4 * j4 + 2]) * rd[j4].z, u2f(r[4 * j4 + 3]) * rd[j4].w);
                    }
                    tmem_st16(tl + TM_VTB + 16 * h, vtl);
                    if (emit) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float f[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) f[u] = u2f(r[8 * q + u]);
                            *(uint4 *)(vprow + sw128(dv, 32 * h + 8 * q)) = pack8(f);
                        }
                    }
                }
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
                    if (init) x = init[(size_t)d * V + dv];
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
        // ================================================================ prep (lane = row of K K^T)
        const int pt = tid - 256, pw = warp - 8;
        const uint32_t tl = tb + ((uint32_t)((warp & 3) * 32) << 16);
        float *sL = (float *)(sm + OFF_L);
        float *sX = (float *)(sm + OFF_X);
        float *pG = (float *)(sm + OFF_PG);               // gam, rgam, G of the chunk being prepared
        float *scr = (float *)(sm + OFF_SCR) + pw * 256;  // per-warp scratch for the block products
        const int g = lane >> 2, tg = lane & 3;
        bool ok = true;
        for (int i = 0; i < nch && ok; ++i) {
            const int s = i & 1;
            ok = mbar_wait(&bars[B_FULL + s], (i >> 1) & 1, status, kStatusTimeout, kWaitNs);
            if (ok) ok = mbar_wait(&bars[B_KQF], i & 1, status, kStatusTimeout, kWaitNs);
            ok = bar_and(1, 128, ok);
            if (!ok) break;
            tc_fence_after();
            const float *gt = (const float *)(sm + OFF_GATE + s * kGateBytes);
            const float factored = gt[GT_G + 63] >= kFactorFloor ? 1.f : 0.f;
            float pg_gam = 0.f, pg_rgam = 0.f, pg_G = 0.f;
            if (pt < 64) {
                // L row r = beta_r * (K K^T)[r, j < r]   (gate-free: the gates enter as Gam * A0)
                const int r = pt;
                const float br = gt[GT_BETA + r];
                pg_gam = gt[GT_GAM + r];
                pg_rgam = gt[GT_RGAM + r];
                pg_G = gt[GT_G + r];
                float diag = 0.f;
#pragma unroll 1
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t kq[32];
                    tmem_ld32(tl + TM_KQ + 32 * hf, kq);
                    tmem_ld_wait();
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const int j = 32 * hf + 4 * j4;
                        float4 w;
                        w.x = (j + 0 < r) ? br * u2f(kq[4 * j4 + 0]) : 0.f;
                        w.y = (j + 1 < r) ? br * u2f(kq[4 * j4 + 1]) : 0.f;
                        w.z = (j + 2 < r) ? br * u2f(kq[4 * j4 + 2]) : 0.f;
                        w.w = (j + 3 < r) ? br * u2f(kq[4 * j4 + 3]) : 0.f;
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            if (j + u == r) diag = u2f(kq[4 * j4 + u]);
                        *(float4 *)(sL + r * kLdX + j) = w;
                    }
                }
                if (check_norm && br * diag > 2.0001f) atomicOr(status, kStatusNormBound);
            }
            tc_fence_before();
            bar_sync(1, 128);
            if (lane == 0) {
                mbar_arrive(&bars[B_KQE]);
                mbar_arrive(&bars[B_EMPTY + s]);  // gates copied; stage no longer read here
            }
            // X / gate copies of the previous chunk must have been turned into A_g
            if (i >= 1) ok = mbar_wait(&bars[B_XFREE], (i - 1) & 1, status, kStatusTimeout, kWaitNs);
            ok = bar_and(1, 128, ok);
            if (!ok) break;
            if (pt < 64) {
                pG[pt] = pg_gam;
                pG[64 + pt] = pg_rgam;
                pG[128 + pt] = pg_G;
                if (pt == 0) pG[192] = factored;
            }

            // ---- (I + L_bb)^-1 for the four 16 x 16 diagonal blocks: 2 threads per (block, column)
            {
                const int task = pt >> 1, hh = pt & 1;
                const int bb = task >> 4, cc = task & 15;
                const int base = 16 * bb;
                const float *Lb = sL + base * kLdX + base;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
                for (int r = 1; r < 16; ++r) {
                    float part = 0.f;
#pragma unroll
                    for (int j = 0; j < r; ++j)
                        if ((j & 1) == hh) part = fmaf(Lb[r * kLdX + j], x[j], part);
                    part += __shfl_xor_sync(0xffffffffu, part, 1);
                    if (r > cc) x[r] = -part;
                }
                float *Xb = sX + base * kLdX + base;
                if (hh == 0) {
#pragma unroll
                    for (int r = 0; r < 16; ++r) Xb[r * kLdX + cc] = x[r];
                } else if (bb == 0 || bb == 2) {
                    // zero the strictly upper 16 x 16 blocks that the 32 x 32 merge reads
#pragma unroll
                    for (int r = 0; r < 16; ++r) Xb[r * kLdX + 16 + cc] = 0.f;
                }
            }
            bar_sync(1, 128);
            // ---- exact block merges (16 -> 32 -> 64), tf32 tensor-core products (the result is
            //      rounded to bf16 for the MMA operand, well above tf32's rounding):
            //      [[A00, 0], [A10, A11]]^-1 = [[X00, 0], [-X11 A10 X00, X11]]
            {
                // 16 -> 32: warps 0,1 merge blocks (1,0); warps 2,3 merge (3,2); one 8-column tile each
                const int ra = (pw >> 1) ? 3 : 1, rb = ra - 1, nt = pw & 1;
                float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const float *Lr = sL + (16 * ra) * kLdX + 16 * rb + 8 * ks;
                    const float *Xr = sX + (16 * rb + 8 * ks) * kLdX + 16 * rb + 8 * nt;
                    mma_tf32(t, Lr[g * kLdX + tg], Lr[(g + 8) * kLdX + tg], Lr[g * kLdX + tg + 4],
                               Lr[(g + 8) * kLdX + tg + 4], Xr[tg * kLdX + g], Xr[(tg + 4) * kLdX + g]);
                }
                scr[g * 8 + 2 * tg] = t[0];
                scr[g * 8 + 2 * tg + 1] = t[1];
                scr[(g + 8) * 8 + 2 * tg] = t[2];
                scr[(g + 8) * 8 + 2 * tg + 1] = t[3];
                __syncwarp();
                float u4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const float *Xa = sX + (16 * ra) * kLdX + 16 * ra + 8 * ks;
                    mma_tf32(u4, Xa[g * kLdX + tg], Xa[(g + 8) * kLdX + tg], Xa[g * kLdX + tg + 4],
                               Xa[(g + 8) * kLdX + tg + 4], scr[(8 * ks + tg) * 8 + g], scr[(8 * ks + tg + 4) * 8 + g]);
                }
                float *dst = sX + (16 * ra) * kLdX + 16 * rb + 8 * nt;
                dst[g * kLdX + 2 * tg] = -u4[0];
                dst[g * kLdX + 2 * tg + 1] = -u4[1];
                dst[(g + 8) * kLdX + 2 * tg] = -u4[2];
                dst[(g + 8) * kLdX + 2 * tg + 1] = -u4[3];
            }
            bar_sync(1, 128);
            {
                // 32 -> 64: X[32:64, 0:32] = -X[32:64, 32:64] * (L[32:64, 0:32] * X[0:32, 0:32]); warp = 8-column tile
                const int nt = pw;
                float t[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const float *Xr = sX + (8 * ks) * kLdX + 8 * nt;
                    const float b0 = Xr[tg * kLdX + g], b1 = Xr[(tg + 4) * kLdX + g];
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        const float *Lr = sL + (32 + 16 * mt) * kLdX + 8 * ks;
                        mma_tf32(t[mt], Lr[g * kLdX + tg], Lr[(g + 8) * kLdX + tg], Lr[g * kLdX + tg + 4],
                                   Lr[(g + 8) * kLdX + tg + 4], b0, b1);
                    }
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    scr[(16 * mt + g) * 8 + 2 * tg] = t[mt][0];
                    scr[(16 * mt + g) * 8 + 2 * tg + 1] = t[mt][1];
                    scr[(16 * mt + g + 8) * 8 + 2 * tg] = t[mt][2];
                    scr[(16 * mt + g + 8) * 8 + 2 * tg + 1] = t[mt][3];
                }
                __syncwarp();
                float u4[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const float b0 = scr[(8 * ks + tg) * 8 + g], b1 = scr[(8 * ks + tg + 4) * 8 + g];
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt) {
                        const float *Xa = sX + (32 + 16 * mt) * kLdX + 32 + 8 * ks;
                        mma_tf32(u4[mt], Xa[g * kLdX + tg], Xa[(g + 8) * kLdX + tg], Xa[g * kLdX + tg + 4],
                                   Xa[(g + 8) * kLdX + tg + 4], b0, b1);
                    }
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    float *dst = sX + (32 + 16 * mt) * kLdX + 8 * nt;
                    dst[g * kLdX + 2 * tg] = -u4[mt][0];
                    dst[g * kLdX + 2 * tg + 1] = -u4[mt][1];
                    dst[(g + 8) * kLdX + 2 * tg] = -u4[mt][2];
                    dst[(g + 8) * kLdX + 2 * tg + 1] = -u4[mt][3];
                }
            }
            bar_sync(1, 128);
            // X (and the gate copies) are ready for the output warps, which form A_g
            if (lane == 0) mbar_arrive(&bars[B_XR]);
        }
    } else {
        // ================================================================ output (lane = dv)
        const int et = tid - 384, dv = et;
        const uint32_t tl = tb + ((uint32_t)((warp & 3) * 32) << 16);
        const float *sX = (const float *)(sm + OFF_X);
        const float *pG = (const float *)(sm + OFF_PG);
        bool ok = true;
        int e = 0;
        for (int it = 0; it <= nch && ok; ++it) {
            if (it < nch) {
                // ---- A_g = Gam * X (lower incl. diagonal) -> bf16, 128-byte swizzled rows, for chunk it
                const int b = it & 1;
                ok = mbar_wait(&bars[B_XR], it & 1, status, kStatusTimeout, kWaitNs);
                if (ok && it >= 2) ok = mbar_wait(&bars[B_AE + b], ((it >> 1) - 1) & 1, status, kStatusTimeout, kWaitNs);
                ok = bar_and(3, 128, ok);
                if (!ok) break;
                const int r = et >> 1, h = et & 1;
                const bool factored = pG[192] != 0.f;
                const float gr = pG[r], Gr = pG[128 + r];
                uint8_t *arow = sm + OFF_A + b * 8192;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int j0 = 32 * h + 8 * q;
                    const float4 x0 = *(const float4 *)(sX + r * kLdX + j0);
                    const float4 x1 = *(const float4 *)(sX + r * kLdX + j0 + 4);
                    const float4 rg0 = *(const float4 *)(pG + 64 + j0);
                    const float4 rg1 = *(const float4 *)(pG + 64 + j0 + 4);
                    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    const float rgv[8] = {rg0.x, rg0.y, rg0.z, rg0.w, rg1.x, rg1.y, rg1.z, rg1.w};
                    float v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = j0 + u;
                        const float gij = factored ? gr * rgv[u] : exp2f(Gr - pG[128 + j]);
                        v[u] = (j <= r) ? gij * xv[u] : 0.f;
                    }
                    *(uint4 *)(arow + sw128(r, j0)) = pack8(v);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars[B_AF + b]);
                    mbar_arrive(&bars[B_XFREE]);
                }
            }
            if (it < 1) continue;
            // ---- O of chunk it - 1
            const int c = cs + it - 1;
            if (!(fwd && c >= c0)) continue;
            const int64_t t0 = bos + (int64_t)c * kChunk;
            const int rows = rows_in(len, c);
            const float *eg = (const float *)(sm + OFF_EG) + ((it - 1) & 7) * 64;  // scale * 2^G of the chunk
            ok = mbar_wait(&bars[B_OF], e & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            __nv_bfloat16 *og = (__nv_bfloat16 *)a.o + ((size_t)t0 * HV + hv) * V + dv;
            const size_t ostride = (size_t)HV * V;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t r1[32], r2[32];
                tmem_ld32(tl + TM_O1 + 32 * h, r1);
                tmem_ld32(tl + TM_O2 + 32 * h, r2);
                tmem_ld_wait();
                if (h == 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_OE]);  // O regions drained
                }
                float ov[32];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 e4 = *(const float4 *)(eg + 32 * h + 4 * j4);
                    ov[4 * j4 + 0] = e4.x * u2f(r1[4 * j4 + 0]) + u2f(r2[4 * j4 + 0]);
                    ov[4 * j4 + 1] = e4.y * u2f(r1[4 * j4 + 1]) + u2f(r2[4 * j4 + 1]);
                    ov[4 * j4 + 2] = e4.z * u2f(r1[4 * j4 + 2]) + u2f(r2[4 * j4 + 2]);
                    ov[4 * j4 + 3] = e4.w * u2f(r1[4 * j4 + 3]) + u2f(r2[4 * j4 + 3]);
                }
                if (rows == kChunk) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) og[(size_t)(32 * h + j) * ostride] = __float2bfloat16_rn(ov[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (32 * h + j < rows) og[(size_t)(32 * h + j) * ostride] = __float2bfloat16_rn(ov[j]);
                }
            }
            ++e;
            __syncwarp();
        }
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

// 3-D map over a [rows, heads, 128] bf16 tensor, box = 64 elements x 1 head x 64 rows, 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, int heads, int64_t rows)
{
    auto enc = get_encoder();
    if (!enc || !base) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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
    static_assert(kSmemTC <= 227 * 1024, "shared memory budget");
    if (a.N * a.HV == 0) return cudaSuccess;
    TcMaps maps;
    memset(&maps, 0, sizeof(maps));
    const int64_t rows = (int64_t)a.B * a.T;
    if (rows > 0) {
        if (!make_map(&maps.q, a.q, a.H, rows) || !make_map(&maps.k, a.k, a.H, rows) ||
            !make_map(&maps.v, a.v, a.HV, rows))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(tc_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTC);
    if (e != cudaSuccess) return e;
    dim3 grid(value_tiles, a.n_seg, a.N * a.HV);
    tc_scan_kernel<<<grid, kThreadsTC, kSmemTC, st>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace gdn

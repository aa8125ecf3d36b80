// Tensor-core engine (sm_103a: tcgen05 + TMEM + TMA) of the chunked gated
// delta rule for bf16 q/k/v, dk = dv = 128, scalar gate, C = 64: the serial scan.
//
// One CTA owns one (sequence, value head, segment) and walks its chunks
// serially.  The state is kept transposed, S^T [dv x dk] fp32, in tensor
// memory (lane = dv), so every product is an M = 128 tcgen05 MMA.  Per chunk
// (G = chunk-local inclusive cumsum of the log-gate in base 2, gam = 2^G,
// Gam_ij = 2^(G_i - G_j), gC = gam of the last row), with the operand tiles
// T_U = A_g diag(beta) and T_W = A_g diag(beta gam) of tc_prep_kernel
// (A_g = Gam * (I + StrictLower(diag(beta) K K^T))^-1, FlashQLA blog, step 1):
//
//   U    = T_U V,  W = T_W K                             WY form (FLA page, sec. 4)
//   V'   = U - W S                                       the only state-dependent product
//   O    = Q~ S + P V',  Q~ = diag(scale gam) Q,  P = scale Lower(Gam) * (Q K^T)
//   S   <- gC S + K^T diag(gC / gam) V'
//
// With Gam_ij = gam_i / gam_j the output factors as
//   O = diag(scale gam) (Q S + (Lower(Q K^T) / gC) (diag(gC / gam) V'))
// so the products take the raw Q, an unscaled causal mask of Q K^T and the
// same gC/gam-scaled V' as the state update, and the O epilogue applies the row
// factors.  2^-G_C must then be finite: a chunk whose decay passes 2^-100
// takes the direct form (Q~ in place, P with its per-entry powers, unscaled V').
//
// The serial chain per chunk is: S -> bf16 copy, one MMA group
// (V'^T = U^T - S^T W^T), V' -> bf16, one MMA group (the state update).
//
// Warp roles (16 warps): 0 TMA producer (q, k, v boxes and the two tiles) + gate
// statistics (and the warmup start), 1 MMA issuer (a fixed program per chunk),
// 2-3 aux (P; Q~ in place for steep chunks), 4-11 chain (state copy, V'; two warps per 32-lane
// slice of tensor memory, each converting half of the columns), 12-15 output
// (W^T -> shared memory, O epilogue).  Every role batches its shared-memory
// loads ahead of the arithmetic: with one or two warps of a role per scheduler,
// a role's speed is its dependency latency, not its instruction count.
// Every wait is bounded in wall time; a wait that runs out records a timeout
// in the status word and the roles leave their loops, so the kernel always
// ends, waits for its copies and products in flight and frees its tensor memory.
#include "gdn_internal.cuh"
#include "gdn_ptx.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace gdn {
namespace {
using namespace ptx;

constexpr int kThreadsTC = 512;
constexpr int kStages = 3;

// ---- shared memory map (bytes from a 1024-aligned base)
// stage: K0 | Q0 | K1 | Q1 | V0 | V1 | T_U | T_W, 8 KB each (64 rows x 64 bf16, 128-byte swizzle).
// Per-channel gates (KDA): K^0 | Q~0 | K^1 | Q~1 | U0 | U1 | -W0 | -W1 | P, the preparation's boxes
// in the same places (and P after them).
constexpr uint32_t sK0 = 0, sQ0 = 8192, sK1 = 16384, sQ1 = 24576, sV0 = 32768, sV1 = 40960, sTU = 49152,
                   sTW = 57344, sKdaP = 65536;
constexpr uint32_t OFF_STAGE = 0;
// gate statistics per chunk: G, raw log-gate, gam, 2^(G_C-G), 2^-G, scale*gam  [64] f32 each (KDA:
// 2^G_C of the 128 channels).  A ring of four: the O epilogue of chunk c still reads its row
// factors while chunk c + 3 is loaded
constexpr int kGateStages = 4;
template <bool ACT>
constexpr uint32_t kGateBytesOf = ACT ? 2048u : 1536u;  // + 1/||k||, 1/||q|| with in-kernel activations
template <bool KDA, bool ACT>
struct TcLayout {
    static constexpr uint32_t kGateBytes = kGateBytesOf<ACT>;
    static constexpr uint32_t kStageBytes = KDA ? 73728u : 65536u;
    static constexpr uint32_t OFF_P = OFF_STAGE + kStages * kStageBytes;  // P [64 x 64] bf16 (scalar gate)
    static constexpr uint32_t OFF_WS = OFF_P + (KDA ? 0u : 8192u);         // -W^T [128 (dk) x 64] bf16, MN-major
    static constexpr uint32_t OFF_GATE = OFF_WS + (KDA ? 0u : 16384u);
    static constexpr uint32_t OFF_BAR = OFF_GATE + kGateStages * kGateBytes;
    static constexpr uint32_t kSmem = OFF_BAR + 512 + 1024;  // + slack for the 1024-byte alignment
};

// gate arrays inside a stage's gate block
constexpr int GT_G = 0, GT_GRAW = 64, GT_GAM = 128, GT_RDEC = 192, GT_GINV = 256, GT_SGAM = 320,
              GT_RK = 384, GT_RQ = 448;  // in-kernel L2 norm: 1 / ||k_t||, 1 / ||q_t|| (both from the preparation)
// G_C >= this: Gam_ij = gam_i * 2^-G_j with every factor inside the fp32 range
constexpr float kFactorFloor = -100.f;

// ---- tensor memory columns (512 allocated)
constexpr uint32_t TM_S = 0, TM_VP = 128, TM_O = 192, TM_W = 256, TM_SBF = 320, TM_VB = 384, TM_VTB = 416,
                   TM_KQ = 448;

enum Bar {
    B_TMA = 0, B_FULL = 3, B_EMPTY = 6, B_QS = 9, B_KQF = 12, B_KQE, B_WF, B_SBF, B_VPF, B_VTF, B_SF, B_PF,
    B_OF, B_OE, B_FIN, B_COUNT
};
static_assert(B_COUNT * 8 + 16 <= 512, "barrier block");  // + TMEM slot, cs, c0, c1

struct TcMaps {
    CUtensorMap q, k, v, o, tiles;
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

__device__ __forceinline__ int rows_in(int64_t len, int c)
{
    const int64_t r = len - (int64_t)c * kChunk;
    return r < kChunk ? (int)r : kChunk;
}

__device__ __forceinline__ uint64_t kmaj(uint32_t addr) { return sdesc_sw128(addr, 16, 1024); }

// true on one lane of a converged warp (the MMA issue of the warp)
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred = 0;
    asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n" : "=r"(pred));
    return pred != 0;
}


// Warmup start of a segment beginning at chunk c0: walk back over whole chunks,
// adding their log2-decays, until the window has decayed to log2_eps or below;
// the chunk where that happens is the start.  If the sequence start is reached
// first, start there (the exact prefix).  One warp; lane l sums tokens l and
// l + 32 of a chunk, eight chunks per round trip to memory.
template <bool ACT>
__device__ __noinline__ int warm_start_of(const float *g, int64_t bos, int64_t len, int HV, int hv, int c0,
                                          float log2_eps, const Act &act)
{
    const int lane = threadIdx.x & 31;
    // the head's activation parameters, taken once
    const float ea = ACT && act.A_log ? expf(act.A_log[hv]) : 0.f;
    const float bias = ACT && act.A_log && act.dt_bias ? act.dt_bias[hv] : 0.f;
    float acc = 0.f;
    for (int c = c0; c > 0; c -= 8) {
        // lane l: tokens l and l + 32 of the chunks c - 1, ..., c - 8 (loads issued together)
        float v[16];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const int cc = c - 1 - b;
            const int rows = cc >= 0 ? rows_in(len, cc) : 0;
            const float *gp = g + ((size_t)(bos + (int64_t)(cc >= 0 ? cc : 0) * kChunk) + lane) * HV + hv;
            v[2 * b] = lane < rows ? gp[0] : 0.f;
            v[2 * b + 1] = lane + 32 < rows ? gp[(size_t)32 * HV] : 0.f;
        }
        if constexpr (ACT) {
            if (act.A_log) {
                // raw gate input: the activation once every load of the round is issued (rows past the end
                // stay 0)
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const int cc = c - 1 - b;
                    const int rows = cc >= 0 ? rows_in(len, cc) : 0;
                    if (lane < rows) v[2 * b] = act_gate_pre(act, v[2 * b], bias, ea);
                    if (lane + 32 < rows) v[2 * b + 1] = act_gate_pre(act, v[2 * b + 1], bias, ea);
                }
            }
        }
#pragma unroll 1
        for (int b = 0; b < 8 && c - 1 - b >= 0; ++b) {
            float part = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q == b) part = v[2 * q] + v[2 * q + 1];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
            acc += part * kRcpLn2;
            if (acc <= log2_eps) return c - 1 - b;
        }
    }
    return 0;
}

// The same walk for per-channel gates over the preparation's bound of each chunk's log2-decay
// (wdec[slot * HV + hv], slot = slot0 + chunk): one warp, lane l takes chunk c - 1 - l, 32 chunks
// per round trip; an inclusive sum over the lanes finds the first chunk where the window reaches
// log2_eps.
__device__ __noinline__ int warm_start_chunks(const float *wdec, int64_t slot0, int HV, int hv, int c0, float log2_eps)
{
    const int lane = threadIdx.x & 31;
    float acc = 0.f;
    for (int c = c0; c > 0; c -= 32) {
        const int cc = c - 1 - lane;
        float v = cc >= 0 ? wdec[(size_t)(slot0 + cc) * HV + hv] : 0.f;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, cc >= 0 && acc + v <= log2_eps);
        if (hit) return c - __ffs(hit);
        acc += __shfl_sync(0xffffffffu, v, 31);
    }
    return 0;
}

template <bool KDA, bool ACT, bool DUMP = false>
__global__ void __launch_bounds__(kThreadsTC, 1) tc_scan_kernel(const ScanArgs a, const __grid_constant__ TcMaps m)
{
    // ACT: the in-kernel input activations (raw gate input, L2 norm of q and k); a separate instance, so
    // that the plain one carries none of their code.  DUMP: also write the state entering every chunk
    // (a.chunk_states, for the backward pass), in an instance of its own for the same reason.
    using Lay = TcLayout<KDA, ACT>;
    constexpr uint32_t kGateBytes = Lay::kGateBytes;
    const float *const rkp = ACT ? a.rk : nullptr;
    const bool nrm = ACT && a.act.qk_l2norm;
    const float *const rqp = nrm ? a.rq : nullptr;  // 1 / ||q_t|| from the preparation
    constexpr uint32_t kStageBytes = Lay::kStageBytes, OFF_P = Lay::OFF_P, OFF_WS = Lay::OFF_WS,
                       OFF_GATE = Lay::OFF_GATE, OFF_BAR = Lay::OFF_BAR;
    extern __shared__ __align__(1024) uint8_t smraw[];
    // 1024-byte aligned base (128-byte swizzle atoms); pointer arithmetic on the
    // __shared__ array keeps every derived access in the shared state space
    uint8_t *sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t *bars = (uint64_t *)(sm + OFF_BAR);
    uint32_t *tslot = (uint32_t *)(sm + OFF_BAR + 8 * B_COUNT);
    int *s_cs = (int *)(sm + OFF_BAR + 8 * B_COUNT + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int vt = blockIdx.x, seg = blockIdx.y, pair = blockIdx.z;
    const int HV = a.HV, V = a.V;
    const int n = a.seq_order ? a.seq_order[pair / HV] : pair / HV, hv = pair % HV, hq = hv / (HV / a.H);
    int64_t bos, len;
    if (a.cu_seqlens) {
        bos = a.cu_seqlens[n];
        len = a.cu_seqlens[n + 1] - bos;
    } else {
        bos = (int64_t)n * a.T;
        len = a.T;
    }
    const int NT = (int)((len + kChunk - 1) / kChunk);
    if (seg > 0 && seg * a.seg_chunks >= NT) return;
    const bool fwd = a.mode == kModeForward;
    const size_t sidx = ((size_t)n * HV + hv) * a.n_seg + seg;
    const bool zero_values = !fwd && vt == 1;   // pre-pass: the M columns carry no values

    if (warp == 0) {
        int c0 = seg * a.seg_chunks, c1 = min(c0 + a.seg_chunks, NT), cs = c0;
        if (fwd && a.warm_in_kernel) {
            // Warmup split with balanced segments: the boundary at nominal chunk c moves to
            // c + w / 4, w = c - (warmup start of c) capped at a segment, so that the segment after
            // it (which also scans its warmup) and the one before do about equal work: a warmup chunk
            // costs about half an emitted one (no q, no output products, no P, no O epilogue).
            const int L = a.seg_chunks;
            // per-channel gates: the preparation's per-chunk bounds; scalar gates: the gates themselves
            auto start = [&](int c) -> int {
                if constexpr (KDA)
                    return warm_start_chunks(a.kda_wdec, tile_slot(bos, n, 0), HV, hv, c, a.warm_log2_eps);
                else
                    return warm_start_of<ACT>(a.g, bos, len, HV, hv, c, a.warm_log2_eps, a.act);
            };
            auto bnd = [&](int j) -> int {
                const int cj = j * L;
                if (j == 0) return 0;
                if (cj >= NT) return NT;
                const int w = cj - start(cj);
                return min(cj + (min(w, L) + 2) / 4, NT);
            };
            c0 = bnd(seg);
            c1 = bnd(seg + 1);
            if (seg > 0) cs = start(c0);
        } else if (fwd && seg > 0) {
            if (a.warm_start) {
                cs = a.warm_start[sidx];
                if (cs < 0 || cs > c0) {
                    if (lane == 0) atomicOr(a.status, kStatusPlan);
                    cs = 0;
                }
            }
        }
        if (lane == 0) {
            s_cs[0] = cs;
            s_cs[1] = c0;
            s_cs[2] = c1;
            if (seg == a.n_seg - 1 && c1 < NT) atomicOr(a.status, kStatusPlan);
        }
    }
    if (tid == 32) {
        for (int j = 0; j < kStages; ++j) {
            mbar_init(&bars[B_TMA + j], 1);
            mbar_init(&bars[B_FULL + j], 1);
            mbar_init(&bars[B_EMPTY + j], 2);  // the issuer's commit and the output warps' O store
            mbar_init(&bars[B_QS + j], 2);
        }
        mbar_init(&bars[B_KQF], 1);
        mbar_init(&bars[B_KQE], 2);
        mbar_init(&bars[B_WF], 1);
        mbar_init(&bars[B_SBF], KDA ? 8 : 12);  // the chain warps' state copy (+ the output warps' -W^T)
        mbar_init(&bars[B_VPF], 1);
        mbar_init(&bars[B_VTF], 8);
        mbar_init(&bars[B_SF], 1);
        mbar_init(&bars[B_PF], 2);
        mbar_init(&bars[B_OF], 1);
        mbar_init(&bars[B_OE], 4);
        mbar_init(&bars[B_FIN], 1);
        fence_mbar_init();
    }
    if (warp == 2) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tslot;
    const int cs = s_cs[0], c0 = s_cs[1], c1 = s_cs[2];
    const int nch = c1 - cs;
    unsigned *status = a.status;
    const uint64_t kWaitNs = a.wait_ns;  // every wait gives up after this long (wall clock)
    auto gates = [&](int i) { return (float *)(sm + OFF_GATE + (i % kGateStages) * kGateBytes); };
    // factored output form (see the header): the chunk's decay 2^-G_C is finite
    auto factored = [&](int i) { return gates(i)[GT_G + 63] >= kFactorFloor; };
    auto emit_of = [&](int i) { return fwd && cs + i >= c0; };

    if (warp == 0) {
        // ================================================================ producer
        // Keeps up to kStages chunks of loads in flight: a chunk's TMA boxes, and its raw log-gates
        // by cp.async, are issued as soon as its stage is free; chunks are then landed in order
        // (gate statistics, inert tail rows, FULL) as their loads complete.  Waiting for each
        // chunk's loads before issuing the next would leave one chunk of HBM traffic in flight.
        bool ok = true;
        int ni = 0, nl = 0;  // next chunk to issue, next chunk to land
        // the head's gate-activation parameters (raw gate input), taken once
        const float act_ea = ACT && a.act.A_log ? expf(a.act.A_log[hv]) : 0.f;
        const float act_bias = ACT && a.act.A_log && a.act.dt_bias ? a.act.dt_bias[hv] : 0.f;
        uint64_t t_last = globaltimer();
        uint32_t idle = 0;
        auto rdy = [&](int b, int ph) {
            return __shfl_sync(0xffffffffu, (int)mbar_test_wait(&bars[b], (uint32_t)ph & 1u), 0) != 0;
        };
        while (nl < nch) {
            bool prog = false;
            if (ni < nch && (ni < kStages || rdy(B_EMPTY + ni % kStages, ni / kStages - 1))) {
                // ---- issue chunk ni (its stage and gate-ring entry are free: chunk ni - 3 is done)
                const int c = cs + ni, s = ni % kStages;
                const int64_t t0 = bos + (int64_t)c * kChunk;
                const int rows = rows_in(len, c);
                const bool emit = emit_of(ni);
                uint8_t *st = sm + OFF_STAGE + s * kStageBytes;
                if constexpr (KDA) {
                    // the preparation's nine boxes of the chunk (three TMA copies of 192 rows), its 2^G_C
                    (void)rows;
                    (void)emit;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bars[B_TMA + s], 73728u);
                        const int trow = (int)((tile_slot(bos, n, c) * HV + hv) * 576);
#pragma unroll
                        for (int b3 = 0; b3 < 3; ++b3)
                            tma_load_2d(st + 24576 * b3, &m.tiles, 0, trow + 192 * b3, &bars[B_TMA + s]);
                    }
                    float *gcd = gates(ni);
                    const float *gsrc = a.kda_gc + ((size_t)tile_slot(bos, n, c) * HV + hv) * 128;
#pragma unroll
                    for (int u = 0; u < 4; ++u) cp_async4(gcd + 4 * lane + u, gsrc + 4 * lane + u, 4u);
                } else {
                    if (lane == 0) {
                        const uint32_t bytes = 32768u + (emit ? 16384u : 0u) + (zero_values ? 0u : 16384u);
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
                        // operand tiles of the chunk: rows (slot * HV + hv) * 128 + {0, 64}
                        const int trow = (int)((tile_slot(bos, n, c) * HV + hv) * 128);
                        tma_load_2d(st + sTU, &m.tiles, 0, trow, &bars[B_TMA + s]);
                        tma_load_2d(st + sTW, &m.tiles, 0, trow + 64, &bars[B_TMA + s]);
                    }
                    // raw log-gates of rows 2l, 2l+1 into the chunk's gate block (zeros past the end)
                    float *graw = gates(ni) + GT_GRAW;
                    const float *gsrc = a.g + (size_t)t0 * HV + hv;
    #pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int r = 2 * lane + u;
                        cp_async4(graw + r, gsrc + (size_t)(r < rows ? r : 0) * HV, r < rows ? 4u : 0u);
                    }
                    if (rkp) {
                        const float *rsrc = rkp + ((size_t)tile_slot(bos, n, c) * HV + hv) * 64;
                        cp_async4(gates(ni) + GT_RK + 2 * lane, rsrc + 2 * lane, 4u);
                        cp_async4(gates(ni) + GT_RK + 2 * lane + 1, rsrc + 2 * lane + 1, 4u);
                    }
                    if (rqp && emit) {
                        const float *qsrc = rqp + ((size_t)tile_slot(bos, n, c) * HV + hv) * 64;
                        cp_async4(gates(ni) + GT_RQ + 2 * lane, qsrc + 2 * lane, 4u);
                        cp_async4(gates(ni) + GT_RQ + 2 * lane + 1, qsrc + 2 * lane + 1, 4u);
                    }
                }
                cp_async_commit();
                ++ni;
                prog = true;
            }
            if (nl < ni && rdy(B_TMA + nl % kStages, nl / kStages)) {
                // ---- land chunk nl: its raw gates are in once at most ni - nl - 1 younger groups are pending
                const int younger = ni - nl - 1;
                if (younger >= 2) cp_async_wait<2>();
                else if (younger == 1) cp_async_wait<1>();
                else cp_async_wait<0>();
                const int c = cs + nl, s = nl % kStages;
                const int rows = rows_in(len, c);
                if constexpr (!KDA) {
                    float *gt = gates(nl);
                    // gate statistics: lane holds rows 2l, 2l+1; base-2 inclusive cumsum
                    const int r0 = 2 * lane, r1 = r0 + 1;
                    const float2 gr = *(const float2 *)(gt + GT_GRAW + r0);
                    // (activated in place when the gate input is raw; rows past the end stay exactly 0)
                    float g0 = gr.x * kRcpLn2, g1 = gr.y * kRcpLn2;
                    if constexpr (ACT) {
                        if (a.act.A_log) {
                            g0 = (r0 < rows ? act_gate_pre(a.act, gr.x, act_bias, act_ea) : 0.f) * kRcpLn2;
                            g1 = (r1 < rows ? act_gate_pre(a.act, gr.y, act_bias, act_ea) : 0.f) * kRcpLn2;
                        }
                    }
                    float sp = g0 + g1;
    #pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, sp, off);
                        if (lane >= off) sp += y;
                    }
                    const float G0 = sp - g1, G1 = sp;
                    const float GC = __shfl_sync(0xffffffffu, sp, 31);
                    const float gm0 = ex2(G0), gm1 = ex2(G1);
                    *(float2 *)(gt + GT_G + r0) = make_float2(G0, G1);
                    *(float2 *)(gt + GT_GAM + r0) = make_float2(gm0, gm1);
                    // the update operand's row factors gC / gam (and 1 / ||k|| of the in-kernel L2 norm)
                    float2 rk2 = make_float2(1.f, 1.f);
                    if (rkp) rk2 = *(const float2 *)(gt + GT_RK + r0);
                    *(float2 *)(gt + GT_RDEC + r0) = make_float2(ex2(GC - G0) * rk2.x, ex2(GC - G1) * rk2.y);
                    *(float2 *)(gt + GT_GINV + r0) = make_float2(ex2(-G0), ex2(-G1));  // read only if G_C >= kFactorFloor
                    // the output's row factors scale * gam (a factored chunk's with 1 / ||q|| of the in-kernel L2
                    // norm folded in; a steep chunk's Q~ and P take it themselves)
                    float2 sg = make_float2(a.scale * gm0, a.scale * gm1);
                    if (rqp && emit_of(nl) && GC >= kFactorFloor) {
                        const float2 q2 = *(const float2 *)(gt + GT_RQ + r0);
                        sg.x *= q2.x;
                        sg.y *= q2.y;
                    }
                    *(float2 *)(gt + GT_SGAM + r0) = sg;
                    if (rows < kChunk) {
                        // rows past the end of the sequence belong to the next one: make them inert zeros
                        uint8_t *st = sm + OFF_STAGE + s * kStageBytes;
                        const bool emit = emit_of(nl);
                        const uint4 z = make_uint4(0, 0, 0, 0);
                        const int nz = (kChunk - rows) * 8;  // 16-byte pieces per box
    #pragma unroll 1
                        for (int bx = 0; bx < 6; ++bx) {
                            if ((bx == 2 || bx == 3) && !emit) continue;
                            if (bx >= 4 && zero_values) continue;
                            const uint32_t boff = bx == 0 ? sK0 : bx == 1 ? sK1 : bx == 2 ? sQ0 : bx == 3 ? sQ1 : bx == 4 ? sV0 : sV1;
                            uint4 *p = (uint4 *)(st + boff + rows * 128);
                            for (int e = lane; e < nz; e += 32) p[e] = z;
                        }
                        fence_proxy_async();
                    }
                } else {
                    (void)rows;
                }
                __syncwarp();
                // (the timeout-path test withholds the first chunk's signal: every role's wait then runs out)
                if (lane == 0 && !(a.withhold_full0 && nl == 0)) mbar_arrive(&bars[B_FULL + s]);
                ++nl;
                prog = true;
            }
            if (prog) {
                idle = 0;
                t_last = globaltimer();
            } else {
                __nanosleep(32);
                if ((++idle & 255u) == 0 && __shfl_sync(0xffffffffu, (int)(globaltimer() - t_last > kWaitNs), 0)) {
                    ok = false;
                    break;
                }
            }
        }
        if (!ok && lane == 0) atomicOr(status, kStatusTimeout);
        // copies still in flight after a failure land before the CTA releases its shared memory
        for (int i = nl; i < ni; ++i)
            mbar_wait(&bars[B_TMA + i % kStages], (i / kStages) & 1, status, kStatusTimeout, kWaitNs);
        cp_async_wait<0>();
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        // A fixed program per chunk, ordered around the serial chain: each chain product is
        // issued as soon as its operands are ready, and the state-independent products are
        // queued behind it so that the tensor pipe stays busy while the chain warps convert.
        // The whole warp follows the program (warp-uniform waits) and one elected lane issues:
        // the operands of tcgen05.mma are then warp-uniform values.
        if (KDA && nch > 0) {
            // per-channel gates: U, -W, K^, Q~ and P come with the stage; the program holds only the chain
            // products and the output products
            const uint32_t idV1K = idesc_bf16_f32(128, 64, 0, 0);  // A in TMEM, K-major B (-W, Q~, P)
            const uint32_t idS = idesc_bf16_f32(128, 128, 0, 1);   // A in TMEM, MN-major B (K^), N = dk
            bool ok = true;
            auto wait = [&](int b, int ph) {
                if (ok) ok = mbar_wait(&bars[b], (uint32_t)ph & 1u, status, kStatusTimeout, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                return ok;
            };
            int e = 0;
            for (int c = 0; c < nch && ok; ++c) {
                const uint32_t st = sbase + OFF_STAGE + (c % kStages) * kStageBytes;
                // the stage's descriptors: a byte offset b adds b / 16 to the address field (no carry: shared
                // memory addresses stay below 256 KB)
                const uint64_t dw = kmaj(st + sTU), dq = kmaj(st + sQ0), dk = sdesc_sw128(st + sK0, 16384, 1024),
                               dp = kmaj(st + sKdaP);
                // ---- -(W S)^T = S^T (-W)^T: -W as K-major B (rows = tokens), fresh accumulator
                if (!wait(B_SBF, c)) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts(tb + TM_VP, tb + TM_SBF + ks * 8, dw + (((ks >> 2) * 8192 + (ks & 3) * 32) >> 4), idV1K,
                               ks > 0 ? 1u : 0u);
                    mma_commit(&bars[B_VPF]);
                }
                __syncwarp();
                // ---- O^T = S^T Q~^T (emitted chunks only: a warmup chunk of the split only carries the state)
                const bool em = emit_of(c);
                if (em) {
                    if (e > 0 && !wait(B_OE, e - 1)) break;
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_ts(tb + TM_O, tb + TM_SBF + ks * 8, dq + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                                   idV1K, ks > 0 ? 1u : 0u);
                    }
                    __syncwarp();
                }
                // ---- S^T += V'^T K^  (B = K^, MN-major: dk atoms 16 KB apart; the per-channel decay is applied
                //      to S^T by the chain)
                if (!wait(B_VTF, c)) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ts(tb + TM_S, tb + TM_VB + ks * 8, dk + ks * 128, idS, 1u);
                    mma_commit(&bars[B_SF]);
                }
                __syncwarp();
                // ---- O^T += V'^T P^T
                if (em) {
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ts(tb + TM_O, tb + TM_VB + ks * 8, dp + ks * 2, idV1K, 1u);
                        mma_commit(&bars[B_OF]);
                    }
                    __syncwarp();
                    ++e;
                }
                if (elect_one()) {
                    mma_commit(&bars[B_EMPTY + c % kStages]);  // every product reading stage c is issued
                    // a warmup chunk stores no output: its second arrival is made here, in chunk order (the
                    // output warps, with no -W^T to wait for, would run ahead of the stage ring)
                    if (!em) mbar_arrive(&bars[B_EMPTY + c % kStages]);
                }
                __syncwarp();
            }
            if (!ok && lane == 0) atomicOr(status, kStatusTimeout);
            if (elect_one()) mma_commit(&bars[B_FIN]);
            __syncwarp();
            mbar_wait(&bars[B_FIN], 0, status, kStatusTimeout, kWaitNs);
        } else if (!KDA && nch > 0) {
            const uint32_t idKQ = idesc_bf16_f32(128, 64, 0, 0);   // K-major A and B
            const uint32_t idMN = idesc_bf16_f32(128, 64, 1, 0);   // MN-major A (V^T, K^T), K-major B
            const uint32_t idV1 = idesc_bf16_f32(128, 64, 0, 1);   // A in TMEM, MN-major B (-W^T)
            const uint32_t idO = idesc_bf16_f32(128, 64, 0, 0);    // A in TMEM, K-major B (Q~, P)
            const uint32_t idS = idesc_bf16_f32(128, 128, 0, 1);   // A in TMEM, MN-major B (K), N = dk
            auto stage = [&](int i) { return sbase + OFF_STAGE + (i % kStages) * kStageBytes; };
            bool ok = true;
            auto wait = [&](int b, int ph) {
                if (ok) ok = mbar_wait(&bars[b], (uint32_t)ph & 1u, status, kStatusTimeout, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                return ok;
            };
            auto ready = [&](int b, int ph) {
                return __shfl_sync(0xffffffffu, (int)mbar_test_wait(&bars[b], (uint32_t)ph & 1u), 0) != 0;
            };
            // Q K^T (lanes 64-127 of [K; Q] K^T) of emitted chunks only; its phases count emitted chunks
            const int ce0 = fwd ? min(max(c0 - cs, 0), nch) : nch;
            int kq = ce0;
            auto issue_kq = [&]() {
                const uint64_t d0 = kmaj(stage(kq));
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t d = d0 + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4);
                        mma_ss(tb + TM_KQ, d, d, idKQ, ks > 0 ? 1u : 0u);
                    }
                    mma_commit(&bars[B_KQF]);
                }
                __syncwarp();
                ++kq;
            };
            // up to chunk lim: blocking (the program needs it now) or only what is ready
            auto kq_upto = [&](int lim, bool block) {
                while (ok && kq < nch && kq <= lim) {
                    const int fs = B_FULL + kq % kStages, fp = kq / kStages;
                    if (block) {
                        if (!wait(fs, fp) || (kq > ce0 && !wait(B_KQE, kq - 1 - ce0))) break;
                    } else if (!ready(fs, fp) || (kq > ce0 && !ready(B_KQE, kq - 1 - ce0))) {
                        break;
                    }
                    issue_kq();
                }
            };
            auto issue_w = [&](int i) {
                // W^T = K^T (A_g diag(beta gam))^T   (A = K, MN-major: dk atoms 16 KB apart)
                const uint32_t s2 = stage(i);
                const uint64_t da = sdesc_sw128(s2 + sK0, 16384, 1024), db = kmaj(s2 + sTW);
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tb + TM_W, da + ks * 128, db + ks * 2, idMN, ks > 0 ? 1u : 0u);
                    mma_commit(&bars[B_WF]);
                }
                __syncwarp();
            };
            auto issue_u = [&](int i) {
                // U^T = V^T (A_g diag(beta))^T into the V' accumulator (A = V, MN-major: dv atoms 8 KB apart)
                if (zero_values) return;
                const uint32_t s2 = stage(i);
                const uint64_t da = sdesc_sw128(s2 + sV0, 8192, 1024), db = kmaj(s2 + sTU);
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tb + TM_VP, da + ks * 128, db + ks * 2, idMN, ks > 0 ? 1u : 0u);
                }
                __syncwarp();
            };
            // descriptors of the fixed operands (-W^T, P): a byte offset b adds b / 16 to the address field
            // (shared-memory addresses stay below 256 KB: no carry out of it)
            const uint64_t dws = sdesc_sw128(sbase + OFF_WS, 8192, 1024), dp = kmaj(sbase + OFF_P);
            // prologue: the first chunk's W and U, Q K^T of the first emitted chunks
            if (wait(B_FULL, 0)) {
                issue_w(0);
                issue_u(0);
            }
            kq_upto(1, false);
            int e = 0;
            for (int c = 0; c < nch && ok; ++c) {
                const bool em = emit_of(c);
                const uint32_t st = stage(c);
                // ---- V'^T (holding U^T, issued before) -= S^T W^T
                if (!wait(B_SBF, c)) break;  // the state copy and -W^T (one barrier: one wait fewer per chunk)
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts(tb + TM_VP, tb + TM_SBF + ks * 8, dws + ks * 128, idV1, (ks > 0 || !zero_values) ? 1u : 0u);
                    mma_commit(&bars[B_VPF]);
                }
                __syncwarp();
                if (em) {
                    // ---- O^T = S^T Q^T, or S^T Q~^T for a steep chunk (S^T is read before the chain
                    //      overwrites it: SF commits after it); the raw Q of a factored chunk is ready
                    //      with the stage, a steep chunk waits for Q~
                    kq_upto(c, true);
                    if ((!factored(c) && !wait(B_QS + c % kStages, c / kStages)) || (e > 0 && !wait(B_OE, e - 1)))
                        break;
                    const uint64_t dq0 = kmaj(st + sQ0);
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_ts(tb + TM_O, tb + TM_SBF + ks * 8, dq0 + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4), idO,
                                   ks > 0 ? 1u : 0u);
                    }
                    __syncwarp();
                }
                // ---- S^T += (V'^T diag(gC/gam)) K   (B = K, MN-major: dk atoms 16 KB apart)
                const uint64_t dks = sdesc_sw128(st + sK0, 16384, 1024);
                if (!wait(B_VTF, c)) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ts(tb + TM_S, tb + TM_VTB + ks * 8, dks + ks * 128, idS, 1u);
                    mma_commit(&bars[B_SF]);
                }
                __syncwarp();
                // ---- the next chunk's W (its conversion then overlaps the state copy)
                if (c + 1 < nch) {
                    if (!wait(B_FULL + (c + 1) % kStages, (c + 1) / kStages)) break;
                    issue_w(c + 1);
                }
                if (em) {
                    // ---- O^T += V'^T P^T, or (V'^T diag(gC/gam)) (Lower(Q K^T) / gC)^T in the factored
                    //      form (before the next V' product: the chain's V' commit covers it)
                    if (!wait(B_PF, e)) break;
                    const uint32_t va = tb + (factored(c) ? TM_VTB : TM_VB);
                    tc_fence_after();
                    if (elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ts(tb + TM_O, va + ks * 8, dp + ks * 2, idO, 1u);
                        mma_commit(&bars[B_OF]);
                    }
                    __syncwarp();
                    ++e;
                }
                if (c + 1 < nch) issue_u(c + 1);  // V'(c) has been read (VTF)
                kq_upto(c + 2, false);
                if (elect_one()) mma_commit(&bars[B_EMPTY + c % kStages]);  // every product reading stage c is issued
                __syncwarp();
            }
            if (!ok && lane == 0) atomicOr(status, kStatusTimeout);
            // every product issued so far has finished before the CTA frees its tensor memory
            if (elect_one()) mma_commit(&bars[B_FIN]);
            __syncwarp();
            mbar_wait(&bars[B_FIN], 0, status, kStatusTimeout, kWaitNs);
        }
    } else if (warp == 2 || warp == 3) {
        if constexpr (!KDA) {
        // ================================================================ aux: Q~ in place, P (lane = row of Q K^T)
        const int r = tid - 64;  // 0..63; TMEM lanes 64..127
        const uint32_t tl = tb + ((uint32_t)((warp & 3) * 32) << 16);
        bool ok = true;
        int e = 0;
        for (int i = 0; i < nch && ok; ++i) {
            const int s = i % kStages;
            if (!emit_of(i)) {
                // warmup chunk: nothing reads its Q~; the arrival keeps the stage barrier's phase count
                if (lane == 0) mbar_arrive(&bars[B_QS + s]);
                continue;
            }
            ok = mbar_wait(&bars[B_FULL + s], (i / kStages) & 1, status, kStatusTimeout, kWaitNs);
            if (ok) ok = mbar_wait(&bars[B_KQF], e & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const float *gt = gates(i);
            // Q K^T row r into registers: the K K^T / Q K^T region is released at once
            uint32_t kq[64];
            tmem_ld32(tl + TM_KQ, kq);
            tmem_ld32(tl + TM_KQ + 32, kq + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_KQE]);
            const bool fac = gt[GT_G + 63] >= kFactorFloor;
            float rq = 1.f;
            // in-kernel L2 norm, steep chunk: 1 / ||q_r|| (from the preparation) for Q~ and P
            if (nrm && !fac) rq = gt[GT_RQ + r];
            if (!fac) {
                // steep chunk: Q~ row r = scale * gam_r * q_r, in place (the Q K^T product has read Q);
                // the 16-byte pieces go in a row-rotated order to spread the banks, all loads first
                uint8_t *st = sm + OFF_STAGE + s * kStageBytes;
                const float f = gt[GT_SGAM + r] * rq;
#pragma unroll 1
                for (int bx = 0; bx < 2; ++bx) {
                    uint8_t *row = st + (bx ? sQ1 : sQ0) + r * 128;
                    uint4 x[8];
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) x[c8] = *(const uint4 *)(row + ((c8 + r) & 7) * 16);
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        __nv_bfloat162 *h2 = (__nv_bfloat162 *)&x[c8];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 fv = __bfloat1622float2(h2[q]);
                            h2[q] = __floats2bfloat162_rn(fv.x * f, fv.y * f);
                        }
                    }
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) *(uint4 *)(row + ((c8 + r) & 7) * 16) = x[c8];
                }
                fence_proxy_async();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_QS + s]);
            if (e > 0) ok = mbar_wait(&bars[B_OF], (e - 1) & 1, status, kStatusTimeout, kWaitNs);  // P free
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            {
                // row r of the intra-chunk operand -> bf16, 128-byte swizzled
                uint8_t *prow = sm + OFF_P;
                if (fac) {
                    // Lower(Q K^T)[r, j] / gC (the gate factors sit in V' and in the O epilogue)
                    const float rg = gt[GT_GINV + 63];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float v[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) v[u] = (8 * q + u <= r) ? u2f(kq[8 * q + u]) * rg : 0.f;
                        *(uint4 *)(prow + sw128(r, 8 * q)) = pack8(v);
                    }
                } else {
                    // P row r = scale * Gam[r, j <= r] * (Q K^T)[r, j]  (/ (||q_r|| ||k_j||) with the L2 norm)
                    // steep decay: 2^-G_j may overflow, so each entry takes its own power
                    const float Gr = gt[GT_G + r], sc = a.scale * rq;
#pragma unroll 1
                    for (int q = 0; q < 8; ++q) {
                        const float4 g0 = *(const float4 *)(gt + GT_G + 8 * q);
                        const float4 g1 = *(const float4 *)(gt + GT_G + 8 * q + 4);
                        const float gj[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                        float v[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            uint32_t x = kq[0];
#pragma unroll
                            for (int qq = 0; qq < 8; ++qq)
                                if (qq == q) x = kq[8 * qq + u];
                            const float rkj = rkp ? gt[GT_RK + 8 * q + u] : 1.f;
                            v[u] = (8 * q + u <= r) ? sc * rkj * ex2(Gr - gj[u]) * u2f(x) : 0.f;
                        }
                        *(uint4 *)(prow + sw128(r, 8 * q)) = pack8(v);
                    }
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_PF]);
            ++e;
        }
        }
    } else if (warp >= 4 && warp < 12) {
        // ================================================================ chain (lane = dv; half hh of the columns)
        const int dv = 32 * (warp & 3) + lane;
        const int hh = (warp - 4) >> 2;
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
        if (nch > 0) {
            // the segment's initial state (dk columns 64 hh .. 64 hh + 63) into the state accumulator
#pragma unroll 1
            for (int q4 = 2 * hh; q4 < 2 * hh + 2; ++q4) {
                uint32_t r[32];
                if (init) {
                    const float *src = init + (size_t)(32 * q4) * V + dv;
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = f2u(__ldg(src + j * V));
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = f2u(identity && 32 * q4 + j == dv ? 1.f : 0.f);
                }
                tmem_st32(tl + TM_S + 32 * q4, r);
            }
            tmem_st_wait();
        }
        for (int i = 0; i < nch && ok; ++i) {
            const int s = i % kStages;
            ok = mbar_wait(&bars[B_FULL + s], (i / kStages) & 1, status, kStatusTimeout, kWaitNs);
            if (ok && i > 0) ok = mbar_wait(&bars[B_SF], (i - 1) & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const float *gt = gates(i);
            const float dec = KDA ? 1.f : gt[GT_GAM + 63];  // gC = 2^G_C (per channel with KDA: below)
            {
                // ---- S_i -> bf16 copy (MMA operand) and gC * S_i (accumulator of this chunk's update)
                uint32_t r[64];
                tmem_ld32(tl + TM_S + 64 * hh, r);
                tmem_ld32(tl + TM_S + 64 * hh + 32, r + 32);
                tmem_ld_wait();
                if constexpr (DUMP) {
                    // S[dk][dv] entering chunk cs + i, dk = 64 hh .. 64 hh + 63 (coalesced over the warp's dv)
                    float *dst = a.chunk_states + ((size_t)tile_slot(bos, n, cs + i) * HV + hv) * 128 * V +
                                 (size_t)(64 * hh) * V + dv;
#pragma unroll
                    for (int j = 0; j < 64; ++j) dst[(size_t)j * V] = u2f(r[j]);
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint32_t p[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) p[j] = pack_bf16(u2f(r[32 * q + 2 * j]), u2f(r[32 * q + 2 * j + 1]));
                    tmem_st16(tl + TM_SBF + 32 * hh + 16 * q, p);
                }
                if constexpr (KDA) {
                    // S^T column dk decays by 2^G_C,dk
#pragma unroll
                    for (int j4 = 0; j4 < 16; ++j4) {
                        const float4 f = *(const float4 *)(gt + 64 * hh + 4 * j4);
                        r[4 * j4] = f2u(u2f(r[4 * j4]) * f.x);
                        r[4 * j4 + 1] = f2u(u2f(r[4 * j4 + 1]) * f.y);
                        r[4 * j4 + 2] = f2u(u2f(r[4 * j4 + 2]) * f.z);
                        r[4 * j4 + 3] = f2u(u2f(r[4 * j4 + 3]) * f.w);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) r[j] = f2u(u2f(r[j]) * dec);
                }
                tmem_st32(tl + TM_S + 64 * hh, r);
                tmem_st32(tl + TM_S + 64 * hh + 32, r + 32);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_SBF]);

            // ---- V'^T (tokens 32 hh .. 32 hh + 31) -> bf16: as the output operand and scaled by
            //      gC/gam as the update operand; the scale factors are loaded while the product runs
            float rd[32];  // GDN: the update operand's factors gC/gam; KDA: U of this thread's column
            if constexpr (KDA) {
                // U[t][dv] for the tokens t of this half, from the chunk's U boxes (128-byte swizzled rows)
                const uint8_t *ub = sm + OFF_STAGE + s * kStageBytes + (dv >= 64 ? sV1 : sV0);
                const int cd = dv & 63;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int t = 32 * hh + j;
                    rd[j] = __bfloat162float(*(const __nv_bfloat16 *)(ub + t * 128 + ((((cd >> 3) ^ (t & 7)) << 4) | ((cd & 7) << 1))));
                }
            } else {
    #pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 x = *(const float4 *)(gt + GT_RDEC + 32 * hh + 4 * j4);
                    rd[4 * j4] = x.x;
                    rd[4 * j4 + 1] = x.y;
                    rd[4 * j4 + 2] = x.z;
                    rd[4 * j4 + 3] = x.w;
                }
            }
            ok = mbar_wait(&bars[B_VPF], i & 1, status, kStatusTimeout, kWaitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            {
                uint32_t r[32];
                tmem_ld32(tl + TM_VP + 32 * hh, r);
                tmem_ld_wait();
                uint32_t vb[16], vtb[16];
                if constexpr (KDA) {
                    // V' = U - W S (the product holds -W S)
#pragma unroll
                    for (int j = 0; j < 16; ++j) vb[j] = pack_bf16(u2f(r[2 * j]) + rd[2 * j], u2f(r[2 * j + 1]) + rd[2 * j + 1]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float x0 = u2f(r[2 * j]), x1 = u2f(r[2 * j + 1]);
                        vb[j] = pack_bf16(x0, x1);
                        vtb[j] = pack_bf16(x0 * rd[2 * j], x1 * rd[2 * j + 1]);
                    }
                    tmem_st16(tl + TM_VTB + 16 * hh, vtb);
                }
                tmem_st16(tl + TM_VB + 16 * hh, vb);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_VTF]);
        }
        // ---- final state of the segment (dk rows 64 hh .. 64 hh + 63)
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
#pragma unroll 1
                for (int d = 64 * hh; d < 64 * hh + 64; ++d) {
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
                    for (int q4 = 2 * hh; q4 < 2 * hh + 2; ++q4) {
                        uint32_t r[32];
                        tmem_ld32(tl + TM_S + 32 * q4, r);
                        tmem_ld_wait();
                        float *p = dst + (size_t)(32 * q4) * dstride;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            *p = u2f(r[j]);
                            p += dstride;
                        }
                    }
                }
            }
        }
    } else {
        // ================================================================ output warps
        const int et = tid - 384;
        const uint32_t tl = tb + ((uint32_t)((warp & 3) * 32) << 16);
        bool ok = true;
        int e = 0;
        for (int it = 0; it <= nch && ok; ++it) {
            if (!KDA && it < nch) {
                // ---- -W^T of chunk it (lane = dk) -> shared memory, MN-major operand of V' = U - W S
                ok = mbar_wait(&bars[B_WF], it & 1, status, kStatusTimeout, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t r[64];
                tmem_ld32(tl + TM_W, r);
                tmem_ld32(tl + TM_W + 32, r + 32);
                tmem_ld_wait();
                if (it >= 1) ok = mbar_wait(&bars[B_VPF], (it - 1) & 1, status, kStatusTimeout, kWaitNs);  // -W^T free
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                uint8_t *wrow = sm + OFF_WS;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float f[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) f[u] = -u2f(r[8 * q + u]);
                    *(uint4 *)(wrow + sw128(et, 8 * q)) = pack8(f);
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_SBF]);  // (with the chain warps' state copy)
            }
            if (it >= 1 && !emit_of(it - 1)) {
                // nothing to store (per-channel gates: the issuer releases a warmup chunk's stage)
                if (!KDA && et == 0) mbar_arrive(&bars[B_EMPTY + (it - 1) % kStages]);
            } else if (it >= 1) {
                // ---- O of chunk it - 1 (lane = dv)
                const int ci = it - 1, c = cs + ci;
                const int64_t t0 = bos + (int64_t)c * kChunk;
                const int rows = rows_in(len, c);
                ok = mbar_wait(&bars[B_OF], e & 1, status, kStatusTimeout, kWaitNs);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t r[64];
                tmem_ld32(tl + TM_O, r);
                tmem_ld32(tl + TM_O + 32, r + 32);
                tmem_ld_wait();
                const float *gt = gates(ci);
                if (!KDA && factored(ci)) {
                    // the row factors scale * gam_t of the factored form (per-channel gates: inside Q~ and P),
                    // with 1 / ||q_t|| of the in-kernel L2 norm folded in by the load warp
#pragma unroll
                    for (int j4 = 0; j4 < 16; ++j4) {
                        const float4 f = *(const float4 *)(gt + GT_SGAM + 4 * j4);
                        r[4 * j4] = f2u(u2f(r[4 * j4]) * f.x);
                        r[4 * j4 + 1] = f2u(u2f(r[4 * j4 + 1]) * f.y);
                        r[4 * j4 + 2] = f2u(u2f(r[4 * j4 + 2]) * f.z);
                        r[4 * j4 + 3] = f2u(u2f(r[4 * j4 + 3]) * f.w);
                    }
                }
                tc_fence_before();
                __syncwarp();
                // O region drained and the chunk's gate block read (the producer reuses it after the
                // next chunk's S^T Q^T product, which waits for this)
                if (lane == 0) mbar_arrive(&bars[B_OE]);
                if (rows == kChunk) {
                    // the O tile goes out by TMA from the chunk's Q boxes, which are dead now (both
                    // products reading them have completed): bf16, 128-byte swizzled rows of 64 dv
                    uint8_t *ob = sm + OFF_STAGE + (ci % kStages) * kStageBytes + (et >= 64 ? sQ1 : sQ0);
                    const int cd = et & 63;
                    uint32_t off[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) off[jj] = ((((uint32_t)cd >> 3) ^ (uint32_t)jj) << 4) + ((uint32_t)(cd & 7) << 1);
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        *(__nv_bfloat16 *)(ob + j * 128 + off[j & 7]) = __float2bfloat16_rn(u2f(r[j]));
                    fence_proxy_async();
                    bar_sync(1, 128);  // the four output warps
                    if (et == 0) {
                        uint8_t *st = sm + OFF_STAGE + (ci % kStages) * kStageBytes;
                        tma_store_3d(&m.o, st + sQ0, 0, hv, (int)t0);
                        tma_store_3d(&m.o, st + sQ1, 64, hv, (int)t0);
                        tma_store_commit();
                        tma_store_wait_read0();  // the stage may be reloaded once the copy has read it
                        mbar_arrive(&bars[B_EMPTY + ci % kStages]);
                    }
                } else {
                    // ragged tail chunk: only the sequence's own rows are written
                    __nv_bfloat16 *p = (__nv_bfloat16 *)a.o + ((size_t)t0 * HV + hv) * V + et;
                    const size_t ostride = (size_t)HV * V;
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        if (j < rows) *p = __float2bfloat16_rn(u2f(r[j]));
                        p += ostride;
                    }
                    if (et == 0) mbar_arrive(&bars[B_EMPTY + ci % kStages]);
                }
                ++e;
            }
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

// 2-D map over the operand tiles, bf16 [rows][64], box = 64 x box_rows, 128-byte swizzle.
bool make_tiles_map(CUtensorMap *map, const void *base, int64_t rows, uint32_t box_rows = 64)
{
    auto enc = get_encoder();
    if (!enc || !base) return false;
    cuuint64_t dims[2] = {64, (cuuint64_t)rows};
    cuuint64_t strides[1] = {64 * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool encode_rows_map(CUtensorMap *map, const void *base, int heads, int64_t rows) { return make_map(map, base, heads, rows); }

bool encode_tiles_map(CUtensorMap *map, const void *base, int64_t rows, uint32_t box_rows)
{
    return make_tiles_map(map, base, rows, box_rows);
}

size_t tc_smem_bytes() { return TcLayout<false, false>::kSmem; }

bool tc_shape_ok(const gdn_shape *s)
{
    // scalar gates, or per-channel gates (their own chunk preparation; no chunk-parallel split).  The
    // operand tiles are addressed by 32-bit TMA row coordinates (576 rows per chunk-head at most).
    if (!(s->qkv_dtype == GDN_BF16 && s->K == 128 && s->V == 128 && (size_t)s->B * s->T < (1ull << 31)))
        return false;
    const int64_t rows = tile_slots((int64_t)s->B * s->T, s->num_seqs) * (int64_t)s->HV * 576;
    return rows < (int64_t)1 << 31;
}

bool tc_supported(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                  const void *o)
{
    if (!tc_shape_ok(s)) return false;
    auto al = [](const void *p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; };
    // per-channel gates are read as float4 rows by the KDA preparation
    const bool g_ok = s->gate_kind != GDN_GATE_CHANNEL || al(g);
    return al(q) && al(k) && al(v) && al(o) && g_ok && get_encoder() != nullptr;
}

cudaError_t launch_tc_scan(const ScanArgs &a, int value_tiles, bool kda, cudaStream_t st)
{
    static_assert(TcLayout<false, false>::kSmem <= 227 * 1024 && TcLayout<false, true>::kSmem <= 227 * 1024 &&
                      TcLayout<true, false>::kSmem <= 227 * 1024,
                  "shared memory budget");
    if (a.N * a.HV == 0) return cudaSuccess;
    TcMaps maps;
    memset(&maps, 0, sizeof(maps));
    const int64_t rows = (int64_t)a.B * a.T;
    if (rows > 0) {
        if (!make_map(&maps.o, a.o, a.HV, rows)) return cudaErrorInvalidValue;
        if (kda) {
            // the preparation's boxes: nine of 64 rows per (slot, value head), copied three at a time
            if (!make_tiles_map(&maps.tiles, a.tiles, (int64_t)a.tile_slots * a.HV * 576, 192))
                return cudaErrorInvalidValue;
        } else if (!make_map(&maps.q, a.q, a.H, rows) || !make_map(&maps.k, a.k, a.H, rows) ||
                   !make_map(&maps.v, a.v, a.HV, rows) ||
                   !make_tiles_map(&maps.tiles, a.tiles, (int64_t)a.tile_slots * a.HV * 128)) {
            return cudaErrorInvalidValue;
        }
    }
    dim3 grid(value_tiles, a.n_seg, a.N * a.HV);
    auto go = [&](auto kern, uint32_t smem) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kThreadsTC, smem, st>>>(a, maps);
        return cudaSuccess;
    };
    // the per-channel engine's operands come prepared (activated, normalised) from its preparation
    const bool act = !kda && (a.act.A_log != nullptr || a.act.qk_l2norm);
    if (a.chunk_states && (kda || act || a.mode != kModeForward)) return cudaErrorInvalidValue;  // no dump there
    cudaError_t e;
    if (kda) e = go(tc_scan_kernel<true, false>, TcLayout<true, false>::kSmem);
    else if (act) e = go(tc_scan_kernel<false, true>, TcLayout<false, true>::kSmem);
    else if (a.chunk_states) e = go(tc_scan_kernel<false, false, true>, TcLayout<false, false>::kSmem);
    else e = go(tc_scan_kernel<false, false>, TcLayout<false, false>::kSmem);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gdn

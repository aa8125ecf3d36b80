// Internal declarations shared by the GB300 gated delta-rule kernels and the
// C-ABI layer.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kChunk = 64;               // chunk size C
constexpr float kRcpLn2 = 1.4426950408889634f;  // 1 / ln 2: log-gates are kept in base 2

// Device status word bits (first 16 bytes of every workspace).
enum : unsigned {
    kStatusTimeout = 1u << 0,      // a bounded mbarrier / flag wait ran out
    kStatusPlan = 1u << 1,         // a kernel found a plan inconsistency and skipped work
    kStatusNormBound = 1u << 2,    // warmup split used although beta*||k||^2 > 2 was seen
};

enum Mode : int { kModeForward = 0, kModePrepass = 1 };

// Input activations applied where the kernels load their inputs ("Flash Linear Attention" page,
// sec. 10, the in-kernel gate / L2-norm / sigma(beta) of the KDA inference backend; "KDA source
// walkthrough", kda_gate_chunk_cumsum for the gate).  All fields zero: inputs are used as given.
struct Act {
    const float *A_log;    // [HV]: the gate input is activated (nullable = g is already the log-decay)
    const float *dt_bias;  // [HV] (scalar gate) or [HV][K] (per-channel gate), nullable
    float lower_bound;     // < 0: g = lower_bound * sigmoid(exp(A_log) (x + bias));
                           // 0: g = -exp(A_log) * softplus(x + bias)
    int beta_logits;       // beta = sigmoid(input)
    int qk_l2norm;         // q, k scaled to unit L2 norm per (token, head) (x / max(||x||, 1e-12))
};
// the log-decay of z = x + bias with ea = exp(A_log): lower_bound sigmoid(ea z), or -ea softplus(z) (linear
// past z = 20 like the usual threshold).  By the fast exponential and logarithm: the softplus of z below
// about -17 rounds to 0 (its value is under 6e-8), and the gate's relative error stays far below the
// bf16 resolution of the operands it scales
__device__ __forceinline__ float act_gate_z(const Act &a, float z, float ea)
{
    if (a.lower_bound < 0.f) return a.lower_bound / (1.f + __expf(-ea * z));
    return -ea * (z > 20.f ? z : __logf(1.f + __expf(z)));
}
// the log-decay of gate input x for value head hv (channel d, or d < 0 for a scalar gate)
__device__ __forceinline__ float act_gate(const Act &a, float x, int hv, int d, int K)
{
    if (!a.A_log) return x;
    const float z = x + (a.dt_bias ? a.dt_bias[d < 0 ? hv : hv * K + d] : 0.f);
    return act_gate_z(a, z, expf(a.A_log[hv]));
}
// act_gate with the per-head factor exp(A_log) and the bias taken once by the caller (the same arithmetic)
__device__ __forceinline__ float act_gate_pre(const Act &a, float x, float bias, float ea)
{
    return act_gate_z(a, x + bias, ea);
}
__device__ __forceinline__ float act_beta(const Act &a, float x) { return a.beta_logits ? 1.f / (1.f + expf(-x)) : x; }
constexpr float kNormEps = 1e-12f;

// Arguments of one scan launch (one engine pass over segments).
struct ScanArgs {
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    const int64_t *cu_seqlens;  // nullable
    void *o;
    float *ht;
    int B, T, H, HV, K, V, N;
    float scale;
    // segmentation
    int seg_chunks;         // chunks per segment
    int n_seg;              // segments per sequence (grid.y bound)
    const int *warm_start;  // [N*HV*n_seg] first chunk a segment processes (warmup), nullable
    int warm_in_kernel;     // tensor-core engine: each CTA finds its own warmup start from g
    float warm_log2_eps;    // threshold of that search (accumulated log2-decay)
    const void *tiles;      // tensor-core engine: operand tiles of tc_prep_kernel / kda_prep_kernel (see tile_slot)
    const float *kda_gc;    // per-channel gates: 2^G_C per (slot, value head, channel)
    const float *kda_wdec;  //   and, for the warmup split, each chunk's log2-decay bound per (slot, value head)
    int tile_slots;         //   chunk slots of that buffer
    const float *seg_init;  // [N*HV*n_seg][K][V] start state per segment (exact split), nullable
    float *seg_out;         // prepass: [N*HV*n_seg][K][V+K] (S* | M)
    float *chunk_states;    // CUDA-core engine, forward: the state entering every chunk, [slot][HV][K][V]
                            //   (slot: tile_slot), for the backward pass; nullable
    int mode;               // Mode
    int vext;               // value columns processed: V (forward) or V + K (prepass)
    unsigned *status;
    const int *seq_order;   // [N] sequence of each grid.z group (longest first), nullable = natural order
    unsigned long long wait_ns;  // wall-clock limit of every device-side wait (tensor-core engine)
    int withhold_full0;     // timeout-path test: the load warp never signals its first chunk
    Act act;
    const float *rk;        // tensor-core engine, in-kernel L2 norm: 1 / ||k_t|| per (slot, value head, row)
    const float *rq;        //   and 1 / ||q_t|| (same layout), both from the chunk preparation
};

struct CombineArgs {
    const float *h0;
    const int64_t *cu_seqlens;
    const float *seg_out;  // [N*HV*n_seg][K][V+K]
    float *seg_init;       // [N*HV*n_seg][K][V]
    int T, HV, K, V, N, seg_chunks, n_seg;
    unsigned *status;
};

struct GateStatsArgs {
    const float *g;
    const float *beta;
    const int64_t *cu_seqlens;
    int *warm_start;       // [N*HV*n_seg]
    int T, HV, K, N, seg_chunks, n_seg, channel;
    float log2_eps;        // threshold on the window's accumulated log2-decay
    int max_warm_chunks;   // walk at most this far back, else start from the sequence start
    Act act;
};

// Arguments of the tensor-core engine's chunk preparation (operand tiles of every chunk).
struct PrepArgs {
    const void *k;
    const float *g, *beta;
    const int64_t *cu_seqlens;  // nullable
    void *tiles;                // bf16 [slot][HV][2][64][64]: T_U, T_W (slot: tile_slot)
    int T, H, HV, N, slots;
    int check_norm;             // flag beta ||k||^2 > 2 in the status word (warmup split)
    unsigned *status;
    int *seq_order;             // nullable: block (0, 0) writes the longest-first sequence order here
    int n_buckets;              //   chunk-count buckets of that sort (<= kOrderBuckets)
    unsigned long long wait_ns; // wall-clock limit of the product-completion wait
    Act act;
    float *rk;                  // qk_l2norm: 1 / ||k_t|| per (slot, value head, row), written for the scan
    float *rq;                  //   and 1 / ||q_t|| (same layout; rows past the end of the sequence 0)
    const void *q;              //   read only for rq
};

// Start states of consecutive pieces of sequences from their (S*, M) summaries (context parallel).
struct ChainArgs {
    const float *summaries;  // [ranks][pairs][K][V + K]
    const float *h0;         // [pairs][K][V], nullable (zero)
    float *starts;           // [ranks][pairs][K][V]
    int ranks, pairs, K, V;
};
cudaError_t launch_chain_states(const ChainArgs &a, cudaStream_t st);
// dst[p][b][a] = src[p][a][b] for p < P (fp32), the state layouts [K][V] <-> [V][K]
cudaError_t launch_transpose(const float *src, float *dst, int P, int A, int B, cudaStream_t st);

// Launchers (return cudaGetLastError() of the launch).
cudaError_t launch_simt_scan(const ScanArgs &a, gdn_dtype dt, gdn_gate_kind gate, cudaStream_t st);
cudaError_t launch_cp_combine(const CombineArgs &a, cudaStream_t st);
cudaError_t launch_gate_stats(const GateStatsArgs &a, cudaStream_t st);
size_t simt_smem_bytes(int K, gdn_gate_kind gate);

// Tensor-core engine (bf16, K = V = 128, scalar gate).  `value_tiles` is 1 for
// the forward pass and 2 for the exact split's pre-pass (S* and M columns).
bool tc_shape_ok(const gdn_shape *s);
bool tc_supported(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                  const void *o);
// Per-key-channel gates on the tensor-core engine: the chunk preparation (gdn_tc_kda.cu).
struct KdaPrepArgs {
    const void *q, *k, *v;
    const float *gk, *beta;     // gk [B*T][HV][128]
    float scale;
    const int64_t *cu_seqlens;  // nullable
    void *tiles;                // bf16 [slot][HV][9][64][64] (see gdn_tc_kda.cu)
    float *gc;                  // [slot][HV][128] per-channel chunk decay 2^G_C
    float *wdec;                // warmup split: [slot][HV] the chunk's bound on the state's log2-decay (the sum
                                //   over its tokens of the slowest channel's log2-gate); nullable
    int check_norm;             // warmup split: flag beta ||k||^2 > 2 in the status word
    unsigned *status;
    int T, H, HV, N, slots;
    int *seq_order;             // as PrepArgs
    int n_buckets;
    Act act;
};
cudaError_t launch_kda_prep(const KdaPrepArgs &a, cudaStream_t st);
constexpr size_t kKdaTileBytesPerChunk = 9 * 64 * 64 * 2 + 128 * 4;  // nine bf16 boxes and gC

cudaError_t launch_tc_scan(const ScanArgs &a, int value_tiles, bool kda, cudaStream_t st);
// 2-D TMA map over the operand tiles, bf16 rows of 64, box 64 x box_rows, 128-byte swizzle
bool encode_tiles_map(CUtensorMap *map, const void *base, int64_t rows, uint32_t box_rows);
// 3-D TMA map over a [rows][heads][128] bf16 tensor (q, k, v, o), box 64 elements x 1 head x 64 rows, 128-byte
// swizzle
bool encode_rows_map(CUtensorMap *map, const void *base, int heads, int64_t rows);
cudaError_t launch_tc_prep(const PrepArgs &a, cudaStream_t st);
constexpr size_t kTcTileBytesPerChunk = 2 * 64 * 64 * 2;  // T_U and T_W, bf16

// Chunk c of a sequence starting at token bos (sequence index n) has the operand-tile
// slot floor(bos / 64) + n + c: consecutive sequences never overlap and a batch of
// `tokens` tokens in `nseq` sequences needs at most tokens / 64 + nseq + 1 slots.
__host__ __device__ inline int64_t tile_slot(int64_t bos, int n, int c) { return bos / kChunk + n + c; }

// Longest-first order of the sequences of a packed batch.  The scan's CTAs are dispatched in grid
// order, so with this order the longest chains start first and the short ones fill in behind them
// (longest-processing-time-first scheduling).  One CTA, every thread: a counting sort on the chunk
// count (counts above n_buckets - 1 share the top bucket), descending; equal counts in any order.
// `hist` is shared-memory scratch of n_buckets + 32 ints.
constexpr int kOrderBuckets = 4096;
__device__ inline void order_longest_first(const int64_t *cu, int N, int n_buckets, int *hist, int *order)
{
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    int *wsum = hist + n_buckets;
    auto key = [&](int m) -> int {
        const long long nc = (cu[m + 1] - cu[m] + kChunk - 1) / kChunk;
        return n_buckets - 1 - (int)(nc < 0 ? 0 : nc > n_buckets - 1 ? n_buckets - 1 : nc);
    };
    for (int i = tid; i < n_buckets; i += nt) hist[i] = 0;
    __syncthreads();
    for (int m = tid; m < N; m += nt) atomicAdd(&hist[key(m)], 1);
    __syncthreads();
    // exclusive prefix sum over the buckets: a contiguous run per thread, then across threads
    const int per = (n_buckets + nt - 1) / nt;
    const int b0 = min(tid * per, n_buckets), b1 = min(b0 + per, n_buckets);
    int s = 0;
    for (int b = b0; b < b1; ++b) s += hist[b];
    int incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int run = incl - s;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int b = b0; b < b1; ++b) {
        const int c = hist[b];
        hist[b] = run;
        run += c;
    }
    __syncthreads();
    for (int m = tid; m < N; m += nt) order[atomicAdd(&hist[key(m)], 1)] = m;
}
__host__ __device__ inline int64_t tile_slots(int64_t tokens, int nseq) { return tokens / kChunk + nseq + 1; }
size_t tc_smem_bytes();

// Token-by-token engine (gdn_recurrent.cu): decode and short continuations.  h0 and ht may be the
// same buffer (the state cache updated in place).
struct RecArgs {
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    const int64_t *cu_seqlens;  // nullable
    void *o;
    float *ht;                  // nullable
    int T, H, HV, K, V, N;
    float scale;
    Act act;
};
cudaError_t launch_recurrent(const RecArgs &a, gdn_dtype dt, gdn_gate_kind gate, cudaStream_t st);

// Backward pass (scalar gates): A and P per chunk; the reverse scan, one CTA per (sequence, value head,
// 32-column value tile), chunks newest first; the state-independent gradient terms per chunk; the
// suffix sum of dG within each chunk into dg.
struct BwdArgs {
    const void *q, *k, *v, *dout;  // q, k [B,T,H,K]; v, dout [B,T,HV,V] (the dtype of v)
    const float *g, *beta;         // [B,T,HV]
    const float *dht;              // [N,HV,K,V], nullable
    const int64_t *cu_seqlens;     // nullable
    const float *chunk_states;     // [slot][HV][K][V]: the state entering every chunk (tile_slot)
    float *dq, *dk;                // [B,T,H,K], zeroed by the host (sums of value tiles and GVA heads)
    float *dv;                     // [B,T,HV,V]
    float *dbeta, *dG;             // [B,T,HV], zeroed by the host (dG: per-row gate gradient before Step 7)
    float *dg;                     // [B,T,HV]
    float *dh0;                    // [N,HV,K,V], nullable
    float *Abuf, *Pbuf;            // [slot][HV][64][64]: A = (I + L)^-1 and P of every chunk
    float *dPbuf, *dAbuf;          // [value tile][slot][HV][64][64]: each tile's part of dO D^T and dD B^T
    size_t chunk_heads;            // slots x HV
    int T, H, HV, K, V, N, max_nt;
    float scale;
};
cudaError_t launch_chunk_bwd(const BwdArgs &a, gdn_dtype dt, cudaStream_t st);
// AUTO engine choice: packed or batched sequences of at most this many tokens go to the token-by-token
// engine (decode, speculative continuations)
constexpr int kAutoRecurrentTokens = 16;

// Host-side checks of one forward call, as the entry points run them before anything is
// enqueued; on GDN_OK *ws_bytes (nullable) is the workspace the call needs.
gdn_status check_call(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                      const float *beta, float scale, const int64_t *cu, int chunk_size, const void *o,
                      const gdn_options *opt, size_t *ws_bytes);
// Synchronise `st`, return the device status recorded in the word at `ws` and clear it.
gdn_status read_status_word(void *ws, cudaStream_t st);

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace gdn

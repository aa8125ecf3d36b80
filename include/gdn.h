/*
 * gdn.h -- C ABI of the GB300 gated delta-rule chunked-prefill forward.
 *
 * The operation (per sequence n, value head h; key/query head h / (HV/H)):
 *
 *   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t = scale * S_t^T q_t,        S_0 = h0[n,h] (or 0),  ht[n,h] = S_T
 *
 * with alpha_t = exp(g_t) for a scalar gate (FlashQLA blog, "Further
 * optimisation via gate decay", the recurrence; "Key problems in FLA's GDN
 * chunked prefill", the chunk form) or alpha_t,d = exp(gk_t,d) for a
 * per-key-channel gate ("KDA source walkthrough", chunk_kda_fwd and the gk
 * branch of chunk_gated_delta_rule_fwd_h).  It is evaluated chunkwise
 * (chunk size C = 64): gate cumsum, gated strictly-lower K K^T, its
 * unit-lower-triangular inverse, the WY form, the serial inter-chunk state
 * scan and the output, optionally split over sequence segments on one GPU
 * (FlashQLA blog, "A balanced solution": the S* / M correction, and "Further
 * optimisation via gate decay": the gate-driven warmup).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers (except in gdn_chunk_fwd_host),
 *    contiguous (row-major, last index fastest) and owned by the caller.
 *  - Shapes (FlashQLA blog, "Usage"; GDN-in-FLA notes, forward signature):
 *      q, k   [B, T, H,  K]    qkv_dtype
 *      v      [B, T, HV, V]    qkv_dtype
 *      o      [B, T, HV, V]    qkv_dtype (written)
 *      g      [B, T, HV]       fp32, natural-log gate (gate_kind SCALAR)
 *      gk     [B, T, HV, K]    fp32, natural-log gate (gate_kind CHANNEL)
 *      beta   [B, T, HV]       fp32
 *      h0     [N, HV, K, V]    fp32, nullable (= zero initial state)
 *      ht     [N, HV, K, V]    fp32, nullable (final state not written)
 *      cu_seqlens [N+1]        int64 token offsets, nullable.  When given the
 *                              input is packed: B must be 1, T is the total
 *                              token count and sequence n spans tokens
 *                              [cu[n], cu[n+1]) ("Flash Linear Attention"
 *                              page, sec. 2, varlen: FlashAttention semantics).
 *                              Without it N = B and each batch row is one
 *                              sequence of T tokens.
 *  - State layout is [K][V] row-major (FLA's default, not state_v_first).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without synchronising.  Argument errors
 *    are reported before anything is enqueued; errors found on the device
 *    (a bounded wait that ran out, a failed plan check) are recorded in the
 *    workspace status word, read with gdn_read_device_status().
 *  - Nothing aborts the process and no entry point calls exit().
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gdn_stream_t; /* identical to cudaStream_t */

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

typedef enum { GDN_GATE_SCALAR = 0, GDN_GATE_CHANNEL = 1 } gdn_gate_kind;

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID = -1,     /* null pointer, negative or inconsistent size       */
    GDN_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. chunk_size != 64) */
    GDN_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed              */
    GDN_ERR_TIMEOUT = -4,     /* a bounded device wait ran out (device status)     */
    GDN_ERR_NOMEM = -5,       /* library-managed workspace could not be allocated  */
    GDN_ERR_WORKSPACE = -6    /* caller workspace smaller than gdn_workspace_size  */
} gdn_status;

typedef struct {
    int B, T, H, HV, K, V;   /* varlen: B == 1 and T == total tokens               */
    gdn_dtype qkv_dtype;     /* q, k, v and o share it; g/beta/h0/ht are fp32      */
    gdn_gate_kind gate_kind; /* SCALAR: g [B,T,HV];  CHANNEL: gk [B,T,HV,K]        */
    int num_seqs;            /* N: B, or len(cu_seqlens) - 1 for packed input       */
} gdn_shape;

/* How a long sequence is split over the GPU (FlashQLA blog, in-GPU CP). */
typedef enum {
    GDN_CP_AUTO = 0,   /* planner decides (split only when (seq, head) pairs are few) */
    GDN_CP_OFF = 1,    /* one serial scan per (sequence, head)                        */
    GDN_CP_EXACT = 2,  /* segments start from S* = 0, M = I; serial S* / M combine
                          (per-channel gates: on the SIMT engine)                    */
    GDN_CP_WARMUP = 3  /* segments re-derive their start state from zero over a
                          warmup window sized from the gate statistics (per-channel
                          gates: each token's slowest channel bounds its decay; AUTO
                          picks it for them on the TC engine only when the (sequence,
                          head) pairs fill at most a quarter of the SMs)             */
} gdn_cp_mode;

typedef enum {
    GDN_ENGINE_AUTO = 0, /* tensor-core engine where supported, else SIMT            */
    GDN_ENGINE_SIMT = 1, /* fp32 CUDA-core engine (any supported shape, fp32 inputs) */
    GDN_ENGINE_TC = 2,   /* tcgen05/TMEM engine: bf16, K = V = 128, scalar or
                            per-channel gate, q/k/v/o (and gk) 16-byte aligned; a
                            call that asks for it on other inputs gets
                            GDN_ERR_INVALID                                       */
    GDN_ENGINE_RECURRENT = 3 /* token by token, no chunks ("Flash Linear Attention"
                            page, sec. 8, fused_recurrent, C = 1): for decode and
                            short continuations; any supported shape; no split.
                            AUTO selects it when no sequence is longer than 16
                            tokens (T, or max_seq_len for packed input).          */
} gdn_engine;

typedef struct {
    gdn_cp_mode cp_mode;
    int segment_chunks;    /* chunks per segment when split (0 = planner's choice)  */
    gdn_engine engine;
    int keys_unit_norm;    /* caller asserts ||k_t||_2 <= 1 and 0 <= beta_t <= 2, so
                              every transition has spectral norm <= its decay; lets
                              AUTO choose the warmup split (qk_l2norm together with
                              beta_logits implies it)                               */
    float warmup_log2_eps; /* warmup stops once the window's decay <= 2^this (0 = -24) */
    int max_seq_len;       /* packed input: bound on one sequence's length, used to
                              size the split grid (0 = T)                             */
    void *const *launch_events; /* optional, caller-owned CUDA events (cudaEvent_t):
                              event i is recorded on the stream right before the
                              call's i-th kernel launch and event `kernels` (see
                              gdn_plan) right after the last one, so consecutive
                              events time each kernel.  NULL: nothing recorded.   */
    int n_launch_events;   /* length of launch_events; extra marks are skipped      */
    int wait_limit_us;     /* wall-clock limit of every device-side wait of the
                              tensor-core kernels, in microseconds (0 = 2 s).  A
                              wait that runs out records GDN_ERR_TIMEOUT in the
                              device status and the kernel ends early.            */
    int test_withhold_first_arrival; /* testing the timeout path only: nonzero makes
                              the tensor-core scan's load warp withhold its "chunk
                              loaded" signal for the first chunk of every CTA, so
                              every role's wait runs out (bounded by
                              wait_limit_us), the device status reads
                              GDN_ERR_TIMEOUT and o / ht are left undefined.  No
                              effect on the SIMT engine.                          */
    /* Input activations done inside the kernels ("Flash Linear Attention" page,
     * sec. 10: the KDA inference backend takes raw tensors and fuses the gate,
     * the L2 norm and sigma(beta); "KDA source walkthrough",
     * kda_gate_chunk_cumsum, for the gate).  All zero: inputs used as given.   */
    const float *gate_A_log;   /* [HV], device; non-NULL: g_or_gk holds the raw
                              gate input x and the log-decay is
                              -exp(A_log[h]) * softplus(x + dt_bias), or with
                              gate_lower_bound < 0:
                              gate_lower_bound * sigmoid(exp(A_log[h]) (x + dt_bias)) */
    const float *gate_dt_bias; /* [HV] (scalar gate) or [HV][K] (per-channel), device,
                              nullable (zero)                                       */
    float gate_lower_bound;    /* < 0 selects the bounded form above; 0: softplus form */
    int beta_logits;           /* beta holds logits: the kernels use sigmoid(beta)     */
    int qk_l2norm;             /* q and k are scaled to unit L2 norm per (token, head)
                              inside the kernels: x / max(||x||_2, 1e-12)            */
    int state_v_first;         /* h0 and ht are [N, HV, V, K] instead of [N, HV, K, V]
                              (the transposed state layout; the library transposes
                              them around the call through its workspace)           */
} gdn_options;

/* Fill `opt` with the defaults (AUTO everywhere, no assertions).  No
 * counterpart in the pages (library infrastructure). */
void gdn_default_options(gdn_options *opt);

/* Human-readable name of a status code (static string, never NULL).  No
 * counterpart in the pages. */
const char *gdn_status_string(gdn_status st);

/* Library version: major * 10000 + minor * 100 + patch.  No counterpart in
 * the pages. */
int gdn_version(void);

/*
 * Bytes of device workspace gdn_chunk_fwd_ws needs for this problem and
 * options (at least 256: the first 256 bytes hold the device status word).
 * Returns 0 if the arguments are invalid or unsupported.  No counterpart in
 * the pages (the pages' kernels allocate their intermediates themselves).
 */
size_t gdn_workspace_size(const gdn_shape *s, int chunk_size, const gdn_options *opt);

/*
 * The forward pass of the problem statement (FlashQLA blog, "Usage":
 * chunk_gated_delta_rule(q, k, v, g, beta, scale, initial_state,
 * output_final_state, cu_seqlens) -> (o, final_state)) with a caller-provided
 * workspace (`workspace`, at least
 * gdn_workspace_size bytes, 256-byte aligned, device memory).  The
 * workspace must not be used by another call that can run concurrently.
 * Returns GDN_OK once all work is enqueued on `stream`.
 */
gdn_status gdn_chunk_fwd_ws(const gdn_shape *s,
                            const void *q, const void *k, const void *v,
                            const float *g_or_gk, const float *beta, float scale,
                            const float *h0, const int64_t *cu_seqlens, int chunk_size,
                            void *o, float *ht, const gdn_options *opt,
                            void *workspace, size_t ws_bytes, gdn_stream_t stream);

/*
 * The forward pass of the problem statement (FlashQLA blog, "Usage"; the
 * GDN-in-FLA notes, forward signature; "KDA source walkthrough",
 * chunk_kda_fwd for the per-channel gate) -- the plain entry point -- with
 * default options and a library-managed workspace,
 * cached per (device, stream) and grown stream-ordered (cudaMallocAsync on
 * `stream`) when a call needs more.  Arguments as in gdn_chunk_fwd_ws.
 */
gdn_status gdn_chunk_fwd(const gdn_shape *s,
                         const void *q, const void *k, const void *v,
                         const float *g_or_gk, const float *beta, float scale,
                         const float *h0, const int64_t *cu_seqlens, int chunk_size,
                         void *o, float *ht, gdn_stream_t stream);

/* As gdn_chunk_fwd with explicit options (NULL = defaults): the split mode
 * and warmup threshold follow the FlashQLA blog, "A balanced solution" and
 * "Further optimisation via gate decay". */
gdn_status gdn_chunk_fwd_ex(const gdn_shape *s,
                            const void *q, const void *k, const void *v,
                            const float *g_or_gk, const float *beta, float scale,
                            const float *h0, const int64_t *cu_seqlens, int chunk_size,
                            void *o, float *ht, const gdn_options *opt, gdn_stream_t stream);

/*
 * The forward pass of the problem statement (FlashQLA blog, "Usage") as an
 * end-to-end call on HOST buffers (pageable or pinned): copies the inputs to
 * a library-owned device arena, runs gdn_chunk_fwd_ex, copies o (and ht when
 * non-NULL) back, and synchronises `stream` before returning.  The call is
 * cut into up to four groups of whole sequences (contiguous token ranges of
 * every tensor); group i runs on `stream` while group i+1's inputs are copied
 * in and group i-1's outputs copied out, each direction on a library-owned
 * stream of the current device.  `cu_seqlens` is a host array here too and is
 * checked on the host (cu[0] == 0, nondecreasing, cu[N] == T).  Same shapes
 * as above.
 */
gdn_status gdn_chunk_fwd_host(const gdn_shape *s,
                              const void *q, const void *k, const void *v,
                              const float *g_or_gk, const float *beta, float scale,
                              const float *h0, const int64_t *cu_seqlens, int chunk_size,
                              void *o, float *ht, const gdn_options *opt,
                              gdn_stream_t stream);

/*
 * No counterpart in the pages (the bounded device waits are this library's).
 * Synchronise `stream`, return the status the device recorded in the
 * workspace since the last read, and clear it.  `workspace` is the buffer
 * given to gdn_chunk_fwd_ws, or NULL for the library-managed workspace of
 * (current device, stream).
 */
gdn_status gdn_read_device_status(void *workspace, gdn_stream_t stream);

/*
 * The forward pass without any allocation (no counterpart in the paper; an
 * interface for callers that cannot allocate device memory when they run the
 * forward: code running inside a memory pool it does not own, runtimes that
 * forbid cudaMalloc on their hot path because it synchronises the device, or
 * embeddings that reserved all device memory up front).  Arguments as in
 * gdn_chunk_fwd_ex; the caller still provides every input and output.
 *
 * Scratch (the device status word and the chunk-parallel split's tables)
 * lives in one fixed 4 MiB device array owned by the library, which every
 * GPU that loads the library holds until the process exits.  A plan that
 * needs more scratch than that (gdn_workspace_size > 4 MiB, e.g. the exact
 * split over many segments) is rejected with GDN_ERR_WORKSPACE before
 * anything is enqueued; choose GDN_CP_OFF or GDN_CP_WARMUP, or use
 * gdn_chunk_fwd_ws with a larger workspace.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress with that device current); make that first call
 * before any stream capture.  Every call uses the same array, which keeps
 * the previous call's contents: calls that can overlap on the GPU -- on
 * different streams, or from different threads -- race on it and must be
 * serialised by the caller.  No cudaMalloc, cudaFree or other allocating
 * routine is called.  Argument errors return the same codes as
 * gdn_chunk_fwd_ex and enqueue nothing.  Errors found on the device (a wait
 * that ran out, a failed plan check, the warmup split's key-norm check) are
 * collected in the array's status word until gdn_read_noalloc_status reads
 * and clears it.
 */
gdn_status gdn_chunk_fwd_noalloc(const gdn_shape *s,
                                 const void *q, const void *k, const void *v,
                                 const float *g_or_gk, const float *beta, float scale,
                                 const float *h0, const int64_t *cu_seqlens, int chunk_size,
                                 void *o, float *ht, const gdn_options *opt, gdn_stream_t stream);

/*
 * The device status of gdn_chunk_fwd_noalloc calls on the current device (no
 * counterpart in the paper): synchronises `stream`, returns the status word of
 * the fixed array as gdn_read_device_status does for a workspace (GDN_OK,
 * GDN_ERR_TIMEOUT or GDN_ERR_INVALID) and clears it.  Allocates nothing.
 */
gdn_status gdn_read_noalloc_status(gdn_stream_t stream);

/*
 * Decode / continuation of the problem statement ("Flash Linear Attention"
 * page, sec. 8: fused_recurrent, the C = 1 form the layer selects for short
 * queries): the same operation and arguments as gdn_chunk_fwd (no chunk
 * size), evaluated token by token on the recurrent engine.  `ht` may be the
 * same buffer as `h0`: the state cache is then updated in place.  Suited to
 * a few tokens per sequence (decode steps continuing from a prefill's final
 * state); longer sequences are faster on gdn_chunk_fwd.
 */
gdn_status gdn_recurrent_fwd(const gdn_shape *s,
                             const void *q, const void *k, const void *v,
                             const float *g_or_gk, const float *beta, float scale,
                             const float *h0, const int64_t *cu_seqlens,
                             void *o, float *ht, gdn_stream_t stream);

/*
 * Backward pass of the chunked forward (GDN-in-FLA notes, backward: the gradients
 * dq, dk, dv, db, dg, dh0 of chunk_gated_delta_rule_bwd, Steps 1-7; "Flash Linear
 * Attention" page, sec. 7: the state gradient scanned in reverse time, the chunk
 * states recomputed).  Given the same inputs as gdn_chunk_fwd (scalar gate) and
 * `dout` [B,T,HV,V] (the dtype of v), the gradient of the loss with respect to o,
 * and `dht` [N,HV,K,V] fp32 (nullable: zero), the gradient with respect to the
 * final state, writes fp32
 *     dq, dk [B,T,H,K]   (with HV > H: summed over the value heads of each head)
 *     dv     [B,T,HV,V]
 *     dbeta  [B,T,HV]
 *     dg     [B,T,HV]    (natural-log gate, as g)
 *     dh0    [N,HV,K,V]  (nullable: not written)
 * The caller owns every buffer; the library-managed workspace of `stream` holds
 * the recomputed states (4 K V bytes per chunk and value head) and a gate buffer.
 * q, k, v, dout, dq and dk must be 16-byte aligned (rows are read by 16-byte loads,
 * four columns of dq and dk added by one 16-byte atomic).
 * Errors: GDN_ERR_INVALID (arguments, a null required pointer, a misaligned one),
 * GDN_ERR_UNSUPPORTED (per-channel gates, chunk_size != 64, K not 32/64/128),
 * GDN_ERR_NOMEM, GDN_ERR_CUDA; nothing is enqueued on an argument error.
 * Asynchronous on `stream`.
 */
gdn_status gdn_chunk_bwd(const gdn_shape *s,
                         const void *q, const void *k, const void *v,
                         const float *g, const float *beta, float scale,
                         const float *h0, const void *dout, const float *dht,
                         const int64_t *cu_seqlens, int chunk_size,
                         float *dq, float *dk, float *dv, float *dbeta, float *dg,
                         float *dh0, gdn_stream_t stream);

/*
 * Context parallel across devices, step 1 (FlashQLA blog, "Key problems in
 * FLA's GDN chunked prefill": the S* / M pre-process; "KDA source
 * walkthrough", the cp_context pre-process of chunk_kda_fwd): the summary of
 * every sequence of this (local) input as one piece of a longer sequence.
 * For sequence n and value head h, with S_end the state after the piece from
 * a start state S_0:  S_end = S*[n,h] + M[n,h] S_0.  Written as
 * summary[N, HV, K, V + K] fp32: row d holds S*[d, 0..V-1] then M[d, 0..K-1].
 * q is not needed.  Arguments otherwise as gdn_chunk_fwd_ex (no h0, no
 * outputs); the split options are ignored (one piece per sequence).
 */
gdn_status gdn_chunk_summary(const gdn_shape *s,
                             const void *k, const void *v,
                             const float *g_or_gk, const float *beta,
                             const int64_t *cu_seqlens, int chunk_size,
                             float *summary, const gdn_options *opt, gdn_stream_t stream);

/*
 * Context parallel, step 2 (same passages): the start state of every piece
 * from the summaries of the pieces before it.  summaries [ranks][pairs][K][V+K]
 * (as gdn_chunk_summary writes them, piece r of each of `pairs` (sequence,
 * head) pairs, gathered in piece order), h0 [pairs][K][V] (nullable: zero),
 * starts [ranks][pairs][K][V]:  starts[0] = h0,
 * starts[r+1] = S*_r + M_r starts[r].  K in {32, 64, 128}; pairs <= 65535.
 * Device pointers; asynchronous on `stream`.
 */
gdn_status gdn_chain_states(int ranks, int pairs, int K, int V, const float *summaries,
                            const float *h0, float *starts, gdn_stream_t stream);

/* Plan summary (host only, no GPU needed) -- what a call would launch: the
 * engine and the in-GPU split (FlashQLA blog, "A balanced solution", the CP
 * enable rule, re-derived for this GPU's SM count). */
typedef struct {
    gdn_engine engine;    /* engine the call would use                    */
    gdn_cp_mode cp_mode;  /* OFF, EXACT or WARMUP after AUTO is resolved   */
    int segment_chunks;   /* chunks per segment (huge when OFF)            */
    int segments;         /* segments per sequence (grid bound)            */
    int value_tiles;      /* CTAs per (sequence, head, segment)            */
    int kernels;          /* kernel launches per call                      */
    size_t workspace_bytes;
} gdn_plan_info;

gdn_status gdn_plan(const gdn_shape *s, int chunk_size, const gdn_options *opt,
                    int num_sms, gdn_plan_info *out);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */

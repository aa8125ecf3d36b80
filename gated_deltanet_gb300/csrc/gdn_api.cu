// C-ABI layer: argument validation, planning, workspace management and the
// launch sequence of one gated delta-rule chunked-prefill forward.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "gdn_internal.cuh"

using namespace gdn;

namespace {

constexpr size_t kStatusBytes = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Plan {
    gdn_engine engine;
    gdn_cp_mode cp;
    int seg_chunks, n_seg, value_tiles, kernels, max_nt;
    float log2_eps;
    // workspace layout
    size_t off_warm, off_segout, off_seginit, off_tiles, off_gc, off_order, tile_slots, bytes;
    size_t off_wdec;  // per-channel gates, warmup split: each chunk's bound on the state's log2-decay
    size_t off_h0t, off_htt, off_rk;  // transposed-state copies; 1 / ||k|| per row (in-kernel L2 norm)
    int n_buckets;
    bool kda;  // tensor-core engine with per-channel gates
};

bool is_varlen(const gdn_shape *s, const int64_t *cu) { return cu != nullptr; }

gdn_status validate_shape(const gdn_shape *s, int chunk_size, const gdn_options *opt)
{
    if (!s) return GDN_ERR_INVALID;
    if (s->B < 0 || s->T < 0 || s->H <= 0 || s->HV <= 0 || s->K <= 0 || s->V <= 0 || s->num_seqs < 0)
        return GDN_ERR_INVALID;
    if (s->HV % s->H != 0) return GDN_ERR_INVALID;
    if (s->qkv_dtype != GDN_F32 && s->qkv_dtype != GDN_BF16) return GDN_ERR_INVALID;
    if (s->gate_kind != GDN_GATE_SCALAR && s->gate_kind != GDN_GATE_CHANNEL) return GDN_ERR_INVALID;
    if (opt) {
        if (opt->cp_mode < GDN_CP_AUTO || opt->cp_mode > GDN_CP_WARMUP) return GDN_ERR_INVALID;
        if (opt->engine < GDN_ENGINE_AUTO || opt->engine > GDN_ENGINE_RECURRENT) return GDN_ERR_INVALID;
        if (opt->segment_chunks < 0 || opt->max_seq_len < 0) return GDN_ERR_INVALID;
        if (!(opt->warmup_log2_eps <= 0.f)) return GDN_ERR_INVALID;
        if (opt->wait_limit_us < 0) return GDN_ERR_INVALID;
        if (!(opt->gate_lower_bound <= 0.f)) return GDN_ERR_INVALID;
        if (opt->gate_dt_bias && !opt->gate_A_log) return GDN_ERR_INVALID;
    }
    if (chunk_size != kChunk) return GDN_ERR_UNSUPPORTED;
    if (s->K != 32 && s->K != 64 && s->K != 128) return GDN_ERR_UNSUPPORTED;
    if (s->V > 4096) return GDN_ERR_UNSUPPORTED;
    return GDN_OK;
}

gdn_status make_plan(const gdn_shape *s, bool varlen, int chunk_size, const gdn_options *optp, int num_sms,
                     Plan *p)
{
    gdn_status st = validate_shape(s, chunk_size, optp);
    if (st != GDN_OK) return st;
    gdn_options opt;
    if (optp) opt = *optp; else gdn_default_options(&opt);
    if (varlen && s->B != 1) return GDN_ERR_INVALID;
    if (!varlen && s->num_seqs != s->B) return GDN_ERR_INVALID;
    if (num_sms <= 0) num_sms = 148;

    const int N = s->num_seqs;
    int maxlen = s->T;
    if (varlen && opt.max_seq_len > 0) maxlen = std::min(opt.max_seq_len, s->T);
    const int max_nt = ceil_div(maxlen, kChunk);

    *p = Plan{};
    const bool channel = s->gate_kind == GDN_GATE_CHANNEL;
    // Token by token ("Flash Linear Attention" page, sec. 8: the layer runs fused_recurrent for short
    // queries): asked for, or AUTO with no sequence longer than kAutoRecurrentTokens.  No split, no
    // workspace beyond the status word.
    if (opt.engine == GDN_ENGINE_RECURRENT ||
        (opt.engine == GDN_ENGINE_AUTO && opt.cp_mode == GDN_CP_AUTO && maxlen <= kAutoRecurrentTokens)) {
        if (opt.cp_mode == GDN_CP_EXACT || opt.cp_mode == GDN_CP_WARMUP) return GDN_ERR_UNSUPPORTED;
        p->engine = GDN_ENGINE_RECURRENT;
        p->cp = GDN_CP_OFF;
        p->value_tiles = ceil_div(s->V, 32);
        p->seg_chunks = std::max(max_nt, 1);
        p->n_seg = 1;
        p->max_nt = max_nt;
        p->kernels = 1;
        p->bytes = kStatusBytes;
        if (opt.state_v_first) {
            const size_t sb = (size_t)s->num_seqs * s->HV * s->K * s->V * sizeof(float);
            p->off_h0t = p->bytes;
            p->off_htt = align_up(p->off_h0t + sb, 256);
            p->bytes = align_up(p->off_htt + sb, 256);
        }
        return GDN_OK;
    }
    // per-channel gates on the tensor-core engine take the warmup split, not the exact one
    const bool tc_ok = tc_shape_ok(s) && !(channel && opt.cp_mode == GDN_CP_EXACT);
    if (opt.engine == GDN_ENGINE_TC && !tc_ok) return GDN_ERR_UNSUPPORTED;
    p->engine = (opt.engine != GDN_ENGINE_SIMT && tc_ok) ? GDN_ENGINE_TC : GDN_ENGINE_SIMT;
    p->kda = p->engine == GDN_ENGINE_TC && channel;
    p->value_tiles = p->engine == GDN_ENGINE_TC ? 1 : ceil_div(s->V, 32);
    p->max_nt = max_nt;
    p->log2_eps = opt.warmup_log2_eps < 0.f ? opt.warmup_log2_eps : -24.f;

    gdn_cp_mode cp = opt.cp_mode;
    const long pairs = (long)N * s->HV;
    if (cp == GDN_CP_AUTO) {
        // Split only when the (sequence, head) pairs leave most SMs idle.  The
        // warmup split costs a few extra chunks per segment; the exact split a
        // pre-pass over the whole sequence plus a serial combine, so it needs
        // a larger idle share to pay off.
        const long base = pairs * p->value_tiles;
        // the warmup split needs ||k|| <= 1 and beta <= 2: asserted by the caller, or made so by the
        // kernels (keys L2-normalised, beta = sigmoid of its logit)
        const bool unit_keys = opt.keys_unit_norm || (opt.qk_l2norm && opt.beta_logits);
        cp = GDN_CP_OFF;
        // per-channel gates bound a window's decay by the slowest channel of every token, so their warmup
        // windows run long and a warmup chunk costs about an emitted one: split them only for four or more
        // segments per pair
        const long need = p->kda ? 4 : 2;
        if (pairs > 0 && unit_keys && base * need <= num_sms && max_nt >= 8) cp = GDN_CP_WARMUP;
        else if (pairs > 0 && base * 4 <= num_sms && max_nt >= 16) cp = GDN_CP_EXACT;
    }
    if (max_nt <= 1 || (p->kda && cp == GDN_CP_EXACT)) cp = GDN_CP_OFF;
    int L;
    if (cp == GDN_CP_OFF) {
        L = std::max(max_nt, 1);
    } else if (opt.segment_chunks > 0) {
        L = opt.segment_chunks;
    } else {
        const long base = std::max(1L, pairs * p->value_tiles);
        // exact: the pre-pass runs S* and M (two value tiles on the tensor-core
        // engine), so leave room for both in one wave
        const long per = cp == GDN_CP_EXACT ? 2 * base : base;
        long segs = std::max(2L, (long)num_sms / per);
        segs = std::min<long>(segs, std::max(2, max_nt / 4));
        L = ceil_div(max_nt, (int)segs);
    }
    L = std::max(L, 1);
    p->cp = cp;
    p->seg_chunks = L;
    p->n_seg = std::max(1, ceil_div(max_nt, L));
    if (p->n_seg == 1 && cp != GDN_CP_OFF) { p->cp = GDN_CP_OFF; cp = GDN_CP_OFF; p->seg_chunks = std::max(max_nt, 1); }

    size_t off = kStatusBytes;
    p->off_warm = p->off_segout = p->off_seginit = p->off_tiles = p->off_gc = p->off_order = p->tile_slots = 0;
    p->off_wdec = 0;
    p->n_buckets = 0;
    if (p->engine == GDN_ENGINE_TC) {
        // operand tiles of every chunk, written by the preparation kernel
        p->tile_slots = (size_t)tile_slots((int64_t)s->B * s->T, N);
        p->off_tiles = off;
        if (p->kda) {
            off = align_up(off + p->tile_slots * s->HV * (kKdaTileBytesPerChunk - 512), 256);
            p->off_gc = off;
            off = align_up(off + p->tile_slots * s->HV * 512, 256);
            if (p->cp == GDN_CP_WARMUP) {
                // the preparation's per-chunk decay bounds, from which each scan CTA finds its warmup start
                p->off_wdec = off;
                off = align_up(off + p->tile_slots * s->HV * sizeof(float), 256);
            }
        } else {
            off = align_up(off + p->tile_slots * s->HV * kTcTileBytesPerChunk, 256);
        }
        if (varlen && N > 1) {
            // packed sequences of different lengths: the preparation sorts them longest first for the scan
            p->off_order = off;
            p->n_buckets = std::min(max_nt + 1, kOrderBuckets);
            off = align_up(off + (size_t)N * sizeof(int), 256);
        }
    }
    const size_t nsegs = (size_t)N * s->HV * p->n_seg;
    if (cp == GDN_CP_WARMUP && p->engine == GDN_ENGINE_TC) {
        p->kernels = 1;  // each CTA of the scan finds its own warmup start
    } else if (cp == GDN_CP_WARMUP) {
        p->off_warm = off;
        off = align_up(off + nsegs * sizeof(int), 256);
        if ((size_t)p->n_seg * L * sizeof(float) > 227 * 1024) return GDN_ERR_UNSUPPORTED;
        p->kernels = 2;
    } else if (cp == GDN_CP_EXACT) {
        p->off_segout = off;
        off = align_up(off + nsegs * s->K * (size_t)(s->V + s->K) * sizeof(float), 256);
        p->off_seginit = off;
        off = align_up(off + nsegs * s->K * (size_t)s->V * sizeof(float), 256);
        p->kernels = 3;
    } else {
        p->kernels = 1;
    }
    if (p->engine == GDN_ENGINE_TC) p->kernels += 1;  // the chunk preparation
    if (opt.qk_l2norm && p->engine == GDN_ENGINE_TC && !p->kda) {
        // 1 / ||k_t|| and 1 / ||q_t|| of every row, from the chunk preparation to the scan
        p->off_rk = off;
        off = align_up(off + 2 * p->tile_slots * s->HV * 64 * sizeof(float), 256);
    }
    if (opt.state_v_first) {
        const size_t sb = (size_t)N * s->HV * s->K * s->V * sizeof(float);
        p->off_h0t = off;
        p->off_htt = align_up(off + sb, 256);
        off = align_up(p->off_htt + sb, 256);
    }
    p->bytes = off;
    return GDN_OK;
}

int current_sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    return sms;
}

gdn_status check_ptrs(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                      const float *beta, const void *o)
{
    const bool any = (size_t)s->B * s->T > 0;
    if (any && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID;
    return GDN_OK;
}

cudaError_t scan_prepass(const ScanArgs &pre, bool tc, const gdn_shape *s, cudaStream_t stream)
{
    if (tc) return launch_tc_scan(pre, 2, false, stream);
    return launch_simt_scan(pre, s->qkv_dtype, s->gate_kind, stream);
}

// Every host-side check of a call, before anything is enqueued: the options (with the engine
// resolved against the pointers' alignment), the plan and the arguments.
gdn_status prepare(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                   const float *beta, float scale, const int64_t *cu, int chunk_size, const void *o,
                   const gdn_options *optp, gdn_options *opt, Plan *p)
{
    if (!s) return GDN_ERR_INVALID;
    if (optp) *opt = *optp; else gdn_default_options(opt);
    // the tensor-core engine needs 16-byte aligned q/k/v/o for its TMA maps (and gk rows)
    if (opt->engine != GDN_ENGINE_SIMT && tc_shape_ok(s) && !tc_supported(s, q, k, v, g, o)) {
        if (opt->engine == GDN_ENGINE_TC) return GDN_ERR_INVALID;
        opt->engine = GDN_ENGINE_SIMT;
    }
    gdn_status st = make_plan(s, is_varlen(s, cu), chunk_size, opt, current_sm_count(), p);
    if (st != GDN_OK) return st;
    if ((st = check_ptrs(s, q, k, v, g, beta, o)) != GDN_OK) return st;
    if (!std::isfinite(scale)) return GDN_ERR_INVALID;
    return GDN_OK;
}

gdn_status run(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
               const float *beta, float scale, const float *h0, const int64_t *cu, int chunk_size, void *o,
               float *ht, const gdn_options *optp, void *ws, size_t ws_bytes, cudaStream_t stream,
               float *chunk_states = nullptr)
{
    Plan p;
    gdn_options opt;
    gdn_status st = prepare(s, q, k, v, g, beta, scale, cu, chunk_size, o, optp, &opt, &p);
    if (st != GDN_OK) return st;
    if (!ws || ws_bytes < p.bytes) return GDN_ERR_WORKSPACE;
    if (((uintptr_t)ws & 255u) != 0) return GDN_ERR_INVALID;

    char *wsb = (char *)ws;
    unsigned *status = (unsigned *)wsb;
    const int N = s->num_seqs;
    const Act act{opt.gate_A_log, opt.gate_dt_bias, opt.gate_lower_bound, opt.beta_logits, opt.qk_l2norm};
    // the transposed state layout: the engines run on canonical [K][V] copies in the workspace
    const float *h0u = h0;
    float *htu = ht;
    if (opt.state_v_first) {
        if (h0) {
            h0u = (const float *)(wsb + p.off_h0t);
            if (launch_transpose(h0, (float *)h0u, N * s->HV, s->V, s->K, stream) != cudaSuccess) return GDN_ERR_CUDA;
        }
        if (ht) htu = (float *)(wsb + p.off_htt);
    }
    auto finish = [&]() -> gdn_status {
        if (opt.state_v_first && ht && launch_transpose(htu, ht, N * s->HV, s->K, s->V, stream) != cudaSuccess)
            return GDN_ERR_CUDA;
        return GDN_OK;
    };

    ScanArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0u; a.cu_seqlens = cu;
    a.o = o; a.ht = htu;
    a.act = act;
    a.B = s->B; a.T = s->T; a.H = s->H; a.HV = s->HV; a.K = s->K; a.V = s->V; a.N = N;
    a.scale = scale;
    a.seg_chunks = p.seg_chunks; a.n_seg = p.n_seg;
    a.mode = kModeForward; a.vext = s->V; a.status = status;
    a.chunk_states = chunk_states;  // (the backward pass: the state entering every chunk; unsplit plans only)
    a.wait_ns = opt.wait_limit_us > 0 ? 1000ull * (unsigned long long)opt.wait_limit_us : 2000000000ull;

    cudaError_t e = cudaSuccess;
    if (p.engine == GDN_ENGINE_RECURRENT) {
        RecArgs ra{};
        ra.q = q; ra.k = k; ra.v = v; ra.g = g; ra.beta = beta; ra.h0 = h0u; ra.cu_seqlens = cu;
        ra.o = o; ra.ht = htu;
        ra.act = act;
        ra.T = s->T; ra.H = s->H; ra.HV = s->HV; ra.K = s->K; ra.V = s->V; ra.N = N; ra.scale = scale;
        if (opt.launch_events && opt.n_launch_events > 0 && opt.launch_events[0])
            cudaEventRecord((cudaEvent_t)opt.launch_events[0], stream);
        e = launch_recurrent(ra, s->qkv_dtype, s->gate_kind, stream);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        if (opt.launch_events && opt.n_launch_events > 1 && opt.launch_events[1])
            cudaEventRecord((cudaEvent_t)opt.launch_events[1], stream);
        return finish();
    }
    // optional per-kernel timing marks on the caller's events
    int n_marks = 0;
    auto mark = [&]() {
        if (opt.launch_events && n_marks < opt.n_launch_events && opt.launch_events[n_marks])
            cudaEventRecord((cudaEvent_t)opt.launch_events[n_marks], stream);
        ++n_marks;
    };
    const bool tc = p.engine == GDN_ENGINE_TC;
    if (tc && p.kda) {
        KdaPrepArgs ka{};
        ka.q = q; ka.k = k; ka.v = v; ka.gk = g; ka.beta = beta; ka.scale = scale; ka.cu_seqlens = cu;
        ka.tiles = wsb + p.off_tiles;
        ka.gc = (float *)(wsb + p.off_gc);
        ka.T = s->T; ka.H = s->H; ka.HV = s->HV; ka.N = N; ka.slots = (int)p.tile_slots;
        if (p.off_order) { ka.seq_order = (int *)(wsb + p.off_order); ka.n_buckets = p.n_buckets; }
        ka.act = act;
        if (p.off_wdec) ka.wdec = (float *)(wsb + p.off_wdec);
        // the warmup split needs beta ||k||^2 <= 2: checked unless the keys are normalised in the kernel
        ka.check_norm = p.cp == GDN_CP_WARMUP && !opt.qk_l2norm;
        ka.status = status;
        a.seq_order = ka.seq_order;
        mark();
        e = launch_kda_prep(ka, stream);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        a.tiles = ka.tiles;
        a.tile_slots = ka.slots;
        a.kda_gc = ka.gc;
        a.kda_wdec = ka.wdec;
    } else if (tc) {
        PrepArgs pa{};
        pa.k = k; pa.g = g; pa.beta = beta; pa.cu_seqlens = cu;
        pa.tiles = wsb + p.off_tiles;
        pa.T = s->T; pa.H = s->H; pa.HV = s->HV; pa.N = N; pa.slots = (int)p.tile_slots;
        pa.check_norm = p.cp == GDN_CP_WARMUP;
        if (p.off_order) { pa.seq_order = (int *)(wsb + p.off_order); pa.n_buckets = p.n_buckets; }
        a.seq_order = pa.seq_order;
        pa.status = status;
        pa.wait_ns = a.wait_ns;
        pa.act = act;
        if (p.off_rk) {
            pa.rk = (float *)(wsb + p.off_rk);
            pa.rq = pa.rk + p.tile_slots * s->HV * 64;
            pa.q = q;
        }
        a.rk = pa.rk;
        a.rq = pa.rq;
        mark();
        e = launch_tc_prep(pa, stream);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        a.tiles = pa.tiles;
        a.tile_slots = pa.slots;
    }
    auto scan = [&](const ScanArgs &sa) -> cudaError_t {
        if (tc) return launch_tc_scan(sa, sa.mode == kModePrepass ? 2 : 1, p.kda, stream);
        return launch_simt_scan(sa, s->qkv_dtype, s->gate_kind, stream);
    };
    if (p.cp == GDN_CP_WARMUP && tc) {
        a.warm_in_kernel = 1;
        a.warm_log2_eps = p.log2_eps;
    } else if (p.cp == GDN_CP_WARMUP) {
        GateStatsArgs gs{};
        gs.g = g; gs.beta = beta; gs.cu_seqlens = cu;
        gs.warm_start = (int *)(wsb + p.off_warm);
        gs.T = s->T; gs.HV = s->HV; gs.K = s->K; gs.N = N;
        gs.seg_chunks = p.seg_chunks; gs.n_seg = p.n_seg;
        gs.channel = s->gate_kind == GDN_GATE_CHANNEL;
        gs.log2_eps = p.log2_eps;
        gs.act = act;
        gs.max_warm_chunks = 1 << 30;
        mark();
        e = launch_gate_stats(gs, stream);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        a.warm_start = gs.warm_start;
    } else if (p.cp == GDN_CP_EXACT) {
        ScanArgs pre = a;
        pre.mode = kModePrepass;
        pre.vext = s->V + s->K;
        pre.seg_out = (float *)(wsb + p.off_segout);
        mark();
        e = scan_prepass(pre, tc, s, stream);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        CombineArgs cb{};
        cb.h0 = h0u; cb.cu_seqlens = cu; cb.seg_out = pre.seg_out;
        cb.seg_init = (float *)(wsb + p.off_seginit);
        cb.T = s->T; cb.HV = s->HV; cb.K = s->K; cb.V = s->V; cb.N = N;
        cb.seg_chunks = p.seg_chunks; cb.n_seg = p.n_seg; cb.status = status;
        mark();
        e = launch_cp_combine(cb, stream);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        a.seg_init = cb.seg_init;
    }
    mark();
    a.withhold_full0 = opt.test_withhold_first_arrival != 0;
    e = scan(a);
    if (e != cudaSuccess) return GDN_ERR_CUDA;
    mark();
    return finish();
}

// ---------------------------------------------------------------- library-managed workspaces
struct WsEntry {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, WsEntry> g_ws;

gdn_status managed_ws(size_t need, cudaStream_t stream, void **out, size_t *out_bytes)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    WsEntry &w = g_ws[{dev, stream}];
    if (w.bytes < need) {
        if (w.ptr) cudaFreeAsync(w.ptr, stream);
        w.ptr = nullptr;
        w.bytes = 0;
        size_t bytes = align_up(std::max<size_t>(need, 1 << 20), 1 << 20);
        if (cudaMallocAsync(&w.ptr, bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return GDN_ERR_NOMEM;
        }
        if (cudaMemsetAsync(w.ptr, 0, kStatusBytes, stream) != cudaSuccess) return GDN_ERR_CUDA;
        w.bytes = bytes;
    }
    *out = w.ptr;
    *out_bytes = w.bytes;
    return GDN_OK;
}

}  // namespace

gdn_status gdn::check_call(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, const int64_t *cu, int chunk_size, const void *o,
                           const gdn_options *opt, size_t *ws_bytes)
{
    Plan p;
    gdn_options o2;
    const gdn_status st = prepare(s, q, k, v, g, beta, scale, cu, chunk_size, o, opt, &o2, &p);
    if (st == GDN_OK && ws_bytes) *ws_bytes = p.bytes;
    return st;
}

gdn_status gdn::read_status_word(void *ws, cudaStream_t st)
{
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof(unsigned), st) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
    if (word & kStatusTimeout) return GDN_ERR_TIMEOUT;
    if (word & (kStatusPlan | kStatusNormBound)) return GDN_ERR_INVALID;
    return GDN_OK;
}

extern "C" {

void gdn_default_options(gdn_options *opt)
{
    if (!opt) return;
    std::memset(opt, 0, sizeof(*opt));
    opt->cp_mode = GDN_CP_AUTO;
    opt->engine = GDN_ENGINE_AUTO;
}

const char *gdn_status_string(gdn_status st)
{
    switch (st) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID: return "GDN_ERR_INVALID: invalid argument";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: valid but not supported";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: CUDA runtime error";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT: a bounded device wait ran out";
    case GDN_ERR_NOMEM: return "GDN_ERR_NOMEM: workspace allocation failed";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace too small";
    }
    return "GDN_ERR_UNKNOWN";
}

int gdn_version(void) { return 100; }

size_t gdn_workspace_size(const gdn_shape *s, int chunk_size, const gdn_options *opt)
{
    if (!s) return 0;
    Plan p;
    // Sized for the worst case over SM counts the planner may see: use the
    // device's count when a device is current, else a nominal one.
    if (make_plan(s, false, chunk_size, opt, current_sm_count(), &p) != GDN_OK &&
        make_plan(s, true, chunk_size, opt, current_sm_count(), &p) != GDN_OK)
        return 0;
    Plan pv;
    if (s->B == 1 && make_plan(s, true, chunk_size, opt, current_sm_count(), &pv) == GDN_OK)
        p.bytes = std::max(p.bytes, pv.bytes);
    return p.bytes;
}

gdn_status gdn_plan(const gdn_shape *s, int chunk_size, const gdn_options *opt, int num_sms, gdn_plan_info *out)
{
    if (!out || !s) return GDN_ERR_INVALID;
    Plan p;
    const bool varlen = s->num_seqs != s->B || (opt && opt->max_seq_len > 0);
    gdn_status st = make_plan(s, varlen, chunk_size, opt, num_sms, &p);
    if (st != GDN_OK) return st;
    out->engine = p.engine;
    out->cp_mode = p.cp;
    out->segment_chunks = p.seg_chunks;
    out->segments = p.n_seg;
    out->value_tiles = p.value_tiles;
    out->kernels = p.kernels;
    out->workspace_bytes = p.bytes;
    return GDN_OK;
}

gdn_status gdn_chunk_fwd_ws(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float scale, const float *h0, const int64_t *cu, int chunk_size,
                            void *o, float *ht, const gdn_options *opt, void *workspace, size_t ws_bytes,
                            gdn_stream_t stream)
{
    return run(s, q, k, v, g, beta, scale, h0, cu, chunk_size, o, ht, opt, workspace, ws_bytes,
               (cudaStream_t)stream);
}

gdn_status gdn_chunk_fwd_ex(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float scale, const float *h0, const int64_t *cu, int chunk_size,
                            void *o, float *ht, const gdn_options *opt, gdn_stream_t stream)
{
    Plan p;
    gdn_status st = make_plan(s, cu != nullptr, chunk_size, opt, current_sm_count(), &p);
    if (st != GDN_OK) return st;
    if ((st = check_ptrs(s, q, k, v, g, beta, o)) != GDN_OK) return st;
    if (!std::isfinite(scale)) return GDN_ERR_INVALID;
    void *ws = nullptr;
    size_t bytes = 0;
    st = managed_ws(p.bytes, (cudaStream_t)stream, &ws, &bytes);
    if (st != GDN_OK) return st;
    return run(s, q, k, v, g, beta, scale, h0, cu, chunk_size, o, ht, opt, ws, bytes, (cudaStream_t)stream);
}

gdn_status gdn_chunk_fwd(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                         const float *beta, float scale, const float *h0, const int64_t *cu, int chunk_size,
                         void *o, float *ht, gdn_stream_t stream)
{
    return gdn_chunk_fwd_ex(s, q, k, v, g, beta, scale, h0, cu, chunk_size, o, ht, nullptr, stream);
}

gdn_status gdn_chunk_summary(const gdn_shape *s, const void *k, const void *v, const float *g, const float *beta,
                             const int64_t *cu, int chunk_size, float *summary, const gdn_options *optp,
                             gdn_stream_t stream)
{
    if (!s || !summary) return GDN_ERR_INVALID;
    gdn_options opt;
    if (optp) opt = *optp; else gdn_default_options(&opt);
    if (opt.engine == GDN_ENGINE_RECURRENT) return GDN_ERR_UNSUPPORTED;
    // one segment per sequence: no split; per-channel gates take the CUDA-core engine's pre-pass
    opt.cp_mode = GDN_CP_OFF;
    if (s->gate_kind == GDN_GATE_CHANNEL) {
        if (opt.engine == GDN_ENGINE_TC) return GDN_ERR_UNSUPPORTED;
        opt.engine = GDN_ENGINE_SIMT;
    }
    Plan p;
    gdn_options o2;
    // q is not read by the pre-pass and o is not written: k and v stand in for their shapes
    gdn_status st = prepare(s, k, k, v, g, beta, 1.f, cu, chunk_size, v, &opt, &o2, &p);
    if (st != GDN_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    if ((st = managed_ws(p.bytes, cs, &ws, &ws_bytes)) != GDN_OK) return st;
    char *wsb = (char *)ws;
    const bool tc = p.engine == GDN_ENGINE_TC;
    ScanArgs a{};
    a.q = k; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = nullptr; a.cu_seqlens = cu;
    a.o = const_cast<void *>(v); a.ht = nullptr;
    a.B = s->B; a.T = s->T; a.H = s->H; a.HV = s->HV; a.K = s->K; a.V = s->V; a.N = s->num_seqs;
    a.scale = 1.f;
    a.seg_chunks = std::max(p.max_nt, 1);
    a.n_seg = 1;
    a.mode = kModePrepass;
    a.vext = s->V + s->K;
    a.seg_out = summary;
    a.status = (unsigned *)wsb;
    a.act = Act{opt.gate_A_log, opt.gate_dt_bias, opt.gate_lower_bound, opt.beta_logits, opt.qk_l2norm};
    a.wait_ns = opt.wait_limit_us > 0 ? 1000ull * (unsigned long long)opt.wait_limit_us : 2000000000ull;
    cudaError_t e;
    if (tc) {
        PrepArgs pa{};
        pa.k = k; pa.g = g; pa.beta = beta; pa.cu_seqlens = cu;
        pa.tiles = wsb + p.off_tiles;
        pa.T = s->T; pa.H = s->H; pa.HV = s->HV; pa.N = s->num_seqs; pa.slots = (int)p.tile_slots;
        if (p.off_order) { pa.seq_order = (int *)(wsb + p.off_order); pa.n_buckets = p.n_buckets; }
        pa.status = a.status;
        pa.wait_ns = a.wait_ns;
        pa.act = a.act;
        if (p.off_rk) {
            pa.rk = (float *)(wsb + p.off_rk);
            pa.rq = pa.rk + p.tile_slots * s->HV * 64;
            pa.q = a.q;
        }
        a.rk = pa.rk;
        a.rq = pa.rq;
        if ((e = launch_tc_prep(pa, cs)) != cudaSuccess) return GDN_ERR_CUDA;
        a.tiles = pa.tiles;
        a.tile_slots = pa.slots;
        a.seq_order = pa.seq_order;
        e = launch_tc_scan(a, 2, false, cs);
    } else {
        e = launch_simt_scan(a, s->qkv_dtype, s->gate_kind, cs);
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_chain_states(int ranks, int pairs, int K, int V, const float *summaries, const float *h0,
                            float *starts, gdn_stream_t stream)
{
    if (ranks < 1 || pairs < 0 || V <= 0 || !starts || (ranks > 1 && !summaries)) return GDN_ERR_INVALID;
    if (K != 32 && K != 64 && K != 128) return GDN_ERR_UNSUPPORTED;
    if (pairs > 65535) return GDN_ERR_UNSUPPORTED;
    ChainArgs a{summaries, h0, starts, ranks, pairs, K, V};
    return launch_chain_states(a, (cudaStream_t)stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_recurrent_fwd(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                             const float *beta, float scale, const float *h0, const int64_t *cu, void *o, float *ht,
                             gdn_stream_t stream)
{
    gdn_options opt;
    gdn_default_options(&opt);
    opt.engine = GDN_ENGINE_RECURRENT;
    return gdn_chunk_fwd_ex(s, q, k, v, g, beta, scale, h0, cu, kChunk, o, ht, &opt, stream);
}

gdn_status gdn_chunk_bwd(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                         const float *beta, float scale, const float *h0, const void *dout, const float *dht,
                         const int64_t *cu, int chunk_size, float *dq, float *dk, float *dv, float *dbeta,
                         float *dg, float *dh0, gdn_stream_t stream)
{
    gdn_status st = validate_shape(s, chunk_size, nullptr);
    if (st != GDN_OK) return st;
    if (s->gate_kind != GDN_GATE_SCALAR) return GDN_ERR_UNSUPPORTED;
    const bool varlen = cu != nullptr;
    if (varlen && s->B != 1) return GDN_ERR_INVALID;
    if (!varlen && s->num_seqs != s->B) return GDN_ERR_INVALID;
    if (!std::isfinite(scale)) return GDN_ERR_INVALID;
    const int64_t tokens = (int64_t)s->B * s->T;
    if (tokens > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dbeta || !dg))
        return GDN_ERR_INVALID;
    // rows of q, k, v and dO are read by 16-byte loads, dq and dk summed four columns at a time by 16-byte
    // atomics
    auto aligned = [](const void *p, uintptr_t m) { return ((uintptr_t)p & (m - 1)) == 0; };
    if (tokens > 0 && (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dout, 16) ||
                       !aligned(dq, 16) || !aligned(dk, 16)))
        return GDN_ERR_INVALID;
    const int N = s->num_seqs;
    cudaStream_t cs = (cudaStream_t)stream;
    // the tensor-core forward recomputes the states when it can (bf16, d = 128, aligned), unsplit
    gdn_options fopt;
    gdn_default_options(&fopt);
    fopt.engine = GDN_ENGINE_TC;
    fopt.cp_mode = GDN_CP_OFF;
    Plan fp;
    const bool tc_engine = tc_shape_ok(s) && tc_supported(s, q, k, v, g, nullptr) &&
                           make_plan(s, varlen, chunk_size, &fopt, current_sm_count(), &fp) == GDN_OK &&
                           fp.engine == GDN_ENGINE_TC;
    // workspace: the forward's (status word first), the state entering every chunk (fp32), the forward's
    // output (scratch, tensor-core engine only), the per-row gate gradient dG
    const size_t slots = (size_t)tile_slots(tokens, N);
    const size_t off_states = align_up(tc_engine ? fp.bytes : kStatusBytes, 256);
    const size_t off_o = align_up(off_states + slots * s->HV * (size_t)s->K * s->V * sizeof(float), 256);
    const size_t off_dG =
        align_up(off_o + (tc_engine ? (size_t)tokens * s->HV * s->V * (s->qkv_dtype == GDN_BF16 ? 2 : 4) : 0), 256);
    const size_t chunk_heads = slots * s->HV, tiles = (size_t)ceil_div(s->V, 32);
    const size_t off_A = align_up(off_dG + (size_t)tokens * s->HV * sizeof(float), 256);
    const size_t off_P = off_A + chunk_heads * 64 * 64 * sizeof(float);
    const size_t off_dP = off_P + chunk_heads * 64 * 64 * sizeof(float);
    const size_t off_dA = off_dP + tiles * chunk_heads * 64 * 64 * sizeof(float);
    const size_t bytes = align_up(off_dA + tiles * chunk_heads * 64 * 64 * sizeof(float), 256);
    void *ws = nullptr;
    size_t ws_bytes = 0;
    if ((st = managed_ws(bytes, cs, &ws, &ws_bytes)) != GDN_OK) return st;
    char *wsb = (char *)ws;
    if (tokens == 0) {
        // no token: dh0 = dht
        if (dh0 && (size_t)N * s->HV > 0) {
            const size_t sb = (size_t)N * s->HV * s->K * s->V * sizeof(float);
            cudaError_t e = dht ? cudaMemcpyAsync(dh0, dht, sb, cudaMemcpyDeviceToDevice, cs)
                                : cudaMemsetAsync(dh0, 0, sb, cs);
            if (e != cudaSuccess) return GDN_ERR_CUDA;
        }
        return GDN_OK;
    }
    // the sums (over value tiles, GVA heads) start at zero
    if (cudaMemsetAsync(dq, 0, (size_t)tokens * s->H * s->K * sizeof(float), cs) != cudaSuccess ||
        cudaMemsetAsync(dk, 0, (size_t)tokens * s->H * s->K * sizeof(float), cs) != cudaSuccess ||
        cudaMemsetAsync(dbeta, 0, (size_t)tokens * s->HV * sizeof(float), cs) != cudaSuccess ||
        cudaMemsetAsync(wsb + off_dG, 0, (size_t)tokens * s->HV * sizeof(float), cs) != cudaSuccess)
        return GDN_ERR_CUDA;
    const int max_nt = ceil_div(s->T, kChunk);
    float *states = (float *)(wsb + off_states);
    // Steps 1-2 of the backward: the states entering every chunk.  On the tensor-core engine when the
    // shape and pointers allow (its forward, unsplit, with a state dump; o to scratch), else by the
    // CUDA-core engine's forward (no output, no split).
    if (tc_engine) {
        if ((st = run(s, q, k, v, g, beta, scale, h0, cu, chunk_size, wsb + off_o, nullptr, &fopt, ws, ws_bytes, cs,
                      states)) != GDN_OK)
            return st;
    } else {
    ScanArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.cu_seqlens = cu;
    a.o = nullptr; a.ht = nullptr;
    a.B = s->B; a.T = s->T; a.H = s->H; a.HV = s->HV; a.K = s->K; a.V = s->V; a.N = N;
    a.scale = scale;
    a.seg_chunks = std::max(max_nt, 1);
    a.n_seg = 1;
    a.mode = kModeForward;
    a.vext = s->V;
    a.status = (unsigned *)wsb;
    a.chunk_states = states;
    if (launch_simt_scan(a, s->qkv_dtype, GDN_GATE_SCALAR, cs) != cudaSuccess) return GDN_ERR_CUDA;
    }
    // Steps 3-7
    BwdArgs b{};
    b.q = q; b.k = k; b.v = v; b.dout = dout; b.g = g; b.beta = beta; b.dht = dht; b.cu_seqlens = cu;
    b.chunk_states = states;
    b.dq = dq; b.dk = dk; b.dv = dv; b.dbeta = dbeta; b.dG = (float *)(wsb + off_dG); b.dg = dg; b.dh0 = dh0;
    b.Abuf = (float *)(wsb + off_A); b.Pbuf = (float *)(wsb + off_P);
    b.dPbuf = (float *)(wsb + off_dP); b.dAbuf = (float *)(wsb + off_dA); b.chunk_heads = chunk_heads;
    b.T = s->T; b.H = s->H; b.HV = s->HV; b.K = s->K; b.V = s->V; b.N = N; b.max_nt = max_nt;
    b.scale = scale;
    return launch_chunk_bwd(b, s->qkv_dtype, cs) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_read_device_status(void *workspace, gdn_stream_t stream)
{
    cudaStream_t st = (cudaStream_t)stream;
    void *ws = workspace;
    if (!ws) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_ws.find({dev, st});
        if (it == g_ws.end() || !it->second.ptr) return GDN_OK;
        ws = it->second.ptr;
    }
    return gdn::read_status_word(ws, st);
}

gdn_status gdn_chunk_fwd_host(const gdn_shape *s, const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float scale, const float *h0, const int64_t *cu, int chunk_size,
                              void *o, float *ht, const gdn_options *opt, gdn_stream_t stream)
{
    Plan p;
    gdn_status st = make_plan(s, cu != nullptr, chunk_size, opt, current_sm_count(), &p);
    if (st != GDN_OK) return st;
    if ((st = check_ptrs(s, q, k, v, g, beta, o)) != GDN_OK) return st;
    const int N = s->num_seqs;
    const int64_t tokens = (int64_t)s->B * s->T;
    if (cu) {
        // host offsets: checked here, since the groups below are cut along them
        if (cu[0] != 0 || cu[N] != tokens) return GDN_ERR_INVALID;
        for (int n = 0; n < N; ++n)
            if (cu[n + 1] < cu[n]) return GDN_ERR_INVALID;
    }
    cudaStream_t cs = (cudaStream_t)stream;
    const size_t esz = s->qkv_dtype == GDN_BF16 ? 2 : 4;
    const size_t gch = s->gate_kind == GDN_GATE_CHANNEL ? (size_t)s->K : 1;
    // bytes per token of each token-major tensor, per sequence of each state
    const size_t tq = (size_t)s->H * s->K * esz, tv = (size_t)s->HV * s->V * esz, tg = (size_t)s->HV * gch * 4,
                 tb = (size_t)s->HV * 4, sh = (size_t)s->HV * s->K * s->V * 4;
    enum { E_Q, E_K, E_V, E_G, E_BETA, E_H0, E_CU, E_O, E_HT, E_N };
    const size_t sizes[E_N] = {tokens * tq, tokens * tq, tokens * tv, tokens * tg, tokens * tb, h0 ? N * sh : 0,
                              cu ? (size_t)(N + 4) * 8 * 4 : 0, tokens * tv, ht ? N * sh : 0};
    size_t offs[E_N], total = 0;
    for (int i = 0; i < E_N; ++i) {
        offs[i] = total;
        total = align_up(total + sizes[i], 256);
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
    // Library-owned per device: the arena (per caller stream) and two copy streams with a pool of
    // events.  The call is split into up to four groups of whole sequences (contiguous token ranges
    // in every tensor): the inputs of group i+1 are copied in while group i runs on the caller's
    // stream and group i-1's outputs are copied out, each direction on its own stream.
    constexpr int kGroups = 4;
    struct HostRes {
        cudaStream_t in = nullptr, out = nullptr;
        cudaEvent_t ev[3 * kGroups + 1] = {};
    };
    static std::map<int, HostRes> res;
    static std::map<std::pair<int, cudaStream_t>, WsEntry> arenas;
    void *arena = nullptr;
    HostRes *r = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        HostRes &hr = res[dev];
        if (!hr.in) {
            if (cudaStreamCreateWithFlags(&hr.in, cudaStreamNonBlocking) != cudaSuccess ||
                cudaStreamCreateWithFlags(&hr.out, cudaStreamNonBlocking) != cudaSuccess) {
                cudaGetLastError();
                return GDN_ERR_CUDA;
            }
            for (auto &e : hr.ev)
                if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return GDN_ERR_CUDA;
        }
        r = &hr;
        WsEntry &w = arenas[{dev, cs}];
        if (w.bytes < total) {
            if (w.ptr) cudaFreeAsync(w.ptr, cs);
            w.ptr = nullptr;
            w.bytes = 0;
            const size_t bytes = align_up(std::max<size_t>(total, 1 << 20), 1 << 20);
            if (cudaMallocAsync(&w.ptr, bytes, cs) != cudaSuccess) {
                cudaGetLastError();
                return GDN_ERR_NOMEM;
            }
            w.bytes = bytes;
        }
        arena = w.ptr;
    }
    char *A = (char *)arena;
    // groups of whole sequences with about equal token counts
    const int G = std::max(1, std::min(N, kGroups));
    int bound[kGroups + 1];
    bound[0] = 0;
    auto seq_start = [&](int n) -> int64_t { return cu ? cu[n] : (int64_t)n * s->T; };
    for (int gi = 1; gi < G; ++gi) {
        int n = bound[gi - 1] + 1;
        while (n < N - (G - gi) && seq_start(n) < tokens * gi / G) ++n;
        bound[gi] = n;
    }
    bound[G] = N;
    // the arena (and the events) must not be in use by a previous call still in flight on the copy
    // streams: each call synchronises the caller's stream, which waits for both, before returning
    if (cudaEventRecord(r->ev[3 * kGroups], cs) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamWaitEvent(r->in, r->ev[3 * kGroups], 0) != cudaSuccess) return GDN_ERR_CUDA;
    int64_t *cu_dev_base = cu ? (int64_t *)(A + offs[E_CU]) : nullptr;
    std::vector<int64_t> cu_rebased;
    if (cu) cu_rebased.resize((size_t)N + G);
    size_t cu_pos = 0;
    for (int gi = 0; gi < G; ++gi) {
        const int n0 = bound[gi], n1 = bound[gi + 1], ng = n1 - n0;
        const int64_t t0 = seq_start(n0), t1 = n1 < N ? seq_start(n1) : tokens, tg_n = t1 - t0;
        auto in = [&](int which, const void *src, size_t off, size_t bytes) -> bool {
            return bytes == 0 || cudaMemcpyAsync(A + offs[which] + off, (const char *)src + off, bytes,
                                                 cudaMemcpyHostToDevice, r->in) == cudaSuccess;
        };
        if (!in(E_Q, q, t0 * tq, tg_n * tq) || !in(E_K, k, t0 * tq, tg_n * tq) || !in(E_V, v, t0 * tv, tg_n * tv) ||
            !in(E_G, g, t0 * tg, tg_n * tg) || !in(E_BETA, beta, t0 * tb, tg_n * tb) ||
            (h0 && !in(E_H0, h0, n0 * sh, (size_t)ng * sh)))
            return GDN_ERR_CUDA;
        const int64_t *cu_g = nullptr;
        if (cu) {
            int64_t *hcu = cu_rebased.data() + cu_pos;
            for (int i = 0; i <= ng; ++i) hcu[i] = cu[n0 + i] - t0;
            // pageable source: staged by the runtime before the call returns
            if (cudaMemcpyAsync(cu_dev_base + cu_pos, hcu, (size_t)(ng + 1) * 8, cudaMemcpyHostToDevice, r->in) !=
                cudaSuccess)
                return GDN_ERR_CUDA;
            cu_g = cu_dev_base + cu_pos;
            cu_pos += (size_t)ng + 1;
        }
        if (cudaEventRecord(r->ev[3 * gi], r->in) != cudaSuccess || cudaStreamWaitEvent(cs, r->ev[3 * gi], 0) != cudaSuccess)
            return GDN_ERR_CUDA;
        gdn_shape sg = *s;
        if (cu) {
            sg.T = (int)tg_n;  // B == 1
        } else {
            sg.B = ng;
        }
        sg.num_seqs = ng;
        st = gdn_chunk_fwd_ex(&sg, A + offs[E_Q] + t0 * tq, A + offs[E_K] + t0 * tq, A + offs[E_V] + t0 * tv,
                              (const float *)(A + offs[E_G] + t0 * tg), (const float *)(A + offs[E_BETA] + t0 * tb), scale,
                              h0 ? (const float *)(A + offs[E_H0] + n0 * sh) : nullptr, cu_g, chunk_size,
                              A + offs[E_O] + t0 * tv, ht ? (float *)(A + offs[E_HT] + n0 * sh) : nullptr, opt, stream);
        if (st != GDN_OK) return st;
        if (cudaEventRecord(r->ev[3 * gi + 1], cs) != cudaSuccess ||
            cudaStreamWaitEvent(r->out, r->ev[3 * gi + 1], 0) != cudaSuccess)
            return GDN_ERR_CUDA;
        if (tg_n > 0 && cudaMemcpyAsync((char *)o + t0 * tv, A + offs[E_O] + t0 * tv, tg_n * tv, cudaMemcpyDeviceToHost,
                                        r->out) != cudaSuccess)
            return GDN_ERR_CUDA;
        if (ht && ng > 0 &&
            cudaMemcpyAsync((char *)ht + n0 * sh, A + offs[E_HT] + n0 * sh, (size_t)ng * sh, cudaMemcpyDeviceToHost,
                            r->out) != cudaSuccess)
            return GDN_ERR_CUDA;
    }
    if (cudaEventRecord(r->ev[3 * kGroups - 1], r->out) != cudaSuccess ||
        cudaStreamWaitEvent(cs, r->ev[3 * kGroups - 1], 0) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // extern "C"

// Allocation-free entry point: the forward pass with its scratch (the
// device status word and the chunk-parallel split's tables) in a fixed
// file-scope device array instead of a caller- or library-allocated workspace.
//
// Some callers cannot allocate device memory at the time they run the
// forward: code that executes inside a memory pool they do not own, a
// runtime that forbids cudaMalloc on its hot path (it would synchronise the
// device and break stream-ordered execution), or an embedding that has
// reserved all device memory up front.  They can use this entry point.
#include <mutex>

#include "gdn_internal.cuh"

namespace {

// Held by every GPU that loads the library, from load until process exit.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_static_scratch on the current device.  The symbol's
// name in host code is only a host-side stand-in; the address must come from
// cudaGetSymbolAddress with the device current (done once per device).
gdn_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return GDN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_chunk_fwd_noalloc(const gdn_shape *s, const void *q, const void *k, const void *v,
                                            const float *g_or_gk, const float *beta, float scale,
                                            const float *h0, const int64_t *cu_seqlens, int chunk_size,
                                            void *o, float *ht, const gdn_options *opt, gdn_stream_t stream)
{
    // Every host-side check first (the same codes as the other entry points), so a rejected call
    // enqueues nothing and leaves the status word of an earlier call untouched.
    size_t need = 0;
    gdn_status st = gdn::check_call(s, q, k, v, g_or_gk, beta, scale, cu_seqlens, chunk_size, o, opt, &need);
    if (st != GDN_OK) return st;
    if (need > kStaticScratchBytes) return GDN_ERR_WORKSPACE;  // plan needs more than the fixed array
    void *ws = nullptr;
    st = scratch_address(&ws);
    if (st != GDN_OK) return st;
    // The array keeps the previous call's contents.  The split tables are written in full before
    // they are read; the status word starts at zero (device memory of the module is zero-initialised)
    // and, as a workspace's, collects the device errors of every call until gdn_read_noalloc_status.
    return gdn_chunk_fwd_ws(s, q, k, v, g_or_gk, beta, scale, h0, cu_seqlens, chunk_size, o, ht, opt, ws,
                            kStaticScratchBytes, stream);
}

extern "C" gdn_status gdn_read_noalloc_status(gdn_stream_t stream)
{
    void *ws = nullptr;
    const gdn_status st = scratch_address(&ws);
    if (st != GDN_OK) return st;
    return gdn::read_status_word(ws, (cudaStream_t)stream);
}

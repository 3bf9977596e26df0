// decode_static.cu -- na_attn_decode with library-owned scratch.
//
// Some callers cannot hand the library a workspace: a plugin running inside
// another runtime that owns every device allocation and exposes no allocator,
// or a serving loop that must not allocate device memory once it has started.
// This entry point runs the same split-KV decode as na_attn_decode, but keeps
// the per-split partial results in a fixed device array defined in this file,
// so the call itself allocates nothing.
//
// The array is NA_STATIC_DECODE_SCRATCH_BYTES (20 MiB) and lives for as long as
// the library is loaded, on every GPU that loads it.  All calls share it and it
// keeps whatever the last call left there.  The decode needs nothing in it to
// start at zero: the split pass writes every partial row and every stream's
// piece span that the merge pass reads, in the same call -- a CTA whose wait
// gave up writes a marker row that the merge pass reports instead of merging.
// Two calls whose kernels overlap on the GPU (different streams, or several
// host threads) race on it and give wrong results.
//
// The array's device address is looked up once per device and kept; a
// cudaDeviceReset() of that device unloads the module and invalidates it, so
// this entry point must not be called on a device after it was reset.
#include <mutex>

#include "na_internal.cuh"

#define NA_STATIC_DECODE_SCRATCH_BYTES (20u << 20)

static __device__ __align__(256) unsigned char g_decode_scratch[NA_STATIC_DECODE_SCRATCH_BYTES];

namespace {

std::mutex g_lock;
void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array for the current device, looked up once
// per device (host code only sees a stand-in for the symbol).
void *scratch_for_current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess)
            return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int na_attn_decode_static_ws(const na_attn_cfg *cfg, int32_t batch, const void *q_rot,
                                        const na_kv_cache *cache, const int32_t *kv_lens,
                                        int32_t max_kv_len, const void *gate, void *out,
                                        float *probs, int32_t probs_stride, int32_t num_splits,
                                        int32_t *status, void *stream)
{
    size_t need = 0;
    int rc = na_decode_workspace_size(cfg, batch, max_kv_len, num_splits, &need);
    if (rc != NA_OK)
        return rc;
    if (need > NA_STATIC_DECODE_SCRATCH_BYTES)
        return NA_ERR_WORKSPACE;
    void *scratch = scratch_for_current_device();
    if (!scratch)
        return NA_ERR_CUDA;
    return na_attn_decode(cfg, batch, q_rot, cache, kv_lens, max_kv_len, gate, out, probs,
                          probs_stride, num_splits, scratch, NA_STATIC_DECODE_SCRATCH_BYTES,
                          status, stream);
}

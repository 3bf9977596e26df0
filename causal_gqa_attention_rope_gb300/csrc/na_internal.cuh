// na_internal.cuh -- device helpers and launch parameter blocks shared by the
// kernels of the attention library (sm_103a).
#pragma once

#include <atomic>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "na.h"

typedef __nv_bfloat16 bf16;

// A kernel gives up a wait after this many SM clock cycles (about a second)
// and reports NA_ERR_DEVICE_TIMEOUT instead of hanging the device.
#define NA_WAIT_LIMIT_CYCLES (1ll << 31)

#define NA_LOG2E 1.4426950408889634f

// ------------------------------------------------------------------ status --

// Keep the first error a kernel reports.
__device__ __forceinline__ void na_report(int32_t *status, int code)
{
    if (status)
        atomicCAS(status, 0, code);
}

// ------------------------------------------------------------------- bf16 --

// Widen eight packed bf16 values (one 16-byte chunk) to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float *f)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Round two fp32 values to bf16 (round to nearest even) and pack them.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float *f)
{
    uint4 u;
    u.x = pack_bf16x2(f[0], f[1]);
    u.y = pack_bf16x2(f[2], f[3]);
    u.z = pack_bf16x2(f[4], f[5]);
    u.w = pack_bf16x2(f[6], f[7]);
    return u;
}

// ------------------------------------------------------ shared-memory sync --

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false after
// NA_WAIT_LIMIT_CYCLES without completion.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long start = clock64();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; i++)
            if (mbar_try_wait(bar, parity))
                return true;
        if (clock64() - start > NA_WAIT_LIMIT_CYCLES)
            return false;
    }
}

// One-dimensional bulk copy global -> shared, completing on `bar` (the
// transaction count must be announced with mbar_arrive_expect_tx).  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Named barrier over a subset of warps.
__device__ __forceinline__ void named_barrier_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------- programmatic dependent launch --
// Every kernel of this library is launched with programmatic stream
// serialization, so it may be scheduled while its predecessor in the stream is
// still finishing.  Each kernel first does the part of its prologue that reads
// no global memory (barrier set-up, tensor-memory allocation, descriptor
// prefetch), then grid_dependency_wait() -- it returns once every prerequisite
// grid has completed and its writes are visible, at once when there is none --
// and then grid_dependents_launch(), after which the next kernel in the stream
// may be scheduled.  A dependent grid is therefore only launched once all CTAs
// of the current grid are resident and past their wait, so a waiting grid can
// never hold the resources its predecessor needs to finish.
constexpr bool kProgrammaticLaunch = true;

__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dependents_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = kProgrammaticLaunch ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Host setup that must run once per device (kernel attributes): `setup`
// (returning cudaError_t, idempotent) runs unless it already succeeded on the
// calling thread's current device.  Threads racing on a first call may both run
// it; the per-device bit is published only after a success.
constexpr int kMaxDevices = 64;

inline int current_device_index()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return -1;  // not cached: the setup runs every time
    return dev;
}

template <typename F>
cudaError_t once_per_device(std::atomic<unsigned long long> &done, F &&setup)
{
    const int dev = current_device_index();
    const unsigned long long bit = dev >= 0 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit))
        return cudaSuccess;
    const cudaError_t e = setup();
    if (e == cudaSuccess && bit)
        done.fetch_or(bit, std::memory_order_release);
    return e;
}

// ------------------------------------------------------ launch parameters --

struct RopeAppendParams {
    int H, KV, d, rd;
    uint32_t flags;
    float eps;
    float rope_scale;
    int batch, capacity, total_tokens;
    const int32_t *cu_seqlens;
    const int32_t *cache_lens;
    const bf16 *q, *k, *v, *qw, *kw;
    bf16 *q_out, *cache_k, *cache_v;
    int32_t *status;
};

struct DecodeParams {
    int H, KV, group, batch, capacity;
    int cache_batch;           // sequences the cache holds (rows of the tensor maps)
    float scale_log2;          // score scale * log2(e)
    int head_chunks;           // group / heads-per-CTA
    int grid;                  // CTAs of the split pass, one key slice each
    int min_slice;             // fewest keys in a CTA's slice
    int max_pieces;            // streams + grid: bound on piece ids
    int max_kv_len;            // host bound on kv_lens (checked on the device)
    uint32_t flags;
    int window;                // > 0: only the last `window` keys are attended
    float cap_in, cap_out;     // soft-capping of log2-domain scores (cap_out 0: off)
    const bf16 *q, *cache_k, *cache_v, *gate;
    const int32_t *kv_lens;
    bf16 *out;
    float *probs;
    long long probs_stride;
    float *part_o;             // [max_pieces][heads-per-CTA][d]
    float *part_ml;            // [max_pieces][heads-per-CTA][2]  (max, sum) in the log2 domain
    int32_t *piece_span;       // [streams][2]  first and last piece id of each stream
    int32_t *status;
};

struct PrefillParams {
    int H, KV, group, batch, capacity;
    float scale_log2;
    int max_new_len;           // host bounds, checked on the device
    int max_total_len;
    int total_tokens;          // host copy of cu_seqlens[batch]
    float softcap;             // > 0: scores capped to softcap * tanh(s / softcap)
    int window;                // > 0: keys pos - window + 1 .. pos only
    int pack;                  // query heads of one kv group per tile (a power of two)
    int tile_tokens;           // tokens per tile: 128 / pack
    int q_tiles;               // ceil(max_new_len / tile_tokens)
    int HG;                    // head groups per sequence: H / pack
    int full_units;            // units (query tile, head group, sequence) run whole, one CTA each
    int tail_units;            // the units after them, each cut into num_splits key ranges
    int split_len;             // keys per piece of a cut unit (multiple of the key tile)
    int num_splits;            // pieces per cut unit (1: the tail units run whole too)
    int kv_read_once;          // every K/V tile is read by one CTA only (L2 evict-first loads)
    uint32_t flags;
    const int32_t *cu_seqlens, *cache_lens;
    const bf16 *q, *cache_k, *cache_v, *gate;
    bf16 *out;
    float *part_o;             // [tail_units][num_splits][128][d]: rows of the pieces
    float *part_ml;            // [tail_units][num_splits][128][2]: (max, sum), log2 domain
    int32_t *status;
};

struct ImportanceParams {
    int H, batch, max_kv_len;
    long long probs_stride, imp_stride;
    int accumulate;
    int vector_ok;             // 16-byte aligned rows: float4 loads and stores
    const float *probs;
    const int32_t *kv_lens;
    float *imp;
    int32_t *status;
};

// Kernel launchers (one translation unit each).
cudaError_t launch_rope_append(const RopeAppendParams &p, const double *inv_freq, int half,
                               cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams &p, int d, int heads_per_cta, cudaStream_t stream);
cudaError_t launch_importance(const ImportanceParams &p, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillParams &p, int d, int total_tokens, int cache_batch,
                           cudaStream_t stream);
size_t rope_append_smem_bytes(int H, int KV, int d, int rd);
int decode_key_tile();
int decode_ctas_per_sm();
int prefill_key_tile();
int prefill_q_tile();

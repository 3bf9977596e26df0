// importance.cu -- Born-rule importance of a decode step (cortiq-engine
// src/attention.rs, fn qwen_attention_core: every head's per-key
// probabilities are summed into `imp`, which the cache accumulates for
// importance-aware eviction; fn attend_all_heads returns the same sum).
//
//   imp[b][j] (+)= sum_h probs[b][h][j]      for j < kv_lens[b]
//
// HBM-bound: per key it reads 4 H bytes of probabilities and writes 4 bytes
// (reads 4 more when accumulating).  With 16-byte aligned rows (the usual
// case) a block covers `keys` keys of one sequence: one 2-D tensor-map copy
// brings the block's [H][keys] probabilities into shared memory (no registers
// held while the bytes are in flight: six 32 KB blocks per SM hold most of a
// call's reads in flight at once) and each thread then adds one key's H
// values in head order.  The grid runs sequence-fastest, so the blocks with
// keys (the low key ranges of every sequence) start first and the empty ones
// past the shorter sequences' ends come last.  Measured on 64 sequences of
// 512..8192 keys and 32 heads: as fast as the load path below when the rows
// are off 128-byte boundaries, 12% faster with a power-of-two row stride,
// where the load path's warps all start on the same DRAM offsets.
//
// Otherwise a block covers 256 keys of one sequence with four groups of 64
// threads; a thread owns four keys and one quarter of the heads, issuing all
// of its loads before adding them.  Each group adds its heads in index order
// and the four group sums are added in group order.  Either way the fp32 sum
// is the same on every run.
#include <cuda.h>
#include <mutex>

#include "na_internal.cuh"
#include "tc_primitives.cuh"

namespace {

// ------------------------------------------------------- tensor-map path --

constexpr size_t kTmaBlockBytes = 32u << 10;  // a block's [H][keys] fp32 tile

__global__ void importance_tma_kernel(const ImportanceParams p,
                                      const __grid_constant__ CUtensorMap map, int keys)
{
    extern __shared__ uint8_t smem_raw[];
    float *rows = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                            ~uintptr_t(127));  // [H][keys]
    __shared__ uint64_t full;
    const int b = blockIdx.x;
    const int kb = blockIdx.y * keys;
    if (threadIdx.x == 0) {
        tc::prefetch_tmap(&map);
        mbar_init(&full, 1);
        fence_barrier_init();
    }
    grid_dependency_wait();
    grid_dependents_launch();
    const int n = __ldg(p.kv_lens + b);
    const bool bad = n < 0 || n > p.max_kv_len;
    if (bad && blockIdx.y == 0 && threadIdx.x == 0)
        na_report(p.status, NA_ERR_CAPACITY);
    if (bad || kb >= n)
        return;  // the whole block: nothing was issued
    __syncthreads();  // the barrier's initialisation is visible to every waiting thread
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&full, (uint32_t)(p.H * keys * 4));
        tc::tma_load_2d(rows, &map, kb, b * p.H, &full);  // [H][keys], zeros past the stride
    }
    if (!mbar_wait_bounded(&full, 0)) {
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
        return;
    }
    const int t = threadIdx.x;
    if (kb + t < n) {
        float s = 0.f;
        for (int h = 0; h < p.H; h++)
            s += rows[h * keys + t];
        float *dst = p.imp + (size_t)b * p.imp_stride + kb + t;
        *dst = p.accumulate ? *dst + s : s;
    }
}

// ---------------------------------------------------------- load path --

constexpr int kImpThreads = 256;
constexpr int kHeadGroups = 4;
constexpr int kQuads = kImpThreads / kHeadGroups;  // key quads per block
constexpr int kKeysPerBlock = kQuads * 4;

__global__ void __launch_bounds__(kImpThreads) importance_kernel(const ImportanceParams p)
{
    __shared__ float4 part[kHeadGroups][kQuads];
    grid_dependency_wait();
    grid_dependents_launch();
    const int b = blockIdx.y;
    const int n = __ldg(p.kv_lens + b);
    if (n < 0 || n > p.max_kv_len) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            na_report(p.status, NA_ERR_CAPACITY);
        return;
    }
    const int kb = blockIdx.x * kKeysPerBlock;
    if (kb >= n)
        return;  // the whole block is past the sequence
    const int quad = threadIdx.x % kQuads, g = threadIdx.x / kQuads;
    const int hpg = (p.H + kHeadGroups - 1) / kHeadGroups;
    const int h0 = g * hpg, h1 = min(p.H, h0 + hpg);
    // This thread's four keys: with 16-byte rows, four consecutive keys (one
    // 16-byte load per head); otherwise keys quad, quad + 64, ... of the block
    // (a warp's loads of a head row are 32 consecutive floats).
    const bool vrows = p.vector_ok;
    const int j0 = vrows ? kb + 4 * quad : kb + quad;
    const int step = vrows ? 1 : kQuads;
    const bool vec = vrows && j0 + 4 <= n;
    const float *src = p.probs + (size_t)b * p.H * p.probs_stride + j0;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (vec) {
        int h = h0;
        for (; h + 8 <= h1; h += 8) {  // eight 16-byte loads in flight per thread
            float4 x[8];
#pragma unroll
            for (int u = 0; u < 8; u++)
                x[u] = __ldg(reinterpret_cast<const float4 *>(src + (size_t)(h + u) * p.probs_stride));
#pragma unroll
            for (int u = 0; u < 8; u++) {
                s.x += x[u].x;
                s.y += x[u].y;
                s.z += x[u].z;
                s.w += x[u].w;
            }
        }
        for (; h < h1; h++) {
            const float4 x = __ldg(reinterpret_cast<const float4 *>(src + (size_t)h * p.probs_stride));
            s.x += x.x;
            s.y += x.y;
            s.z += x.z;
            s.w += x.w;
        }
    } else {
        float t[4] = {0.f, 0.f, 0.f, 0.f};
        for (int h = h0; h < h1; h++) {
#pragma unroll
            for (int k = 0; k < 4; k++)
                if (j0 + k * step < n)
                    t[k] += __ldg(src + (size_t)h * p.probs_stride + k * step);
        }
        s = make_float4(t[0], t[1], t[2], t[3]);
    }
    part[g][quad] = s;
    __syncthreads();
    if (g != 0)
        return;
#pragma unroll
    for (int q = 1; q < kHeadGroups; q++) {
        const float4 o = part[q][quad];
        s = make_float4(s.x + o.x, s.y + o.y, s.z + o.z, s.w + o.w);
    }
    float *dst = p.imp + (size_t)b * p.imp_stride + j0;
    if (vec) {
        float4 *d4 = reinterpret_cast<float4 *>(dst);
        if (p.accumulate) {
            const float4 o = *d4;
            s = make_float4(o.x + s.x, o.y + s.y, o.z + s.z, o.w + s.w);
        }
        *d4 = s;
        return;
    }
    const float t[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int k = 0; k < 4; k++)
        if (j0 + k * step < n)
            dst[k * step] = p.accumulate ? dst[k * step] + t[k] : t[k];
}

}  // namespace

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Rows of fp32 probabilities, [batch * H][probs_stride], read in boxes of
// `keys` keys x `heads` rows, unswizzled (rows land back to back in shared
// memory); past the stride the box reads zeros.
bool make_probs_map(CUtensorMap *map, const ImportanceParams &p, int keys, int heads)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)p.probs_stride, (cuuint64_t)p.batch * p.H};
    const cuuint64_t strides[1] = {(cuuint64_t)p.probs_stride * 4};
    const cuuint32_t box[2] = {(cuuint32_t)keys, (cuuint32_t)heads};
    const cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(p.probs), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_importance(const ImportanceParams &p, cudaStream_t stream)
{
    if (p.batch <= 0 || p.max_kv_len <= 0)
        return cudaSuccess;
    // keys per block: 256 down to 32 so that a block's tile stays within 32 KB
    int keys = 256;
    while (keys > 32 && (size_t)p.H * keys * 4 > kTmaBlockBytes)
        keys >>= 1;
    const size_t smem = (size_t)p.H * keys * 4 + 128;  // + alignment slack
    const long long ky = (p.max_kv_len + keys - 1) / keys;
    CUtensorMap map;
    // one box of all H rows (box sides <= 256), within the default 48 KB
    if (p.vector_ok && p.H <= 256 && smem + 64 <= 48u * 1024 && ky <= 65535 &&
        (long long)p.batch * p.H < (1ll << 31) && make_probs_map(&map, p, keys, p.H))
        return launch_kernel(importance_tma_kernel, dim3(p.batch, (unsigned)ky), dim3(keys), smem,
                             stream, p, map, keys);
    const dim3 grid((p.max_kv_len + kKeysPerBlock - 1) / kKeysPerBlock, p.batch);
    return launch_kernel(importance_kernel, grid, dim3(kImpThreads), 0, stream, p);
}

// importance.cu -- Born-rule importance of a decode step (cortiq-engine
// src/attention.rs, fn qwen_attention_core: every head's per-key
// probabilities are summed into `imp`, which the cache accumulates for
// importance-aware eviction; fn attend_all_heads returns the same sum).
//
//   imp[b][j] (+)= sum_h probs[b][h][j]      for j < kv_lens[b]
//
// HBM-bound: per key it reads 4 H bytes of probabilities and writes 4 bytes
// (reads 4 more when accumulating).  Each thread owns four consecutive keys of
// one sequence and walks the heads in index order with 16-byte loads, eight in
// flight (the warp's loads of one head row are contiguous); the adds keep the
// head order, so the fp32 sum is the same on every run.
#include "na_internal.cuh"

namespace {

constexpr int kImpThreads = 256;
constexpr int kKeysPerThread = 4;

__global__ void __launch_bounds__(kImpThreads) importance_kernel(const ImportanceParams p)
{
    grid_dependency_wait();
    grid_dependents_launch();
    const int b = blockIdx.y;
    const int n = __ldg(p.kv_lens + b);
    if (n < 0 || n > p.max_kv_len) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            na_report(p.status, NA_ERR_CAPACITY);
        return;
    }
    const int j0 = (blockIdx.x * kImpThreads + threadIdx.x) * kKeysPerThread;
    if (j0 >= n)
        return;
    const float *src = p.probs + (size_t)b * p.H * p.probs_stride + j0;
    float *dst = p.imp + (size_t)b * p.imp_stride + j0;
    if (p.vector_ok && j0 + kKeysPerThread <= n) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        int h = 0;
        for (; h + 8 <= p.H; h += 8) {  // eight 16-byte loads in flight per thread
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
        for (; h < p.H; h++) {
            const float4 x = __ldg(reinterpret_cast<const float4 *>(src + (size_t)h * p.probs_stride));
            s.x += x.x;
            s.y += x.y;
            s.z += x.z;
            s.w += x.w;
        }
        float4 *d4 = reinterpret_cast<float4 *>(dst);
        if (p.accumulate) {
            const float4 o = *d4;
            s = make_float4(o.x + s.x, o.y + s.y, o.z + s.z, o.w + s.w);
        }
        *d4 = s;
        return;
    }
    const int m = min(kKeysPerThread, n - j0);
    for (int k = 0; k < m; k++) {
        float s = 0.f;
        for (int h = 0; h < p.H; h++)
            s += __ldg(src + (size_t)h * p.probs_stride + k);
        dst[k] = p.accumulate ? dst[k] + s : s;
    }
}

}  // namespace

cudaError_t launch_importance(const ImportanceParams &p, cudaStream_t stream)
{
    const int per_block = kImpThreads * kKeysPerThread;
    const dim3 grid((p.max_kv_len + per_block - 1) / per_block, p.batch);
    if (grid.x == 0)
        return cudaSuccess;
    return launch_kernel(importance_kernel, grid, dim3(kImpThreads), 0, stream, p);
}

// importance.cu -- Born-rule importance of a decode step (cortiq-engine
// src/attention.rs, fn qwen_attention_core: every head's per-key
// probabilities are summed into `imp`, which the cache accumulates for
// importance-aware eviction; fn attend_all_heads returns the same sum).
//
//   imp[b][j] (+)= sum_h probs[b][h][j]      for j < kv_lens[b]
//
// HBM-bound: per key it reads 4 H bytes of probabilities and writes 4 bytes
// (reads 4 more when accumulating).  A block covers 256 keys of one sequence
// with four groups of 64 threads; a thread owns four keys and one quarter of
// the heads, issuing all of its loads (eight 16-byte loads for 32 heads when
// the rows are 16-byte aligned) before adding them, so one wave of blocks
// keeps enough bytes in flight.  A warp's loads of one head row are
// contiguous.  Each group adds its heads in
// index order and the four group sums are added in group order, so the fp32
// sum is the same on every run.
#include "na_internal.cuh"

namespace {

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

cudaError_t launch_importance(const ImportanceParams &p, cudaStream_t stream)
{
    const dim3 grid((p.max_kv_len + kKeysPerBlock - 1) / kKeysPerBlock, p.batch);
    if (grid.x == 0 || grid.y == 0)
        return cudaSuccess;
    return launch_kernel(importance_kernel, grid, dim3(kImpThreads), 0, stream, p);
}

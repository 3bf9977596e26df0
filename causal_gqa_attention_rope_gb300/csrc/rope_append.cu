// rope_append.cu -- fused qk-RMSNorm, V-norm, RoPE and KV-cache append.
//
// Computes, per new token t of sequence b at pos = cache_lens[b] + (t - cu_seqlens[b]):
//   q_out[t][h]        = RoPE(norm_q(q[t][h]), pos)
//   cache_k[b][g][pos] = RoPE(norm_k(k[t][g]), pos)
//   cache_v[b][g][pos] = vnorm(v[t][g])
// following cortiq-engine src/attention.rs, fns finish_projection (norms before
// RoPE, partial rotary over the first rd dims), rmsnorm_head, vnorm_head and
// rope_rotate_scaled (half-split pairs (x[i], x[i + rd/2]), both outputs scaled
// by the attention factor).
//
// One CTA per token.  The token's H + 2 KV rows (a few KB, contiguous in q, k
// and v) are read with 16-byte loads, staged in shared memory as fp32, normed
// and rotated by one warp per row, and written back with 16-byte stores: q_out
// contiguously, K and V into their head-major cache slots.  The angle table is
// computed once per token and shared by all heads: the angle pos * inv_freq[i]
// is formed in double, reduced by whole turns in double (exact to ~1e-12 rad
// for positions up to 2^31 and frequencies <= 1), and only the reduced angle in
// [-pi, pi] goes through single-precision sincosf.  The kernel is bound by HBM
// traffic: 2 * (H + 2 KV) * d * 2 bytes per token.
#include "na_internal.cuh"

namespace {

struct RopeTable {
    double inv_freq[64];  // rd / 2 <= 64 (head_dim <= 128)
};

constexpr int kThreads = 256;
constexpr double kTwoPi = 6.283185307179586476925286766559;

__global__ void __launch_bounds__(kThreads) rope_append_kernel(const RopeAppendParams p,
                                                               const RopeTable tab)
{
    extern __shared__ float smem_f[];
    const int t = blockIdx.x;
    const int H = p.H, KV = p.KV, d = p.d, rows = H + 2 * KV;
    const int half = p.rd / 2;

    // Owner sequence: the last b with cu_seqlens[b] <= t (empty sequences skipped).
    int lo = 0, hi = p.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.cu_seqlens + mid) <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int b = lo;
    const int pos = __ldg(p.cache_lens + b) + (t - __ldg(p.cu_seqlens + b));
    if (pos < 0 || pos >= p.capacity) {
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_CAPACITY);
        return;
    }

    float *xs = smem_f;                                      // [rows][d]
    float2 *cs = reinterpret_cast<float2 *>(smem_f + rows * d);  // [half] (cos, sin) * scale

    for (int i = threadIdx.x; i < half; i += kThreads) {
        const double angle = (double)pos * tab.inv_freq[i];
        const double turns = rint(angle * (1.0 / kTwoPi));
        const float r = (float)fma(-turns, kTwoPi, angle);
        float s, c;
        sincosf(r, &s, &c);
        cs[i] = make_float2(c * p.rope_scale, s * p.rope_scale);
    }

    const int cpr = d / 8;  // 16-byte chunks per row
    for (int c = threadIdx.x; c < rows * cpr; c += kThreads) {
        const int r = c / cpr, j = c - r * cpr;
        const bf16 *src;
        if (r < H)
            src = p.q + ((size_t)t * H + r) * d;
        else if (r < H + KV)
            src = p.k + ((size_t)t * KV + (r - H)) * d;
        else
            src = p.v + ((size_t)t * KV + (r - H - KV)) * d;
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(src) + j);
        float f[8];
        bf16x8_to_f32(u, f);
        float4 *dst = reinterpret_cast<float4 *>(xs + r * d + j * 8);
        dst[0] = make_float4(f[0], f[1], f[2], f[3]);
        dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool qk_norm = (p.flags & NA_QK_NORM) != 0;
    const bool zero_centered = (p.flags & NA_QK_NORM_ZERO_CENTERED) != 0;
    const bool v_norm = (p.flags & NA_V_NORM) != 0;
    for (int r = warp; r < rows; r += kThreads / 32) {
        float *x = xs + r * d;
        const bool is_v = r >= H + KV;
        const bool normed = is_v ? v_norm : qk_norm;
        if (normed) {
            float ss = 0.f;
            for (int i = lane; i < d; i += 32)
                ss += x[i] * x[i];
#pragma unroll
            for (int o = 16; o; o >>= 1)
                ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float inv = 1.0f / sqrtf(ss / (float)d + p.eps);
            if (is_v) {
                for (int i = lane; i < d; i += 32)
                    x[i] *= inv;
            } else {
                const bf16 *w = r < H ? p.qw : p.kw;
                for (int i = lane; i < d; i += 32) {
                    float wi = __bfloat162float(w[i]);
                    if (zero_centered)
                        wi += 1.0f;
                    x[i] = x[i] * inv * wi;
                }
            }
            __syncwarp();
        }
        if (!is_v) {
            for (int i = lane; i < half; i += 32) {
                const float2 c = cs[i];
                const float x0 = x[i], x1 = x[i + half];
                x[i] = x0 * c.x - x1 * c.y;
                x[i + half] = x0 * c.y + x1 * c.x;
            }
        }
    }
    __syncthreads();

    const size_t cap = (size_t)p.capacity;
    for (int c = threadIdx.x; c < rows * cpr; c += kThreads) {
        const int r = c / cpr, j = c - r * cpr;
        bf16 *dst;
        if (r < H)
            dst = p.q_out + ((size_t)t * H + r) * d;
        else if (r < H + KV)
            dst = p.cache_k + (((size_t)b * KV + (r - H)) * cap + pos) * d;
        else
            dst = p.cache_v + (((size_t)b * KV + (r - H - KV)) * cap + pos) * d;
        reinterpret_cast<uint4 *>(dst)[j] = f32_to_bf16x8(xs + r * d + j * 8);
    }
}

}  // namespace

cudaError_t launch_rope_append(const RopeAppendParams &p, const double *inv_freq, int half,
                               cudaStream_t stream)
{
    RopeTable tab;
    for (int i = 0; i < 64; i++)
        tab.inv_freq[i] = i < half ? inv_freq[i] : 0.0;
    const size_t smem = ((size_t)(p.H + 2 * p.KV) * p.d + 2 * (size_t)half) * sizeof(float);
    static size_t configured = 0;
    if (smem > 48 * 1024 && smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(rope_append_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
        configured = smem;
    }
    rope_append_kernel<<<p.total_tokens, kThreads, smem, stream>>>(p, tab);
    return cudaGetLastError();
}

size_t rope_append_smem_bytes(int H, int KV, int d, int rd)
{
    return ((size_t)(H + 2 * KV) * d + 2 * (size_t)(rd / 2)) * sizeof(float);
}

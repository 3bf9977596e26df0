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
// contiguously, K and V into their head-major cache slots.  The kernel is bound
// by HBM traffic: 2 * (H + 2 KV) * d * 2 bytes per token.
//
// Precision.  The stored bf16 value is the correctly rounded result of the
// exact rotation in all but vanishing cases, also where x0 cos - x1 sin nearly
// cancels: the angle pos * inv_freq[i] is formed and reduced by whole turns in
// double, its cos and sin come from double sincos (once per token and pair
// index, shared by all heads) and are split into fp32 hi + lo parts; the
// rotation is evaluated with error-free fp32 products (fmaf residuals) and an
// error-free sum, so its absolute error is ~2^-44 of the operands.  The norm
// weight enters as the exact product x * w of two bf16 values (for the
// zero-centred style, x + x * w is kept as an fp32 hi + lo pair), and the row
// factors (1 / rms, and the attention factor on the rotated dims) are applied
// last as one relative rounding.
#include "na_internal.cuh"

namespace {

struct RopeTable {
    double inv_freq[64];  // rd / 2 <= 64 (head_dim <= 128)
};

constexpr int kThreads = 256;
constexpr double kTwoPi = 6.283185307179586476925286766559;

// a = x * w as an unevaluated fp32 sum hi + lo (exact).
struct F2 {
    float hi, lo;
};

__device__ __forceinline__ F2 weighted(float x, float w, bool zero_centered)
{
    const float p = x * w;
    const float pe = fmaf(x, w, -p);  // exact residual of the product
    if (!zero_centered)
        return {p, pe};
    // x * (1 + w) = x + x * w: error-free sum of x and p, residuals folded into lo
    const float s = x + p;
    const float bb = s - x;
    const float se = (x - (s - bb)) + (p - bb);
    return {s, se + pe};
}

// u * c + v * d with u, v as hi + lo pairs and c, d as hi + lo pairs, returned
// as hi + lo.  Leading products are exact (fmaf residuals); the leading sum is
// error-free; the cross terms are small and rounded once.
__device__ __forceinline__ F2 dot2(F2 u, float ch, float cl, F2 v, float dh, float dl)
{
    const float p0 = u.hi * ch;
    const float e0 = fmaf(u.hi, ch, -p0);
    const float p1 = v.hi * dh;
    const float e1 = fmaf(v.hi, dh, -p1);
    const float s = p0 + p1;
    const float bb = s - p0;
    const float t = (p0 - (s - bb)) + (p1 - bb);
    const float cross = fmaf(u.hi, cl, fmaf(u.lo, ch, fmaf(v.hi, dl, v.lo * dh)));
    return {s, t + (e0 + e1) + cross};
}

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

    float *xs = smem_f;                                          // [rows][d]
    float4 *cs = reinterpret_cast<float4 *>(smem_f + rows * d);  // [half] (cos hi, cos lo, sin hi, sin lo)

    for (int i = threadIdx.x; i < half; i += kThreads) {
        const double angle = (double)pos * tab.inv_freq[i];
        const double r = fma(-rint(angle * (1.0 / kTwoPi)), kTwoPi, angle);
        double sd, cd;
        sincos(r, &sd, &cd);
        const float ch = (float)cd, sh = (float)sd;
        cs[i] = make_float4(ch, (float)(cd - (double)ch), sh, (float)(sd - (double)sh));
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
        float f = 1.0f;  // row factor (1 / rms), applied last
        if (normed) {
            float ss = 0.f;  // squares of bf16 values are exact in fp32
            for (int i = lane; i < d; i += 32)
                ss = fmaf(x[i], x[i], ss);
#pragma unroll
            for (int o = 16; o; o >>= 1)
                ss += __shfl_xor_sync(0xffffffffu, ss, o);
            f = 1.0f / sqrtf(ss / (float)d + p.eps);
        }
        if (is_v) {
            for (int i = lane; i < d; i += 32)
                x[i] *= f;
            continue;
        }
        const bf16 *wp = normed ? (r < H ? p.qw : p.kw) : nullptr;
        auto a_of = [&](int i) -> F2 {
            if (!wp)
                return {x[i], 0.f};
            return weighted(x[i], __bfloat162float(wp[i]), zero_centered);
        };
        const float fr = f * p.rope_scale;  // the attention factor scales rotated dims only
        for (int i = lane; i < half; i += 32) {
            const float4 c = cs[i];
            const F2 a0 = a_of(i), a1 = a_of(i + half);
            const F2 neg_a1 = {-a1.hi, -a1.lo};
            const F2 y0 = dot2(a0, c.x, c.y, neg_a1, c.z, c.w);  // a0 cos - a1 sin
            const F2 y1 = dot2(a0, c.z, c.w, a1, c.x, c.y);      // a0 sin + a1 cos
            x[i] = fmaf(y0.hi, fr, y0.lo * fr);
            x[i + half] = fmaf(y1.hi, fr, y1.lo * fr);
        }
        for (int i = p.rd + lane; i < d; i += 32) {
            const F2 a = a_of(i);
            x[i] = fmaf(a.hi, f, a.lo * f);
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
    const size_t smem = rope_append_smem_bytes(p.H, p.KV, p.d, p.rd);
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
    return ((size_t)(H + 2 * KV) * d + 4 * (size_t)(rd / 2)) * sizeof(float);
}

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
// The kernel moves 2 * (H + 2 KV) * d * 2 bytes per token and is bound by the
// latency of its one round trip, so everything a thread needs is requested
// first, the work between the loads and the stores is short and free of double
// precision, and many small CTAs share an SM to overlap their round trips:
//   - rope_append_kernel (rotary_dim a multiple of 16): a CTA of 64 threads
//     takes 64 / (d / 16) rows of one token (grid: tokens x row groups); each
//     thread owns one 32-byte unit of a row -- chunks [8k, 8k + 8) and
//     [rd/2 + 8k, ...) of the rotated part (eight rotation pairs), two
//     consecutive chunks of the non-rotated tail, or of a V row -- loads it
//     with two 16-byte loads, takes the row's sum of squares with shuffles
//     among the row's lanes, rotates in registers and stores it with two
//     16-byte stores.  The only shared data are the cos/sin of the rd/2 pair
//     indices, computed by the CTA (one 256-entry table lookup each, read
//     through the cache).  One CTA per token of all rows left one CTA per SM
//     and measured ~39 us per 2048-token chunk of 56 rows.
//   - rope_append_staged_kernel (any even rotary_dim): the rows are staged in
//     shared memory and every thread works on independent (row, pair) slots.
//
// Precision.  Before its final rounding to bf16 a rotated value differs from
// the exact rotation by at most ~2^-23 of its own magnitude (plus ~2^-43 of
// its inputs), so the stored bf16 is the correctly rounded value unless the
// exact one lies that close to a bf16 rounding boundary; then it may be the
// neighbour, one ulp off (measured: about 7 in a million rotated values):
//   - The angle is taken in turns: pos * inv_freq / (2 pi) is formed exactly
//     modulo 1 in 64-bit fixed point (inv_freq / (2 pi) is passed as a 96-bit
//     fixed-point fraction, from a double-double division on the host; the
//     product needs only integer multiplies).  Its top 8 bits select cos and sin
//     of a multiple of 2 pi / 256 from a table built at compile time; the rest,
//     |r| <= pi / 256, goes through the Taylor series of cos and sin evaluated
//     in fp32 pairs (hi + lo, fmaf residuals for the leading products), and the
//     two are combined with the angle-sum formulas.  Absolute error of cos and
//     sin below 2^-43 (the rounding of the ~3e-7 low parts).
//   - The rotation keeps every rounding relative to its own result: one of the
//     two leading products is split exactly (its error recovered by an fmaf),
//     the other enters an fmaf unrounded (inputs carried as fp32 pairs use
//     error-free products and sums instead); the norm weight enters as the
//     exact product x * w of two bf16 values (for the zero-centred style,
//     x + x * w is kept as an fp32 hi + lo pair); the row factors (1 / rms,
//     and the attention factor on the rotated dims) are applied last as one
//     relative rounding.
#include "na_internal.cuh"

namespace {

// inv_freq[i] / (2 pi) in turns per position, as the 96-bit fixed-point
// fraction hi * 2^-64 + lo * 2^-96.
struct RopeTurns {
    unsigned long long hi[64];  // rd / 2 <= 64 (head_dim <= 128)
    unsigned int lo[64];
};

constexpr int kStagedThreads = 256;

// pi as an unevaluated sum of two doubles (the high part is pi rounded to
// double, the low part the next 53 bits).
constexpr double kPiHi = 3.141592653589793116;
constexpr double kPiLo = 1.2246467991473532e-16;
constexpr double kStep = kPiHi / 128.0;  // 2 pi / 256

// ------------------------------------------------- compile-time table --

// Taylor series about 0, used by the table builder for |x| <= pi / 4 where
// the terms fall below 1e-30 long before the loop ends.
constexpr double series_sin(double x)
{
    double term = x, sum = x;
    for (int n = 1; n < 20; ++n) {
        term *= -x * x / ((2.0 * n) * (2.0 * n + 1.0));
        sum += term;
    }
    return sum;
}

constexpr double series_cos(double x)
{
    double term = 1.0, sum = 1.0;
    for (int n = 1; n < 20; ++n) {
        term *= -x * x / ((2.0 * n - 1.0) * (2.0 * n));
        sum += term;
    }
    return sum;
}

struct alignas(16) TrigEntry {
    float ch, cl, sh, sl;  // cos and sin of 2 pi j / 256 as fp32 hi + lo pairs
};
struct TrigTable {
    TrigEntry e[256];
};

// cos and sin of 2 pi j / 256: the angle is written as a quarter turn q plus
// an offset within +-pi/4, whose series is evaluated; the quarter turn is
// applied by exact swaps and sign changes.
constexpr TrigTable make_trig_table()
{
    TrigTable t{};
    for (int j = 0; j < 256; ++j) {
        const int q = ((j + 32) / 64) % 4;
        const int off = j - 64 * ((j + 32) / 64);  // in [-32, 32)
        const double x = off * kStep;
        const double c0 = series_cos(x), s0 = series_sin(x);
        double c = c0, s = s0;
        if (q == 1) {
            c = -s0;
            s = c0;
        } else if (q == 2) {
            c = -c0;
            s = -s0;
        } else if (q == 3) {
            c = s0;
            s = -c0;
        }
        const float ch = (float)c, sh = (float)s;
        t.e[j] = TrigEntry{ch, (float)(c - (double)ch), sh, (float)(s - (double)sh)};
    }
    return t;
}

__device__ const TrigTable kTrig = make_trig_table();

// 2 pi as an fp32 pair.
constexpr float kTwoPiHi = (float)(2.0 * kPiHi);
constexpr float kTwoPiLo = (float)((2.0 * kPiHi - (double)kTwoPiHi) + 2.0 * kPiLo);

// ----------------------------------------------- fp32 pair arithmetic --

struct F2 {
    float hi, lo;  // unevaluated sum
};

// a * b + c * d of two pairs' products as a pair: leading products exact, their
// sum error-free, cross terms rounded once.
__host__ __device__ __forceinline__ F2 prod_sum(F2 a, F2 b, F2 c, F2 d)
{
    const float p0 = a.hi * b.hi;
    const float e0 = fmaf(a.hi, b.hi, -p0);
    const float p1 = c.hi * d.hi;
    const float e1 = fmaf(c.hi, d.hi, -p1);
    const float s = p0 + p1;
    const float bb = s - p0;
    const float t = (p0 - (s - bb)) + (p1 - bb);
    const float cross = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, fmaf(c.hi, d.lo, c.lo * d.hi)));
    return {s, t + (e0 + e1) + cross};
}

// cos and sin of 2 pi * pos * (fhi 2^-64 + flo 2^-96) as fp32 pairs
// (cos hi, cos lo, sin hi, sin lo).
__host__ __device__ __forceinline__ float4 cos_sin_turns(unsigned int pos, unsigned long long fhi,
                                                         unsigned int flo, const TrigEntry *tab)
{
    // Fraction of a turn in units of 2^-64 (exact but for the dropped bits
    // below 2^-64), rounded to the nearest 1/256 turn j plus a remainder.
    unsigned long long u = (unsigned long long)pos * fhi + (((unsigned long long)pos * flo) >> 32);
    u += 1ull << 55;
    const int j = (int)(u >> 56);
    const long long rem = (long long)(u & ((1ull << 56) - 1)) - (1ll << 55);  // |rem| <= 2^55
    // rem * 2^-64 as an fp32 pair: three exactly representable pieces.
    const int a_part = (int)(rem >> 32);  // |.| <= 2^23
    const unsigned int b_part = (unsigned int)(rem & 0xffffffffll);
    const float t1 = (float)a_part * 0x1p-32f;
    const float t2 = (float)(b_part >> 8) * 0x1p-56f;
    const float t3 = (float)(b_part & 255u) * 0x1p-64f;
    const float rh0 = t1 + t2;
    const float bb = rh0 - t1;
    const float rl0 = ((t1 - (rh0 - bb)) + (t2 - bb)) + t3;
    // r = 2 pi * remainder, radians, |r| <= pi / 256
    const float dh = rh0 * kTwoPiHi;
    const float dl = fmaf(rh0, kTwoPiHi, -dh) + fmaf(rh0, kTwoPiLo, rl0 * kTwoPiHi);

    // Series of the remainder.
    const float z = dh * dh;
    const float ze = fmaf(dh, dh, -z);
    // sin r = dh - dh^3/6 + dh^5/120 + dl (1 - dh^2/2)
    const float p3 = dh * z;
    const float p3e = fmaf(dh, z, -p3) + dh * ze;
    const float sin_lo = dl * fmaf(z, -0.5f, 1.0f) - (p3 * (1.0f / 6.0f) + p3e * (1.0f / 6.0f)) +
                         p3 * z * (1.0f / 120.0f);
    const F2 sn = {dh, sin_lo};
    // cos r = 1 - r^2/2 + r^4/24 - r^6/720, with r^2 = z + ze + 2 dh dl
    const float half_z = 0.5f * z;
    const float c0 = 1.0f - half_z;
    const float c0e = (1.0f - c0) - half_z;
    const float z2 = z * z;
    const float cos_lo = c0e - 0.5f * ze - dh * dl + z2 * (1.0f / 24.0f) - z2 * z * (1.0f / 720.0f);
    const F2 cs = {c0, cos_lo};

    const TrigEntry e = tab[j];
    const F2 tc = {e.ch, e.cl}, ts = {e.sh, e.sl};
    const F2 nts = {-e.sh, -e.sl};
    const F2 c = prod_sum(tc, cs, nts, sn);  // cos(t + r) = cos t cos r - sin t sin r
    const F2 s = prod_sum(ts, cs, tc, sn);   // sin(t + r) = sin t cos r + cos t sin r
    return make_float4(c.hi, c.lo, s.hi, s.lo);
}

// a = x * w as an unevaluated fp32 sum hi + lo (exact).
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

// Rotated pair (y0, y1) = (a0 cos - a1 sin, a0 sin + a1 cos) * fr.
__device__ __forceinline__ void rotate(F2 a0, F2 a1, float4 c, float fr, float &y0, float &y1)
{
    const F2 r0 = prod_sum(a0, F2{c.x, c.y}, F2{-a1.hi, -a1.lo}, F2{c.z, c.w});
    const F2 r1 = prod_sum(a0, F2{c.z, c.w}, a1, F2{c.x, c.y});
    y0 = fmaf(r0.hi, fr, r0.lo * fr);
    y1 = fmaf(r1.hi, fr, r1.lo * fr);
}

// The same for exact inputs (no low parts).  Of the two leading products one
// is split exactly -- t = a1 sin_hi rounded, e its error from an fma -- and
// the other enters an fma unrounded, so h = a0 cos_hi - t carries a single
// rounding relative to itself; e and the low parts of cos and sin are added
// once.  Before the final rounding to bf16 the result is within ~2^-23 of
// itself (plus ~2^-48 of the inputs).
__device__ __forceinline__ void rotate_exact(float a0, float a1, float4 c, float fr, float &y0,
                                             float &y1)
{
    {
        const float t = a1 * c.z;
        const float e = fmaf(a1, c.z, -t);
        const float h = fmaf(a0, c.x, -t);
        const float lo = fmaf(a0, c.y, -a1 * c.w) - e;
        y0 = fmaf(h, fr, lo * fr);
    }
    {
        const float t = a1 * c.x;
        const float e = fmaf(a1, c.x, -t);
        const float h = fmaf(a0, c.z, t);
        const float lo = fmaf(a0, c.w, a1 * c.y) + e;
        y1 = fmaf(h, fr, lo * fr);
    }
}

__device__ __forceinline__ const bf16 *row_src(const RopeAppendParams &p, int t, int r)
{
    if (r < p.H)
        return p.q + ((size_t)t * p.H + r) * p.d;
    if (r < p.H + p.KV)
        return p.k + ((size_t)t * p.KV + (r - p.H)) * p.d;
    return p.v + ((size_t)t * p.KV + (r - p.H - p.KV)) * p.d;
}

__device__ __forceinline__ bf16 *row_dst(const RopeAppendParams &p, int t, int r, int b, int slot)
{
    const size_t cap = (size_t)p.capacity;
    if (r < p.H)
        return p.q_out + ((size_t)t * p.H + r) * p.d;
    if (r < p.H + p.KV)
        return p.cache_k + (((size_t)b * p.KV + (r - p.H)) * cap + slot) * p.d;
    return p.cache_v + (((size_t)b * p.KV + (r - p.H - p.KV)) * cap + slot) * p.d;
}

// Owner sequence b of token t (the last b with cu_seqlens[b] <= t, empty
// sequences skipped) and the token's position, a warp at a time: cu_seqlens
// and cache_lens are read in the same round.
__device__ __forceinline__ void owner_of(const RopeAppendParams &p, int t, int lane, int &b,
                                         int &pos)
{
    b = 0;
    pos = -1;
    for (int base = 0; base < p.batch; base += 32) {
        const int i = base + lane;
        int cu = 0x7fffffff, cl = 0;
        if (i < p.batch) {
            cu = __ldg(p.cu_seqlens + i);
            cl = __ldg(p.cache_lens + i);
        }
        const unsigned m = __ballot_sync(0xffffffffu, cu <= t);
        if (m) {
            const int src = 31 - __clz(m);
            b = base + src;
            pos = __shfl_sync(0xffffffffu, cl, src) + (t - __shfl_sync(0xffffffffu, cu, src));
        }
        if (m != 0xffffffffu)
            break;
    }
}

// 16-byte read-only load kept where it is written (the compiler may not sink
// it past the barriers that follow, so its latency overlaps theirs).
__device__ __forceinline__ uint4 ldg_early(const void *p)
{
    uint4 u;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                 : "l"(p));
    return u;
}

// ------------------------------------------------------ register path --

constexpr int kAppendThreads = 64;  // one 32-byte row unit each: 4 rows of d = 128, 8 of d = 64

template <int D>
__global__ void __launch_bounds__(kAppendThreads) rope_append_kernel(const RopeAppendParams p,
                                                                const RopeTurns turns)
{
    constexpr int UPR = D / 16;  // 32-byte units per row
    __shared__ float4 cs[64];
    const int t = blockIdx.x;
    const int H = p.H, KV = p.KV, rows = H + 2 * KV;
    const int row0 = blockIdx.y * (kAppendThreads / UPR);  // the CTA's first row
    const int half = p.rd / 2;
    const int lane = threadIdx.x & 31;
    const bool qk_norm = (p.flags & NA_QK_NORM) != 0;
    const bool zero_centered = (p.flags & NA_QK_NORM_ZERO_CENTERED) != 0;
    const bool v_norm = (p.flags & NA_V_NORM) != 0;

    // This thread's unit: row r, 8-element chunks starting at e0 and e1.
    const int unit = threadIdx.x;
    const int r = row0 + unit / UPR, k = unit % UPR;
    const bool active = r < rows;
    const bool is_v = r >= H + KV;
    const bool rot = !is_v && k < p.rd / 16;
    int e0, e1;
    if (is_v) {
        e0 = 16 * k;
        e1 = e0 + 8;
    } else if (rot) {
        e0 = 8 * k;
        e1 = half + 8 * k;
    } else {
        e0 = p.rd + 16 * (k - p.rd / 16);
        e1 = e0 + 8;
    }

    // Kernel parameters go before the wait: this thread's frequency (a
    // dynamically indexed parameter).
    unsigned long long fhi = 0;
    unsigned int flo = 0;
    if ((int)threadIdx.x < half) {
        fhi = turns.hi[threadIdx.x];
        flo = turns.lo[threadIdx.x];
    }
    grid_dependency_wait();
    grid_dependents_launch();

    // Everything the token needs is requested first.
    uint4 xa = make_uint4(0, 0, 0, 0), xb = xa, wa = xa, wb = xa;
    if (active) {
        const uint4 *src = reinterpret_cast<const uint4 *>(row_src(p, t, r));
        xa = ldg_early(src + e0 / 8);
        xb = ldg_early(src + e1 / 8);
        if (qk_norm && !is_v) {
            const uint4 *w = reinterpret_cast<const uint4 *>(r < H ? p.qw : p.kw);
            wa = ldg_early(w + e0 / 8);
            wb = ldg_early(w + e1 / 8);
        }
    }
    int b, pos;
    owner_of(p, t, lane, b, pos);
    const bool ring = (p.flags & NA_RING_CACHE) != 0;  // slot = pos % capacity
    if (pos < 0 || (!ring && pos >= p.capacity)) {
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_CAPACITY);
        return;
    }
    const int slot = ring ? pos % p.capacity : pos;
    __syncthreads();
    if ((int)threadIdx.x < half)  // stored [i][k] for pair 8k + i: a row's lanes read adjacent entries
        cs[(threadIdx.x & 7) * 8 + (threadIdx.x >> 3)] = cos_sin_turns((unsigned)pos, fhi, flo, kTrig.e);
    __syncthreads();

    float a[8], c[8];
    bf16x8_to_f32(xa, a);
    bf16x8_to_f32(xb, c);
    const bool normed = is_v ? v_norm : qk_norm;
    float f = 1.0f;
    if (qk_norm || v_norm) {  // every lane shuffles; rows are aligned to UPR lanes
        float ss = 0.f;      // squares of bf16 values are exact in fp32
#pragma unroll
        for (int i = 0; i < 8; i++)
            ss = fmaf(a[i], a[i], fmaf(c[i], c[i], ss));
#pragma unroll
        for (int o = UPR / 2; o; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (normed)
            f = 1.0f / sqrtf(ss / (float)D + p.eps);
    }
    if (!active)
        return;

    float ya[8], yb[8];
    if (is_v) {
#pragma unroll
        for (int i = 0; i < 8; i++) {
            ya[i] = a[i] * f;
            yb[i] = c[i] * f;
        }
    } else {
        F2 xa2[8], xb2[8];
        if (qk_norm) {
            float wfa[8], wfb[8];
            bf16x8_to_f32(wa, wfa);
            bf16x8_to_f32(wb, wfb);
#pragma unroll
            for (int i = 0; i < 8; i++) {
                xa2[i] = weighted(a[i], wfa[i], zero_centered);
                xb2[i] = weighted(c[i], wfb[i], zero_centered);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                xa2[i] = F2{a[i], 0.f};
                xb2[i] = F2{c[i], 0.f};
            }
        }
        if (rot) {
            const float fr = f * p.rope_scale;  // the attention factor scales rotated dims only
            if (qk_norm && zero_centered) {
#pragma unroll
                for (int i = 0; i < 8; i++)
                    rotate(xa2[i], xb2[i], cs[i * 8 + k], fr, ya[i], yb[i]);
            } else if (qk_norm) {
                // x * w of two bf16 values is exact in fp32 (its low part is 0):
                // the exact-input rotation gives the same value with fewer terms
#pragma unroll
                for (int i = 0; i < 8; i++)
                    rotate_exact(xa2[i].hi, xb2[i].hi, cs[i * 8 + k], fr, ya[i], yb[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; i++)
                    rotate_exact(a[i], c[i], cs[i * 8 + k], fr, ya[i], yb[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                ya[i] = fmaf(xa2[i].hi, f, xa2[i].lo * f);
                yb[i] = fmaf(xb2[i].hi, f, xb2[i].lo * f);
            }
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(row_dst(p, t, r, b, slot));
    dst[e0 / 8] = f32_to_bf16x8(ya);
    dst[e1 / 8] = f32_to_bf16x8(yb);
}

// -------------------------------------------------------- staged path --

__global__ void __launch_bounds__(kStagedThreads) rope_append_staged_kernel(const RopeAppendParams p,
                                                                           const RopeTurns turns)
{
    extern __shared__ float smem_f[];
    const int t = blockIdx.x;
    const int H = p.H, KV = p.KV, d = p.d, rows = H + 2 * KV;
    const int half = p.rd / 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool qk_norm = (p.flags & NA_QK_NORM) != 0;
    const bool zero_centered = (p.flags & NA_QK_NORM_ZERO_CENTERED) != 0;
    const bool v_norm = (p.flags & NA_V_NORM) != 0;

    float *xs = smem_f;                                          // [rows][d]
    float4 *cs = reinterpret_cast<float4 *>(xs + rows * d);      // [64] (cos hi, lo, sin hi, lo)
    TrigEntry *trig = reinterpret_cast<TrigEntry *>(cs + 64);    // [256]
    float *wq = reinterpret_cast<float *>(trig + 256);           // [d] q norm weights
    float *wk = wq + d;                                          // [d] k norm weights
    float *rf = wk + d;                                          // [rows] 1 / rms per row

    const int cpr = d / 8;  // 16-byte chunks per row
    const int chunks = rows * cpr;
    for (int i = threadIdx.x; i < 256; i += kStagedThreads)
        reinterpret_cast<uint4 *>(trig)[i] = __ldg(reinterpret_cast<const uint4 *>(&kTrig) + i);
    grid_dependency_wait();
    grid_dependents_launch();
    int b, pos;
    owner_of(p, t, lane, b, pos);
    const bool ring = (p.flags & NA_RING_CACHE) != 0;  // slot = pos % capacity
    if (pos < 0 || (!ring && pos >= p.capacity)) {
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_CAPACITY);
        return;
    }
    const int slot = ring ? pos % p.capacity : pos;
    if (qk_norm) {
        for (int i = threadIdx.x; i < 2 * d; i += kStagedThreads)
            wq[i] = __bfloat162float(i < d ? p.qw[i] : p.kw[i - d]);
    }
    for (int c = threadIdx.x; c < chunks; c += kStagedThreads) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(row_src(p, t, c / cpr)) + (c % cpr));
        float f[8];
        bf16x8_to_f32(u, f);
        float4 *dst = reinterpret_cast<float4 *>(xs + c * 8);
        dst[0] = make_float4(f[0], f[1], f[2], f[3]);
        dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    __syncthreads();

    // cos/sin per pair index (two warps) while the other warps take row norms.
    if (threadIdx.x < 64) {
        if ((int)threadIdx.x < half)
            cs[threadIdx.x] = cos_sin_turns((unsigned)pos, turns.hi[threadIdx.x],
                                            turns.lo[threadIdx.x], trig);
    } else if (qk_norm || v_norm) {
        for (int r = warp - 2; r < rows; r += kStagedThreads / 32 - 2) {
            const bool is_v = r >= H + KV;
            float f = 1.0f;
            if (is_v ? v_norm : qk_norm) {
                const float *x = xs + r * d;
                float ss = 0.f;
                for (int i = lane; i < d; i += 32)
                    ss = fmaf(x[i], x[i], ss);
#pragma unroll
                for (int o = 16; o; o >>= 1)
                    ss += __shfl_xor_sync(0xffffffffu, ss, o);
                f = 1.0f / sqrtf(ss / (float)d + p.eps);
            }
            if (lane == 0)
                rf[r] = f;
        }
    }
    __syncthreads();

    // Every row has d/2 slots.  Q and K rows: slot i < half is the pair
    // (i, i + half), the rest cover the non-rotated tail two elements at a
    // time; V rows: elements (2i, 2i + 1).
    const int slots = d / 2;
    const int items = rows * slots;
    const bool any_norm = qk_norm || v_norm;
    for (int it = threadIdx.x; it < items; it += kStagedThreads) {
        const int r = it / slots, i = it - r * slots;
        float *x = xs + r * d;
        const float f = any_norm ? rf[r] : 1.0f;
        if (r >= H + KV) {
            if (v_norm) {
                x[2 * i] *= f;
                x[2 * i + 1] *= f;
            }
            continue;
        }
        const float *w = qk_norm ? (r < H ? wq : wk) : nullptr;
        auto a_of = [&](int e) -> F2 {
            if (!w)
                return {x[e], 0.f};
            return weighted(x[e], w[e], zero_centered);
        };
        if (i < half) {
            float y0, y1;
            rotate(a_of(i), a_of(i + half), cs[i], f * p.rope_scale, y0, y1);
            x[i] = y0;
            x[i + half] = y1;
        } else {
            const int e0 = p.rd + 2 * (i - half);
            const F2 a0 = a_of(e0), a1 = a_of(e0 + 1);
            x[e0] = fmaf(a0.hi, f, a0.lo * f);
            x[e0 + 1] = fmaf(a1.hi, f, a1.lo * f);
        }
    }
    __syncthreads();

    for (int c = threadIdx.x; c < chunks; c += kStagedThreads) {
        const int r = c / cpr, j = c - r * cpr;
        reinterpret_cast<uint4 *>(row_dst(p, t, r, b, slot))[j] = f32_to_bf16x8(xs + r * d + j * 8);
    }
}

// inv_freq / (2 pi) as a 96-bit fixed-point fraction.  The quotient is formed
// as a double-double (error ~2^-104 relative), then each part is converted to
// fixed point exactly.
void turns_fixed_point(double inv_freq, unsigned long long &hi, unsigned int &lo)
{
    const double bh = 2.0 * kPiHi, bl = 2.0 * kPiLo;
    const double q1 = inv_freq / bh;
    const double p = q1 * bh;
    const double pe = fma(q1, bh, -p);
    const double rsd = ((inv_freq - p) - pe) - q1 * bl;
    const double q2 = rsd / bh;
    const __int128 x = (__int128)ldexp(q1, 96) + (__int128)nearbyint(ldexp(q2, 96));
    hi = (unsigned long long)(x >> 32);
    lo = (unsigned int)(x & 0xffffffff);
}

}  // namespace

cudaError_t launch_rope_append(const RopeAppendParams &p, const double *inv_freq, int half,
                               cudaStream_t stream)
{
    RopeTurns turns{};
    for (int i = 0; i < half && i < 64; i++)
        turns_fixed_point(inv_freq[i], turns.hi[i], turns.lo[i]);
    if (p.rd % 16 == 0) {
        const int rows_per_cta = kAppendThreads / (p.d / 16);
        const dim3 grid(p.total_tokens, (p.H + 2 * p.KV + rows_per_cta - 1) / rows_per_cta);
        if (p.d == 128)
            return launch_kernel(rope_append_kernel<128>, grid, dim3(kAppendThreads), 0, stream, p,
                                 turns);
        return launch_kernel(rope_append_kernel<64>, grid, dim3(kAppendThreads), 0, stream, p, turns);
    }
    const size_t smem = rope_append_smem_bytes(p.H, p.KV, p.d, p.rd);
    // the largest dynamic shared memory granted so far, per device
    static std::atomic<size_t> configured[kMaxDevices];
    const int dev = current_device_index();
    if (smem > 48 * 1024 && (dev < 0 || smem > configured[dev].load(std::memory_order_acquire))) {
        cudaError_t e = cudaFuncSetAttribute(rope_append_staged_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0) {
            size_t cur = configured[dev].load(std::memory_order_relaxed);
            while (cur < smem && !configured[dev].compare_exchange_weak(cur, smem))
                ;
        }
    }
    return launch_kernel(rope_append_staged_kernel, dim3(p.total_tokens), dim3(kStagedThreads), smem,
                         stream, p, turns);
}

size_t rope_append_smem_bytes(int H, int KV, int d, int rd)
{
    (void)rd;
    const size_t rows = (size_t)(H + 2 * KV);
    return (rows * d + 64 * 4 + 256 * 4 + 2 * (size_t)d + rows) * sizeof(float);
}

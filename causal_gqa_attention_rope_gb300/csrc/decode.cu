// decode.cu -- single-token GQA decode over the KV cache, split over keys,
// with per-key probabilities (cortiq-engine src/attention.rs, fn
// attention_head: softmax(q.k / sqrt(d)) . V and the returned probabilities;
// fn attend_all_heads: each KV group's keys and values are streamed once for
// all of its query heads).
//
// Split pass (persistent, one CTA per SM).  A work unit is (split, sequence,
// kv head, head chunk): up to `split_len` consecutive keys of one KV head, for
// HPC query heads of its group.  One producer lane streams the unit's key and
// value tiles (DEC_TILE keys, contiguous in the head-major cache) into a
// DEC_STAGES-deep shared-memory ring with 1-D bulk async copies completing on
// mbarriers; eight consumer warps score and accumulate.  Scores never touch
// tensor cores: per key the group does 2 * HPC * d flops over 4 d bytes, far
// below the SIMT rate, so the pass is bound by HBM bandwidth.
//
// Consumer lane layout: a warp takes 2 keys per step (key group kg = lane / 16);
// the 16 lanes of a key group split head_dim into slices of d/16 elements.
// Each lane forms HPC partial dot products with packed fp32x2 FMAs, and a
// 4-level butterfly leaves the full score of (key kg, head (lane%16) / (16/HPC))
// in that lane.  The running maximum is only raised when a tile's maximum
// exceeds it by more than 2^8 (factor 256), so the accumulator rescale runs a
// handful of times per split instead of per tile; scores are carried in the
// log2 domain (q pre-scaled by scale * log2 e).  Two CTAs share an SM (about
// 112 KB of shared memory and <= 112 registers per thread each).
//
// Raw log2-domain scores are written to the probability buffer; the combine
// pass turns them into probabilities once the global maximum and sum are known,
// and merges the splits' partial outputs (flash-decoding style) with the gate.
#include "na_internal.cuh"

namespace {

constexpr int DEC_TILE = 64;
constexpr int DEC_STAGES = 3;
constexpr int DEC_CWARPS = 8;
constexpr int DEC_THREADS = (DEC_CWARPS + 1) * 32;
constexpr int LPK = 16;                    // lanes per key
constexpr int KPS = 32 / LPK;              // keys per warp step
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int HPC>
struct DecSmem {
    bf16 k[DEC_STAGES][DEC_TILE * D];
    bf16 v[DEC_STAGES][DEC_TILE * D];
    float merge_o[DEC_CWARPS][HPC][D];
    float merge_m[DEC_CWARPS][HPC];
    float merge_l[DEC_CWARPS][HPC];
    uint64_t full[DEC_STAGES];
    uint64_t empty[DEC_STAGES];
    int abort_flag;
};

struct Unit {
    int split, b, kvh, hc;
};

__device__ __forceinline__ Unit unit_of(int u, const DecodeParams &p)
{
    Unit r;
    r.hc = u % p.head_chunks;
    u /= p.head_chunks;
    r.kvh = u % p.KV;
    u /= p.KV;
    r.b = u % p.batch;
    r.split = u / p.batch;
    return r;
}

// Key range [s0, s1) of a unit; empty when s0 >= s1.  Lengths past the cache
// capacity or the host bound are skipped here and reported by the combine pass.
__device__ __forceinline__ void unit_keys(const Unit &w, const DecodeParams &p, int &s0, int &s1)
{
    const int n = __ldg(p.kv_lens + w.b);
    s0 = w.split * p.split_len;
    s1 = min(n, s0 + p.split_len);
    if (n < 0 || n > p.capacity || n > p.max_kv_len)
        s1 = s0;
}

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// N 32-bit words (2N bf16) from a 16-byte (N = 4) or 8-byte (N = 2) aligned address.
template <int N>
__device__ __forceinline__ void load_words(const bf16 *src, uint32_t (&w)[N])
{
    if constexpr (N == 4) {
        const uint4 u = *reinterpret_cast<const uint4 *>(src);
        w[0] = u.x;
        w[1] = u.y;
        w[2] = u.z;
        w[3] = u.w;
    } else {
        static_assert(N == 2, "2 or 4 words");
        const uint2 u = *reinterpret_cast<const uint2 *>(src);
        w[0] = u.x;
        w[1] = u.y;
    }
}

template <int D, int HPC>
__global__ void __launch_bounds__(DEC_THREADS, 2) decode_split_kernel(const DecodeParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    DecSmem<D, HPC> &sm = *reinterpret_cast<DecSmem<D, HPC> *>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < DEC_STAGES; s++) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], DEC_CWARPS);
        }
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const size_t cap = (size_t)p.capacity;

    if (warp == DEC_CWARPS) {
        // ---------------------------------------------------------- producer --
        if (lane != 0)
            return;
        const uint64_t policy = l2_policy_evict_first();
        uint32_t it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
            const Unit w = unit_of(u, p);
            int s0, s1;
            unit_keys(w, p, s0, s1);
            const size_t head_base = ((size_t)w.b * p.KV + w.kvh) * cap * D;
            for (int j0 = s0; j0 < s1; j0 += DEC_TILE, it++) {
                const int stage = it % DEC_STAGES;
                const uint32_t parity = ((it / DEC_STAGES) & 1) ^ 1;
                if (!mbar_wait_bounded(&sm.empty[stage], parity) ||
                    *(volatile int *)&sm.abort_flag) {
                    na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
                    *(volatile int *)&sm.abort_flag = 1;
                    ok = false;
                    break;
                }
                const int n = min(DEC_TILE, s1 - j0);
                const uint32_t bytes = (uint32_t)(n * D * (int)sizeof(bf16));
                mbar_arrive_expect_tx(&sm.full[stage], 2 * bytes);
                bulk_copy_g2s(sm.k[stage], p.cache_k + head_base + (size_t)j0 * D, bytes,
                              &sm.full[stage], policy);
                bulk_copy_g2s(sm.v[stage], p.cache_v + head_base + (size_t)j0 * D, bytes,
                              &sm.full[stage], policy);
            }
        }
        // Let every copy this lane issued land before the CTA can exit.
        for (int s = 0; s < DEC_STAGES; s++) {
            if ((int)it - 1 - s < 0)
                break;
            const uint32_t last = it - 1 - s;
            mbar_wait_bounded(&sm.full[last % DEC_STAGES], (last / DEC_STAGES) & 1);
        }
        return;
    }

    // ------------------------------------------------------------ consumers --
    constexpr int EPL = D / LPK;   // head_dim elements per lane
    constexpr int R = LPK / HPC;   // lanes holding the same (key, head) score
    constexpr int KPW = DEC_TILE / DEC_CWARPS;  // keys per warp per tile
    constexpr int STEPS = KPW / KPS;
    const int kg = lane / LPK, sub = lane % LPK;
    const int hsel = sub / R;      // head whose score this lane ends up holding
    const unsigned FULL = 0xffffffffu;
    uint32_t it = 0;
    // A warp whose wait timed out keeps walking the units so that every warp
    // joins the same named barriers, but does no more waits or writes.
    bool aborted = false;

    for (int u = blockIdx.x; u < p.total_units; u += gridDim.x) {
        const Unit w = unit_of(u, p);
        int s0, s1;
        unit_keys(w, p, s0, s1);
        if (s0 >= s1)
            continue;
        if (*(volatile int *)&sm.abort_flag)
            aborted = true;
        const int head0 = w.kvh * p.group + w.hc * HPC;

        float2 q[HPC][EPL / 2];
#pragma unroll
        for (int h = 0; h < HPC; h++) {
            uint32_t wd[EPL / 2];
            load_words<EPL / 2>(p.q + ((size_t)w.b * p.H + head0 + h) * D + sub * EPL, wd);
#pragma unroll
            for (int e = 0; e < EPL / 2; e++) {
                const float2 f = bf16x2_to_f2(wd[e]);
                q[h][e] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
            }
        }
        float2 acc[HPC][EPL / 2];
        float m_ref[HPC];
#pragma unroll
        for (int h = 0; h < HPC; h++) {
            m_ref[h] = -INFINITY;
#pragma unroll
            for (int e = 0; e < EPL / 2; e++)
                acc[h][e] = make_float2(0.f, 0.f);
        }
        float l_lane = 0.f;
        float *probs_row = p.probs ? p.probs + ((size_t)w.b * p.H + head0 + hsel) * p.probs_stride
                                   : nullptr;

        for (int j0 = s0; j0 < s1 && !aborted; j0 += DEC_TILE, it++) {
            const int stage = it % DEC_STAGES;
            if (!mbar_wait_bounded(&sm.full[stage], (it / DEC_STAGES) & 1)) {
                if (lane == 0) {
                    na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
                    *(volatile int *)&sm.abort_flag = 1;
                }
                aborted = true;
                break;
            }
            const bf16 *kt = sm.k[stage];
            const bf16 *vt = sm.v[stage];
            const bool full_tile = j0 + DEC_TILE <= s1;
            float s[STEPS];
#pragma unroll
            for (int st = 0; st < STEPS; st++) {
                const int kl = warp * KPW + st * KPS + kg;  // key within the tile
                float2 part2[HPC];
#pragma unroll
                for (int h = 0; h < HPC; h++)
                    part2[h] = make_float2(0.f, 0.f);
                uint32_t wd[EPL / 2];
                load_words<EPL / 2>(kt + kl * D + sub * EPL, wd);
#pragma unroll
                for (int e = 0; e < EPL / 2; e++) {
                    const float2 kf = bf16x2_to_f2(wd[e]);
#pragma unroll
                    for (int h = 0; h < HPC; h++)
                        part2[h] = __ffma2_rn(q[h][e], kf, part2[h]);
                }
                float part[HPC];
#pragma unroll
                for (int h = 0; h < HPC; h++)
                    part[h] = part2[h].x + part2[h].y;
                // Butterfly over the LPK lanes of the key group: halve the head
                // set at each level while it has more than one head.
                int cnt = HPC;
#pragma unroll
                for (int m = LPK / 2; m >= 1; m >>= 1) {
                    if (cnt > 1) {
                        const bool up = (sub & m) != 0;
                        const int half = cnt / 2;
#pragma unroll
                        for (int i = 0; i < HPC / 2; i++) {
                            if (i < half) {
                                const float keep = up ? part[half + i] : part[i];
                                const float send = up ? part[i] : part[half + i];
                                part[i] = keep + __shfl_xor_sync(FULL, send, m);
                            }
                        }
                        cnt = half;
                    } else {
                        part[0] += __shfl_xor_sync(FULL, part[0], m);
                    }
                }
                const int j = j0 + kl;
                s[st] = (full_tile || j < s1) ? part[0] : -INFINITY;
                if (probs_row && (full_tile || j < s1) && (sub % R) == 0)
                    probs_row[j] = part[0];
            }
            // Tile maximum per head, then (rarely) raise the reference maximum.
            float tmax = s[0];
#pragma unroll
            for (int st = 1; st < STEPS; st++)
                tmax = fmaxf(tmax, s[st]);
#pragma unroll
            for (int m = LPK; m < 32; m <<= 1)
                tmax = fmaxf(tmax, __shfl_xor_sync(FULL, tmax, m));
            float hmax[HPC];
            bool raise = false;
#pragma unroll
            for (int h = 0; h < HPC; h++) {
                hmax[h] = __shfl_sync(FULL, tmax, h * R);
                raise |= hmax[h] > m_ref[h] + kRescaleThreshold;
            }
            if (raise) {  // warp-uniform
#pragma unroll
                for (int h = 0; h < HPC; h++) {
                    const float m_new = fmaxf(m_ref[h], hmax[h]);
                    const float alpha = (m_ref[h] == -INFINITY) ? 0.f : exp2f(m_ref[h] - m_new);
                    m_ref[h] = m_new;
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int e = 0; e < EPL / 2; e++)
                        acc[h][e] = __fmul2_rn(acc[h][e], a2);
                    if (h == hsel)
                        l_lane *= alpha;
                }
            }
            float m_mine = m_ref[0];
#pragma unroll
            for (int h = 1; h < HPC; h++)
                if (h == hsel)
                    m_mine = m_ref[h];
#pragma unroll
            for (int st = 0; st < STEPS; st++) {
                const float pr = (s[st] == -INFINITY) ? 0.f : exp2f(s[st] - m_mine);
                l_lane += pr;
                const int kl = warp * KPW + st * KPS + kg;
                const bool valid = full_tile || (j0 + kl) < s1;
                float2 pv[HPC];
#pragma unroll
                for (int h = 0; h < HPC; h++) {
                    const float x = __shfl_sync(FULL, pr, kg * LPK + h * R);
                    pv[h] = make_float2(x, x);
                }
                uint32_t wd[EPL / 2];
                load_words<EPL / 2>(vt + kl * D + sub * EPL, wd);
#pragma unroll
                for (int e = 0; e < EPL / 2; e++) {
                    float2 vf = bf16x2_to_f2(wd[e]);
                    if (!valid)  // stale shared memory past the last key
                        vf = make_float2(0.f, 0.f);
#pragma unroll
                    for (int h = 0; h < HPC; h++)
                        acc[h][e] = __ffma2_rn(pv[h], vf, acc[h][e]);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.empty[stage]);
        }

        // Merge the key groups of the warp, then the warps of the CTA.
#pragma unroll
        for (int m = LPK; m < 32; m <<= 1) {
#pragma unroll
            for (int h = 0; h < HPC; h++)
#pragma unroll
                for (int e = 0; e < EPL / 2; e++) {
                    acc[h][e].x += __shfl_xor_sync(FULL, acc[h][e].x, m);
                    acc[h][e].y += __shfl_xor_sync(FULL, acc[h][e].y, m);
                }
            l_lane += __shfl_xor_sync(FULL, l_lane, m);
        }
        if (kg == 0) {
#pragma unroll
            for (int h = 0; h < HPC; h++)
#pragma unroll
                for (int e = 0; e < EPL / 2; e++)
                    *reinterpret_cast<float2 *>(&sm.merge_o[warp][h][sub * EPL + 2 * e]) = acc[h][e];
            if ((sub % R) == 0) {
                float m_mine = m_ref[0];
#pragma unroll
                for (int h = 1; h < HPC; h++)
                    if (h == hsel)
                        m_mine = m_ref[h];
                sm.merge_m[warp][hsel] = m_mine;
                sm.merge_l[warp][hsel] = l_lane;
            }
        }
        named_barrier_sync(1, DEC_CWARPS * 32);
        for (int idx = threadIdx.x; idx < HPC * D; idx += DEC_CWARPS * 32) {
            const int h = idx / D, e = idx - h * D;
            float M = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < DEC_CWARPS; ww++)
                M = fmaxf(M, sm.merge_m[ww][h]);
            float o = 0.f, l = 0.f;
#pragma unroll
            for (int ww = 0; ww < DEC_CWARPS; ww++) {
                const float mw = sm.merge_m[ww][h];
                if (mw != -INFINITY) {
                    const float f = exp2f(mw - M);
                    o += sm.merge_o[ww][h][e] * f;
                    l += sm.merge_l[ww][h] * f;
                }
            }
            if (aborted)
                continue;
            const size_t row = ((size_t)w.b * p.H + head0 + h) * p.max_splits + w.split;
            p.part_o[row * D + e] = o;
            if (e == 0) {
                p.part_ml[row * 2] = M;
                p.part_ml[row * 2 + 1] = l;
            }
        }
        named_barrier_sync(1, DEC_CWARPS * 32);
    }
}

// Combine pass: one CTA per (sequence, query head).
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p)
{
    const int bh = blockIdx.x;
    const int b = bh / p.H;
    const int n = __ldg(p.kv_lens + b);
    bf16 *out = p.out + (size_t)bh * D;
    if (n < 0 || n > p.capacity || n > p.max_kv_len) {
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_CAPACITY);
        for (int e = threadIdx.x; e < D; e += blockDim.x)
            out[e] = __float2bfloat16_rn(0.f);
        return;
    }
    if (n == 0) {
        for (int e = threadIdx.x; e < D; e += blockDim.x)
            out[e] = __float2bfloat16_rn(0.f);
        return;
    }
    const int ns = (n + p.split_len - 1) / p.split_len;
    const float *ml = p.part_ml + (size_t)bh * p.max_splits * 2;
    float M = -INFINITY;
    for (int s = 0; s < ns; s++)
        M = fmaxf(M, ml[2 * s]);
    float L = 0.f;
    for (int s = 0; s < ns; s++)
        L += ml[2 * s + 1] * exp2f(ml[2 * s] - M);
    const float inv_l = 1.0f / L;
    const float *po = p.part_o + (size_t)bh * p.max_splits * D;
    for (int e = threadIdx.x; e < D; e += blockDim.x) {
        float o = 0.f;
        for (int s = 0; s < ns; s++)
            o += po[(size_t)s * D + e] * exp2f(ml[2 * s] - M);
        o *= inv_l;
        if ((p.flags & NA_OUT_GATE) && p.gate) {
            const float g = __bfloat162float(p.gate[(size_t)bh * D + e]);
            o *= 1.0f / (1.0f + __expf(-g));
        }
        out[e] = __float2bfloat16_rn(o);
    }
    if (p.probs) {
        float *pr = p.probs + (size_t)bh * p.probs_stride;
        if ((p.probs_stride & 3) == 0) {
            const int n4 = n >> 2;
            float4 *pr4 = reinterpret_cast<float4 *>(pr);
            for (int i = threadIdx.x; i < n4; i += blockDim.x) {
                float4 x = pr4[i];
                x.x = exp2f(x.x - M) * inv_l;
                x.y = exp2f(x.y - M) * inv_l;
                x.z = exp2f(x.z - M) * inv_l;
                x.w = exp2f(x.w - M) * inv_l;
                pr4[i] = x;
            }
            for (int j = (n4 << 2) + threadIdx.x; j < n; j += blockDim.x)
                pr[j] = exp2f(pr[j] - M) * inv_l;
        } else {
            for (int j = threadIdx.x; j < n; j += blockDim.x)
                pr[j] = exp2f(pr[j] - M) * inv_l;
        }
    }
}

template <int D, int HPC>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t stream)
{
    const size_t smem = sizeof(DecSmem<D, HPC>);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, HPC>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_split_kernel<D, HPC>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = p.total_units < 2 * sms ? p.total_units : 2 * sms;  // two CTAs per SM
    if (grid > 0)
        decode_split_kernel<D, HPC><<<grid, DEC_THREADS, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    decode_combine_kernel<D><<<p.batch * p.H, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

int decode_key_tile() { return DEC_TILE; }

cudaError_t launch_decode(const DecodeParams &p, int d, int heads_per_cta, cudaStream_t stream)
{
    if (d == 128) {
        if (heads_per_cta == 4)
            return launch_decode_t<128, 4>(p, stream);
        if (heads_per_cta == 2)
            return launch_decode_t<128, 2>(p, stream);
        return launch_decode_t<128, 1>(p, stream);
    }
    if (heads_per_cta == 4)
        return launch_decode_t<64, 4>(p, stream);
    if (heads_per_cta == 2)
        return launch_decode_t<64, 2>(p, stream);
    return launch_decode_t<64, 1>(p, stream);
}

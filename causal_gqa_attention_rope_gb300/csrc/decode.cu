// decode.cu -- single-token GQA decode over the KV cache, split over keys,
// with per-key probabilities (cortiq-engine src/attention.rs, fn
// attention_head: softmax(q.k / sqrt(d)) . V and the returned probabilities;
// fn attend_all_heads: each KV group's keys and values are streamed once for
// all of its query heads).
//
// Split pass (persistent, two CTAs per SM).  The keys to read form S streams,
// one per (sequence, kv head, head chunk) -- a head chunk being the HPC query
// heads of a KV group that one CTA scores together -- laid end to end in
// sequence-major order.  CTA c takes the contiguous slice [c P, (c + 1) P) of
// that concatenation, P = max(ceil(total / grid), min_slice): every CTA reads
// the same number of keys whatever the mix of sequence lengths, so none idles
// while others finish long sequences.  A slice cuts streams into pieces; the
// piece of stream s in CTA c gets the id s + c, unique and consecutive along a
// stream, and its partial output lands in workspace row id.  The CTA holding a
// stream's first (last) key records that piece id for the combine pass.
//
// In each CTA one producer lane streams the piece's key and value tiles
// (DEC_TILE keys, contiguous in the head-major cache) into a DEC_STAGES-deep
// shared-memory ring with 1-D bulk async copies completing on mbarriers;
// seven consumer warps score and accumulate.  Scores never touch tensor cores:
// per key the group does 2 * HPC * d flops over 4 d bytes, far below the SIMT
// rate, so the pass is bound by HBM bandwidth.
//
// Consumer lane layout: a warp takes 2 keys per step (key group kg = lane / 16);
// the 16 lanes of a key group split head_dim into slices of d/16 elements.
// Each lane forms HPC partial dot products with packed fp32x2 FMAs, and a
// 4-level butterfly leaves the full score of (key kg, head (lane%16) / (16/HPC))
// in that lane.  The running maximum is only raised when a tile's maximum
// exceeds it by more than 2^8 (factor 256), so the accumulator rescale runs a
// handful of times per split instead of per tile; scores are carried in the
// log2 domain (q pre-scaled by scale * log2 e).  Two CTAs share an SM (about
// 100 KB of shared memory each).  Eight warps per CTA keep four warps per SM
// sub-partition, so each thread may hold 128 registers: the d = 128, four-head
// instance needs 127 and spilled to local memory under the 96-register cap
// that nine-warp CTAs impose (measured 22% slower).
//
// Raw log2-domain scores are written to the probability buffer; the combine
// pass turns them into probabilities once the global maximum and sum are known,
// and merges the splits' partial outputs (flash-decoding style) with the gate.
#include "na_internal.cuh"

namespace {

constexpr int DEC_TILE = 56;  // DEC_CWARPS warps x 8 keys
constexpr int DEC_STAGES = 3;
constexpr int DEC_CWARPS = 7;
constexpr int DEC_THREADS = (DEC_CWARPS + 1) * 32;
constexpr int LPK = 16;                    // lanes per key
constexpr int KPS = 32 / LPK;              // keys per warp step
constexpr float kRescaleThreshold = 8.0f;  // log2 units


// Keys of sequence b that are attended -- the last `window` of its length, or
// all of them without a window -- with *first the index of the first one; 0
// for a length past the cache capacity or the host bound (skipped here,
// reported by the combine pass).
__device__ __forceinline__ int attended_keys(const DecodeParams &p, int b, int &first)
{
    const int n = __ldg(p.kv_lens + b);
    const bool ring = (p.flags & NA_RING_CACHE) != 0;  // positions wrap at the capacity
    if (n < 0 || (!ring && n > p.capacity) || n > p.max_kv_len) {
        first = 0;
        return 0;
    }
    const int len = (p.window > 0 && n > p.window) ? p.window : n;
    first = n - len;
    return len;
}

__device__ __forceinline__ int valid_len(const DecodeParams &p, int b)
{
    int first;
    return attended_keys(p, b, first);
}

// Where this CTA's key slice starts: computed by one full warp, then shared.
struct Slice {
    long long start, end;  // [start, end) in the concatenation of all streams
    long long off;         // offset of the stream holding `start`
    int b, si;             // its sequence and stream index within the sequence
    int empty;
};

template <int D, int HPC>
struct DecSmem {
    bf16 k[DEC_STAGES][DEC_TILE * D];
    bf16 v[DEC_STAGES][DEC_TILE * D];
    float merge_o[DEC_CWARPS][HPC][D];
    float merge_m[DEC_CWARPS][HPC];
    float merge_l[DEC_CWARPS][HPC];
    uint64_t full[DEC_STAGES];
    uint64_t empty[DEC_STAGES];
    Slice slice;
    int abort_flag;
};

// One piece: the keys [k0, k1) of stream (b, kvh, hc) that this CTA reads.
struct Piece {
    int b, kvh, hc, k0, k1, id;
    int kf;            // cache index of the stream's first attended key
    bool first, last;  // holds the stream's first / last key
};

__device__ __forceinline__ void locate_slice(const DecodeParams &p, int lane, Slice &out)
{
    const unsigned FULL = 0xffffffffu;
    const int spb = p.KV * p.head_chunks;  // streams per sequence
    long long t = 0;
    for (int b = lane; b < p.batch; b += 32)
        t += valid_len(p, b);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        t += __shfl_xor_sync(FULL, t, m);
    const long long total = t * spb;
    const long long grid = gridDim.x;
    long long P = (total + grid - 1) / grid;
    if (P < p.min_slice)
        P = p.min_slice;
    Slice sl{};
    sl.start = (long long)blockIdx.x * P;
    sl.end = min(sl.start + P, total);
    sl.empty = sl.start >= total;
    if (!sl.empty) {
        // First sequence whose streams extend past `start`.
        long long base = 0;
        for (int b0 = 0; b0 < p.batch; b0 += 32) {
            const int b = b0 + lane;
            const int n = b < p.batch ? valid_len(p, b) : 0;
            const long long w = (long long)n * spb;
            long long incl = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long y = __shfl_up_sync(FULL, incl, o);
                if (lane >= o)
                    incl += y;
            }
            const long long excl = base + incl - w;
            const unsigned hit = __ballot_sync(FULL, w > 0 && sl.start < excl + w && sl.start >= excl);
            if (hit) {
                const int src = __ffs(hit) - 1;
                sl.b = b0 + src;
                const long long off_b = __shfl_sync(FULL, excl, src);
                const int nb = __shfl_sync(FULL, n, src);
                sl.si = (int)((sl.start - off_b) / nb);
                sl.off = off_b + (long long)sl.si * nb;
                break;
            }
            base += __shfl_sync(FULL, incl, 31);
        }
    }
    if (lane == 0)
        out = sl;
}

// Walks this CTA's pieces in order; every thread of the CTA walks the same way.
struct Walker {
    long long start, end, off;
    int b, si, len, kfirst, spb, c;
    bool done;

    __device__ __forceinline__ void init(const Slice &sl, const DecodeParams &p)
    {
        start = sl.start;
        end = sl.end;
        off = sl.off;
        b = sl.b;
        si = sl.si;
        spb = p.KV * p.head_chunks;
        c = blockIdx.x;
        done = sl.empty != 0;
        kfirst = 0;
        len = done ? 0 : attended_keys(p, b, kfirst);
    }

    __device__ __forceinline__ bool next(const DecodeParams &p, Piece &pc)
    {
        while (!done && b < p.batch && off < end) {
            const long long s_off = off;
            const int n = len, sb = b, ssi = si, kfs = kfirst;
            off += n;
            if (++si == spb) {
                si = 0;
                if (++b < p.batch)
                    len = attended_keys(p, b, kfirst);
            }
            const long long lo = start > s_off ? start - s_off : 0;
            const long long hi = end - s_off < n ? end - s_off : n;
            if (lo < hi) {
                pc.b = sb;
                pc.kvh = ssi / p.head_chunks;
                pc.hc = ssi - pc.kvh * p.head_chunks;
                pc.k0 = (int)lo;
                pc.k1 = (int)hi;
                pc.id = sb * spb + ssi + c;
                pc.kf = kfs;
                pc.first = lo == 0;
                pc.last = hi == n;
                return true;
            }
        }
        return false;
    }
};

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

template <int D, int HPC, bool CAPPED>
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
    grid_dependency_wait();
    grid_dependents_launch();
    if (warp == DEC_CWARPS)
        locate_slice(p, lane, sm.slice);
    __syncthreads();
    Walker walk;
    walk.init(sm.slice, p);
    Piece pc;

    const size_t cap = (size_t)p.capacity;

    if (warp == DEC_CWARPS) {
        // ---------------------------------------------------------- producer --
        if (lane != 0)
            return;
        const uint64_t policy = l2_policy_evict_first();
        uint32_t it = 0;
        bool ok = true;
        while (ok && walk.next(p, pc)) {
            const int s0 = pc.k0, s1 = pc.k1;
            const size_t head_base = ((size_t)pc.b * p.KV + pc.kvh) * cap * D;
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
                // Slot of the tile's first key; with a ring a tile that reaches the
                // end of the slab continues at slot 0 (two copies, same stage).
                int slot = pc.kf + j0;
                int n1 = n;
                if (p.flags & NA_RING_CACHE) {
                    slot %= p.capacity;
                    n1 = min(n, p.capacity - slot);
                }
                const uint32_t b1 = (uint32_t)(n1 * D * (int)sizeof(bf16));
                bulk_copy_g2s(sm.k[stage], p.cache_k + head_base + (size_t)slot * D, b1,
                              &sm.full[stage], policy);
                bulk_copy_g2s(sm.v[stage], p.cache_v + head_base + (size_t)slot * D, b1,
                              &sm.full[stage], policy);
                if (n1 < n) {
                    bulk_copy_g2s(sm.k[stage] + (size_t)n1 * D, p.cache_k + head_base, bytes - b1,
                                  &sm.full[stage], policy);
                    bulk_copy_g2s(sm.v[stage] + (size_t)n1 * D, p.cache_v + head_base, bytes - b1,
                                  &sm.full[stage], policy);
                }
            }
        }
        // Let every copy this lane issued land before the CTA can exit.
        for (int s = 0; s < DEC_STAGES; s++) {
            if ((int)it - 1 - s < 0)
                break;
            const uint32_t last = it - 1 - s;
            if (!mbar_wait_bounded(&sm.full[last % DEC_STAGES], (last / DEC_STAGES) & 1))
                na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
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
    // A warp whose wait timed out keeps walking the pieces so that every warp
    // joins the same named barriers, but does no more waits or writes.
    bool aborted = false;

    while (walk.next(p, pc)) {
        const int s0 = pc.k0, s1 = pc.k1;
        if (*(volatile int *)&sm.abort_flag)
            aborted = true;
        const int head0 = pc.kvh * p.group + pc.hc * HPC;

        float2 q[HPC][EPL / 2];
#pragma unroll
        for (int h = 0; h < HPC; h++) {
            uint32_t wd[EPL / 2];
            load_words<EPL / 2>(p.q + ((size_t)pc.b * p.H + head0 + h) * D + sub * EPL, wd);
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
        float *probs_row = p.probs ? p.probs + ((size_t)pc.b * p.H + head0 + hsel) * p.probs_stride
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
                float sc = part[0];
                if constexpr (CAPPED) {  // c tanh(s / c) in the log2 domain, tanh(y) = 1 - 2 / (e^2y + 1)
                    const float e = exp2f(sc * p.cap_in);
                    sc = p.cap_out * (1.0f - __fdividef(2.0f, e + 1.0f));
                }
                s[st] = (full_tile || j < s1) ? sc : -INFINITY;
                if (probs_row && (full_tile || j < s1) && (sub % R) == 0)
                    probs_row[pc.kf + j] = sc;
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
        // Every consumer warp has finished this piece's tiles (or given up): the
        // abort flag is final for the piece.  A piece of a CTA whose wait gave up
        // is written as the marker (max -inf, sum -1), which the merge passes
        // report instead of merging, so no call ever merges another call's rows.
        const bool bad = *(volatile int *)&sm.abort_flag != 0;
        for (int idx = threadIdx.x; idx < HPC * D; idx += DEC_CWARPS * 32) {
            const int h = idx / D, e = idx - h * D;
            if (bad) {
                if (e == 0) {
                    const size_t row = (size_t)pc.id * HPC + h;
                    p.part_ml[row * 2] = -INFINITY;
                    p.part_ml[row * 2 + 1] = -1.0f;
                }
                continue;
            }
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
            const size_t row = (size_t)pc.id * HPC + h;
            p.part_o[row * D + e] = o;
            if (e == 0) {
                p.part_ml[row * 2] = M;
                p.part_ml[row * 2 + 1] = l;
            }
        }
        if (threadIdx.x == 0) {  // the span follows from the slicing alone: always written
            const int stream = pc.id - blockIdx.x;
            if (pc.first)
                p.piece_span[2 * stream] = pc.id;
            if (pc.last)
                p.piece_span[2 * stream + 1] = pc.id;
        }
        named_barrier_sync(1, DEC_CWARPS * 32);
    }
}

// Row maximum M and 1/L of a head over its stream's ns pieces, from the
// log2-domain (max, sum) pairs at ml[2 hpc s], ml[2 hpc s + 1].  Every lane of
// the calling warp gets the same values: lanes take pieces lane, lane + 32, ...
// and reduce with butterflies (a fixed order: the same result on every run and
// in both merge passes).  Returns false, on every lane, when a piece carries
// the marker of a split-pass CTA whose wait gave up (a negative sum).
__device__ __forceinline__ bool merge_weights_from(float m0, float l0, const float *ml, int hpc,
                                                   int ns, int lane, float &M, float &inv_l)
{
    const unsigned FULL = 0xffffffffu;
    bool bad = lane < ns && l0 < 0.f;
    M = m0;
    for (int s = lane + 32; s < ns; s += 32)
        M = fmaxf(M, ml[2 * hpc * s]);
#pragma unroll
    for (int o = 16; o; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
    float L = m0 == -INFINITY ? 0.f : l0 * exp2f(m0 - M);
    for (int s = lane + 32; s < ns; s += 32) {
        const float m = ml[2 * hpc * s], l = ml[2 * hpc * s + 1];
        bad |= l < 0.f;
        if (m != -INFINITY)
            L += l * exp2f(m - M);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
        L += __shfl_xor_sync(FULL, L, o);
    inv_l = L > 0.f ? 1.0f / L : 0.f;
    return !__any_sync(FULL, bad);
}

// The lane's own piece (lane < ns), loaded: (max, sum), or (-inf, 0).
__device__ __forceinline__ void merge_lane_piece(const float *ml, int hpc, int ns, int lane,
                                                 float &m0, float &l0)
{
    m0 = -INFINITY;
    l0 = 0.f;
    if (lane < ns) {
        m0 = ml[2 * hpc * lane];
        l0 = ml[2 * hpc * lane + 1];
    }
}

__device__ __forceinline__ bool merge_weights(const float *ml, int hpc, int ns, int lane, float &M,
                                              float &inv_l)
{
    float m0, l0;
    merge_lane_piece(ml, hpc, ns, lane, m0, l0);
    return merge_weights_from(m0, l0, ml, hpc, ns, lane, M, inv_l);
}

// Element e of a head's merged output: the pieces' partial rows weighted by
// 2^(m_s - M), summed in piece order, times 1/L; then the optional gate.
template <int D>
__device__ __forceinline__ float merge_out_elem(const float *po, const float *ml, int hpc, int ns,
                                                int e, float M, float inv_l)
{
    float o = 0.f;
    int s = 0;
    for (; s + 4 <= ns; s += 4) {  // four pieces' loads in flight; adds stay in piece order
        float m[4], x[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            m[u] = ml[2 * hpc * (s + u)];
            x[u] = po[(size_t)(s + u) * hpc * D + e];
        }
#pragma unroll
        for (int u = 0; u < 4; u++)
            if (m[u] != -INFINITY)
                o += x[u] * exp2f(m[u] - M);
    }
    for (; s < ns; s++) {
        const float m = ml[2 * hpc * s];
        if (m != -INFINITY)
            o += po[(size_t)s * hpc * D + e] * exp2f(m - M);
    }
    return o * inv_l;
}

__device__ __forceinline__ float gated_elem(float o, bf16 g)
{
    return o * (1.0f / (1.0f + __expf(-__bfloat162float(g))));
}

// Probability of key j from its raw log2-domain score (0 before the window).
__device__ __forceinline__ float prob_of(float raw, int j, int kf, float M, float inv_l)
{
    return j < kf ? 0.f : exp2f(raw - M) * inv_l;
}

// Combine pass: one CTA per (sequence, query head).
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeParams p)
{
    grid_dependency_wait();
    grid_dependents_launch();
    const int bh = blockIdx.x;
    const int b = bh / p.H;
    const int n = __ldg(p.kv_lens + b);
    bf16 *out = p.out + (size_t)bh * D;
    if (n < 0 || (!(p.flags & NA_RING_CACHE) && n > p.capacity) || n > p.max_kv_len) {
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
    // Pieces of this head's stream: ids first..last, HPC heads per row group.
    const int h = bh - b * p.H;
    const int hpc = p.group / p.head_chunks;
    const int kvh = h / p.group, r = h - kvh * p.group;
    const int stream = (b * p.KV + kvh) * p.head_chunks + r / hpc;
    const int first = p.piece_span[2 * stream], last = p.piece_span[2 * stream + 1];
    if (first < 0 || last < first || last >= p.max_pieces) {  // the split pass gave up
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
        for (int e = threadIdx.x; e < D; e += blockDim.x)
            out[e] = __float2bfloat16_rn(0.f);
        return;
    }
    const int ns = last - first + 1;
    const size_t row0 = (size_t)first * hpc + (r % hpc);
    const float *ml = p.part_ml + row0 * 2;

    // The first batch of this row's raw scores is requested before the merge
    // arithmetic, so its latency overlaps the pieces' loads.
    constexpr int PV = 8;  // 16-byte loads in flight per thread
    constexpr int NT = 256;
    // The row is walked as a scalar head up to its first 16-byte boundary,
    // 16-byte groups of four keys, and a scalar tail (any stride).
    float *pr = p.probs ? p.probs + (size_t)bh * p.probs_stride : nullptr;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(pr);
    const int pre = (addr & 3) ? n : min(n, (int)(((16 - (addr & 15)) & 15) >> 2));
    const int n4 = pr ? (n - pre) >> 2 : 0;
    float4 *pr4 = reinterpret_cast<float4 *>(pr + pre);
    float4 x[PV];
#pragma unroll
    for (int u = 0; u < PV; u++) {
        const int i = threadIdx.x + u * NT;
        if (i < n4)
            x[u] = pr4[i];
    }

    // Row maximum and sum over the pieces: every warp reduces them.
    const int lane = threadIdx.x & 31;
    float M, inv_l;
    if (!merge_weights(ml, hpc, ns, lane, M, inv_l)) {  // a split-pass wait gave up
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
        for (int e = threadIdx.x; e < D; e += NT)
            out[e] = __float2bfloat16_rn(0.f);
        return;
    }

    const float *po = p.part_o + row0 * D;
    for (int e = threadIdx.x; e < D; e += NT) {
        float o = merge_out_elem<D>(po, ml, hpc, ns, e, M, inv_l);
        if ((p.flags & NA_OUT_GATE) && p.gate)
            o = gated_elem(o, p.gate[(size_t)bh * D + e]);
        out[e] = __float2bfloat16_rn(o);
    }
    if (pr) {
        // keys before the window (none without one) get probability 0
        const int kf = (p.window > 0 && n > p.window) ? n - p.window : 0;
        auto prob = [&](float raw, int j) { return prob_of(raw, j, kf, M, inv_l); };
        for (int base = 0; base < n4; base += PV * NT) {
            if (base > 0) {
#pragma unroll
                for (int u = 0; u < PV; u++) {
                    const int i = base + threadIdx.x + u * NT;
                    if (i < n4)
                        x[u] = pr4[i];
                }
            }
#pragma unroll
            for (int u = 0; u < PV; u++) {
                const int i = base + threadIdx.x + u * NT;
                if (i < n4) {
                    const int j = pre + 4 * i;
                    float4 y = x[u];
                    y.x = prob(y.x, j);
                    y.y = prob(y.y, j + 1);
                    y.z = prob(y.z, j + 2);
                    y.w = prob(y.w, j + 3);
                    pr4[i] = y;
                }
            }
        }
        for (int j = threadIdx.x; j < pre; j += NT)
            pr[j] = prob(pr[j], j);
        for (int j = pre + (n4 << 2) + threadIdx.x; j < n; j += NT)
            pr[j] = prob(pr[j], j);
    }
}

template <int D, int HPC, bool CAPPED>
cudaError_t launch_split(const DecodeParams &p, cudaStream_t stream)
{
    const size_t smem = sizeof(DecSmem<D, HPC>);
    static std::atomic<unsigned long long> configured{0};
    const cudaError_t e = once_per_device(configured, [smem] {
        cudaError_t r = cudaFuncSetAttribute(decode_split_kernel<D, HPC, CAPPED>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(decode_split_kernel<D, HPC, CAPPED>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        return r;
    });
    if (e != cudaSuccess)
        return e;
    return launch_kernel(decode_split_kernel<D, HPC, CAPPED>, dim3(p.grid), dim3(DEC_THREADS), smem,
                         stream, p);
}

template <int D, int HPC>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t stream)
{
    cudaError_t e = p.cap_out > 0.f ? launch_split<D, HPC, true>(p, stream)
                                    : launch_split<D, HPC, false>(p, stream);
    if (e != cudaSuccess)
        return e;
    return launch_kernel(decode_combine_kernel<D>, dim3(p.batch * p.H), dim3(256), 0, stream, p);
}

}  // namespace

int decode_key_tile() { return DEC_TILE; }

int decode_ctas_per_sm() { return 2; }

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

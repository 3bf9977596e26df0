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
// In each CTA a producer warp streams the piece's key and value rows
// (DEC_TILE keys per tile, one 1-D bulk async copy per row into rows padded by
// 16 bytes) into a DEC_STAGES-deep shared-memory ring completing on mbarriers;
// four consumer warps take 16 keys of each tile.  Scores and the P.V product
// run on warp-level bf16 MMAs (m16n8k16, fp32 accumulation) with the HPC <= 8
// query heads of the chunk as the n8 dimension: the heads beyond HPC are
// padding, which the tensor pipe absorbs many times over, and the pass is
// left to stream HBM.  (With the scores on fp32 FMAs and a butterfly over
// lanes, the arithmetic took ~10% of the pass.)  The running maximum is only
// raised when a tile's maximum exceeds it by more than 2^8 (factor 256), so the
// accumulator rescale runs a handful of times per split instead of per tile;
// scores are carried in the log2 domain (scale * log2 e applied after the
// MMA).  Two CTAs share an SM (about 109 KB of shared memory each).
//
// Raw log2-domain scores are written to the probability buffer; the combine
// pass turns them into probabilities once the global maximum and sum are known,
// and merges the splits' partial outputs (flash-decoding style) with the gate.
#include <algorithm>

#include "na_internal.cuh"
#include "tc_primitives.cuh"

namespace {

constexpr int DEC_TILE = 64;    // keys per tile: DEC_CWARPS warps x 16 keys
constexpr int DEC_STAGES = 3;
constexpr int DEC_CWARPS = 4;   // consumer warps
constexpr int DEC_THREADS = (DEC_CWARPS + 1) * 32;
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
// A tile of K (and of V) is D / 64 boxes of 64 keys x 64 elements, each a
// 128-byte-swizzled 8 KB block as the tensor-map copies write it: 16-byte
// chunk c of row r sits at chunk c ^ (r % 8), so the eight rows an 8x8
// ldmatrix reads fall in different bank groups.
template <int D, int HPC>
struct __align__(1024) DecSmem {
    bf16 k[DEC_STAGES][DEC_TILE * D];
    bf16 v[DEC_STAGES][DEC_TILE * D];
    float obuf[HPC][D];  // the warps' partial outputs, added in warp order
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

// ------------------------------------------------ warp-level bf16 MMA --
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) and its fragment loads.  For a
// 16x16 A tile, lane l holds rows l/4 and l/4 + 8 at columns 2(l%4), +1 and
// 2(l%4) + 8, +9; for a 16x8 B tile, rows 2(l%4), +1 and +8, +9 of column l/4;
// the 16x8 accumulator holds rows l/4 and l/4 + 8 at columns 2(l%4), +1.

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// The transpose of an 8x8 b16 matrix held one 32-bit pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Byte offset, within a tile of K or V, of 16-byte chunk c (0 .. D/8 - 1) of
// row r: box c / 8, swizzled chunk (c % 8) ^ (r % 8).
__device__ __forceinline__ uint32_t tile_chunk_off(int r, int c)
{
    return (uint32_t)((c >> 3) * (DEC_TILE * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D, int HPC, bool CAPPED>
__global__ void __launch_bounds__(DEC_THREADS, 2)
    decode_split_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v)
{
    constexpr int KS = D / 16;  // k-steps of the score MMA, d-blocks of the PV MMA
    constexpr uint32_t STAGE_BYTES = DEC_TILE * D * (uint32_t)sizeof(bf16);
    extern __shared__ uint8_t smem_raw[];
    DecSmem<D, HPC> &sm = *reinterpret_cast<DecSmem<D, HPC> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;

    if (threadIdx.x == 0) {
        for (int s = 0; s < DEC_STAGES; s++) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], DEC_CWARPS);
        }
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == DEC_CWARPS && lane == 0) {
        tc::prefetch_tmap(&map_k);
        tc::prefetch_tmap(&map_v);
    }
    grid_dependency_wait();
    grid_dependents_launch();
    if (warp == DEC_CWARPS)
        locate_slice(p, lane, sm.slice);
    __syncthreads();
    Walker walk;
    walk.init(sm.slice, p);
    Piece pc;
    const bool ring = (p.flags & NA_RING_CACHE) != 0;  // capacity a multiple of DEC_TILE

    // A piece's keys are positions [kf + k0, kf + k1); its tiles are the
    // DEC_TILE-aligned position ranges covering them (with a ring, aligned
    // ranges map to aligned slot ranges that never cross the end).  Keys of a
    // tile outside the piece are masked.
    if (warp == DEC_CWARPS) {
        // ---------------------------------------------------------- producer --
        if (lane != 0)
            return;
        // K/V lines are read once: first in line for eviction, so the L2 keeps
        // what the caller's other work left there (and the scores the merge
        // pass reads back) instead of writing it back to make room.
        const uint64_t policy = l2_policy_evict_first();
        uint32_t it = 0;
        bool ok = true;
        while (ok && walk.next(p, pc)) {
            const int lo = pc.kf + pc.k0, hi = pc.kf + pc.k1;
            const int row_base = (pc.b * p.KV + pc.kvh) * p.capacity;
            for (int t0 = lo / DEC_TILE * DEC_TILE; t0 < hi; t0 += DEC_TILE, it++) {
                const int stage = it % DEC_STAGES;
                const uint32_t parity = ((it / DEC_STAGES) & 1) ^ 1;
                if (!mbar_wait_bounded(&sm.empty[stage], parity) ||
                    *(volatile int *)&sm.abort_flag) {
                    na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
                    *(volatile int *)&sm.abort_flag = 1;
                    ok = false;
                    break;
                }
                const int row = row_base + (ring ? t0 % p.capacity : t0);
                mbar_arrive_expect_tx(&sm.full[stage], 2 * STAGE_BYTES);
#pragma unroll
                for (int bx = 0; bx < D / 64; bx++) {
                    tc::tma_load_2d_hint(sm.k[stage] + bx * DEC_TILE * 64, &map_k, bx * 64, row,
                                         &sm.full[stage], policy);
                    tc::tma_load_2d_hint(sm.v[stage] + bx * DEC_TILE * 64, &map_v, bx * 64, row,
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
    // Warp w scores keys 16 w .. 16 w + 15 of each tile against the HPC heads
    // (padded to 8) with S^T = K Q^T on m16n8k16 MMAs: K rows from shared
    // memory (ldmatrix), Q as the B operand in registers.  The accumulator
    // leaves lane l with keys l/4 and l/4 + 8 of heads 2(l%4) and 2(l%4) + 1;
    // their bf16 probabilities, transposed in registers (movmatrix), are the B
    // operand of O^T += V^T P^T, whose A operand is the V rows read transposed
    // (ldmatrix .trans).  Products are exact in fp32 and summed in fp32; the
    // scores are scaled to the log2 domain after the MMA.
    const int g = lane >> 2, t = lane & 3;
    const int h0 = 2 * t, h1 = 2 * t + 1;  // this lane's heads (columns)
    const bool v0 = h0 < HPC, v1 = h1 < HPC;
    const uint32_t k_base = smem_addr(sm.k[0]), v_base = smem_addr(sm.v[0]);
    // ldmatrix row addresses: lane l feeds row l % 8 of 8x8 matrix l / 8; the
    // score operand takes matrices (rows +0/+8, columns +0/+8) in the order
    // (0,0) (8,0) (0,8) (8,8), the value operand (transposed) (0,0) (0,8) (8,0) (8,8).
    const int mi = lane >> 3, mr = lane & 7;
    const int ka_row = warp * 16 + (mi & 1) * 8 + mr, ka_col = mi >> 1;
    const int va_row = warp * 16 + (mi >> 1) * 8 + mr, va_col = mi & 1;
    uint32_t it = 0;
    // A warp whose wait timed out keeps walking the pieces so that every warp
    // joins the same named barriers, but does no more waits or writes.
    bool aborted = false;

    while (walk.next(p, pc)) {
        const int lo = pc.kf + pc.k0, hi = pc.kf + pc.k1;
        if (*(volatile int *)&sm.abort_flag)
            aborted = true;
        const int head0 = pc.kvh * p.group + pc.hc * HPC;

        // Q as the B operand: column g is head g (zero past HPC), rows are d.
        uint32_t qf[KS][2];
        {
            const bf16 *qrow = p.q + ((size_t)pc.b * p.H + head0 + min(g, HPC - 1)) * D;
#pragma unroll
            for (int s = 0; s < KS; s++) {
                const uint32_t w0 = *reinterpret_cast<const uint32_t *>(qrow + 16 * s + 2 * t);
                const uint32_t w1 = *reinterpret_cast<const uint32_t *>(qrow + 16 * s + 2 * t + 8);
                qf[s][0] = g < HPC ? w0 : 0u;
                qf[s][1] = g < HPC ? w1 : 0u;
            }
        }
        float acc[KS][4];
#pragma unroll
        for (int s = 0; s < KS; s++)
#pragma unroll
            for (int i = 0; i < 4; i++)
                acc[s][i] = 0.f;
        float m_ref[2] = {-INFINITY, -INFINITY};
        float l_sum[2] = {0.f, 0.f};
        float *prow0 = (p.probs && v0) ? p.probs + ((size_t)pc.b * p.H + head0 + h0) * p.probs_stride
                                        : nullptr;
        float *prow1 = (p.probs && v1) ? p.probs + ((size_t)pc.b * p.H + head0 + h1) * p.probs_stride
                                        : nullptr;

        for (int t0 = lo / DEC_TILE * DEC_TILE; t0 < hi && !aborted; t0 += DEC_TILE, it++) {
            const int stage = it % DEC_STAGES;
            const bool got = mbar_wait_bounded(&sm.full[stage], (it / DEC_STAGES) & 1);
            if (!__all_sync(FULL, got)) {  // warp-uniform before the .sync.aligned MMAs
                if (lane == 0) {
                    na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
                    *(volatile int *)&sm.abort_flag = 1;
                }
                aborted = true;
                break;
            }
            const uint32_t kst = k_base + stage * STAGE_BYTES;
            const uint32_t vst = v_base + stage * STAGE_BYTES;
            const bool partial = t0 < lo || t0 + DEC_TILE > hi;  // the same in every warp
            if (partial) {
                // V rows of masked keys are zeroed: they meet a zero probability
                // in the PV MMA and must not be NaN (unwritten cache slots).
                uint8_t *vrow = reinterpret_cast<uint8_t *>(sm.v[stage]);
                for (int c = lane; c < 16 * (D / 8); c += 32) {
                    const int r = warp * 16 + c / (D / 8), ch = c % (D / 8);
                    const int pos = t0 + r;
                    if (pos < lo || pos >= hi)
                        *reinterpret_cast<uint4 *>(vrow + tile_chunk_off(r, ch)) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }

            // S^T = K Q^T for this warp's 16 keys.
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s = 0; s < KS; s++) {
                uint32_t a[4];
                ldsm_x4(kst + tile_chunk_off(ka_row, 2 * s + ka_col), a);
                mma_bf16_16816(sc, a, qf[s][0], qf[s][1]);
            }
            // Scores (log2 domain), masked outside the piece and for the padding
            // heads; recorded for the combine pass.
            const int pa = t0 + warp * 16 + g, pb = pa + 8;  // this lane's key positions
            const bool ina = pa >= lo && pa < hi, inb = pb >= lo && pb < hi;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                float x = sc[i] * p.scale_log2;
                if constexpr (CAPPED) {  // c tanh(s / c) in the log2 domain, tanh(y) = 1 - 2 / (e^2y + 1)
                    const float e = exp2f(x * p.cap_in);
                    x = p.cap_out * (1.0f - __fdividef(2.0f, e + 1.0f));
                }
                const bool ok = ((i & 2) ? inb : ina) && ((i & 1) ? v1 : v0);
                sc[i] = ok ? x : -INFINITY;
            }
            if (prow0) {
                if (ina)
                    prow0[pa] = sc[0];
                if (inb)
                    prow0[pb] = sc[2];
            }
            if (prow1) {
                if (ina)
                    prow1[pa] = sc[1];
                if (inb)
                    prow1[pb] = sc[3];
            }
            // Tile maximum per head (over the 8 lanes sharing the column), then
            // (rarely) raise the reference maximum.
            float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
            for (int m = 4; m < 32; m <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(FULL, mx0, m));
                mx1 = fmaxf(mx1, __shfl_xor_sync(FULL, mx1, m));
            }
            const bool raise = mx0 > m_ref[0] + kRescaleThreshold || mx1 > m_ref[1] + kRescaleThreshold;
            if (__any_sync(FULL, raise)) {  // warp-uniform
                const float n0 = fmaxf(m_ref[0], mx0), n1 = fmaxf(m_ref[1], mx1);
                const float a0 = (m_ref[0] == -INFINITY) ? 0.f : exp2f(m_ref[0] - n0);
                const float a1 = (m_ref[1] == -INFINITY) ? 0.f : exp2f(m_ref[1] - n1);
                m_ref[0] = n0;
                m_ref[1] = n1;
                l_sum[0] *= a0;
                l_sum[1] *= a1;
#pragma unroll
                for (int s = 0; s < KS; s++) {
                    acc[s][0] *= a0;
                    acc[s][1] *= a1;
                    acc[s][2] *= a0;
                    acc[s][3] *= a1;
                }
            }
            float pr[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                pr[i] = (sc[i] == -INFINITY) ? 0.f : exp2f(sc[i] - m_ref[i & 1]);
                l_sum[i & 1] += pr[i];
            }
            // P^T as the B operand: keys 2(l%4).. of head l/4.
            const uint32_t b0 = movmatrix_trans(pack_bf16x2(pr[0], pr[1]));
            const uint32_t b1 = movmatrix_trans(pack_bf16x2(pr[2], pr[3]));
            // O^T += V^T P^T, one 16-row block of d at a time.
#pragma unroll
            for (int s = 0; s < KS; s++) {
                uint32_t a[4];
                ldsm_x4_trans(vst + tile_chunk_off(va_row, 2 * s + va_col), a);
                mma_bf16_16816(acc[s], a, b0, b1);
            }
            if (partial)
                tc::fence_proxy_async_smem();  // the zeroed rows before the stage's next copy
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.empty[stage]);
        }
        // Sums over the 8 lanes of each column; then the warps' partials are
        // merged in warp order.
#pragma unroll
        for (int m = 4; m < 32; m <<= 1) {
            l_sum[0] += __shfl_xor_sync(FULL, l_sum[0], m);
            l_sum[1] += __shfl_xor_sync(FULL, l_sum[1], m);
        }
        if (g == 0) {
            if (v0) {
                sm.merge_m[warp][h0] = m_ref[0];
                sm.merge_l[warp][h0] = l_sum[0];
            }
            if (v1) {
                sm.merge_m[warp][h1] = m_ref[1];
                sm.merge_l[warp][h1] = l_sum[1];
            }
        }
        named_barrier_sync(1, DEC_CWARPS * 32);
        float M0 = -INFINITY, M1 = -INFINITY;
        if (v0)
#pragma unroll
            for (int ww = 0; ww < DEC_CWARPS; ww++)
                M0 = fmaxf(M0, sm.merge_m[ww][h0]);
        if (v1)
#pragma unroll
            for (int ww = 0; ww < DEC_CWARPS; ww++)
                M1 = fmaxf(M1, sm.merge_m[ww][h1]);
        const float f0 = (m_ref[0] == -INFINITY) ? 0.f : exp2f(m_ref[0] - M0);
        const float f1 = (m_ref[1] == -INFINITY) ? 0.f : exp2f(m_ref[1] - M1);
        for (int ww = 0; ww < DEC_CWARPS; ww++) {
            if (warp == ww) {
#pragma unroll
                for (int s = 0; s < KS; s++) {
                    const int e = 16 * s + g;
                    if (v0) {
                        float *o0 = &sm.obuf[h0][e];
                        o0[0] = ww == 0 ? acc[s][0] * f0 : o0[0] + acc[s][0] * f0;
                        o0[8] = ww == 0 ? acc[s][2] * f0 : o0[8] + acc[s][2] * f0;
                    }
                    if (v1) {
                        float *o1 = &sm.obuf[h1][e];
                        o1[0] = ww == 0 ? acc[s][1] * f1 : o1[0] + acc[s][1] * f1;
                        o1[8] = ww == 0 ? acc[s][3] * f1 : o1[8] + acc[s][3] * f1;
                    }
                }
            }
            named_barrier_sync(1, DEC_CWARPS * 32);
        }
        // Every consumer warp has finished this piece's tiles (or given up): the
        // abort flag is final for the piece.  A piece of a CTA whose wait gave up
        // is written as the marker (max -inf, sum -1), which the merge pass
        // reports instead of merging, so no call ever merges another call's rows.
        const bool bad = *(volatile int *)&sm.abort_flag != 0;
        for (int idx = threadIdx.x; idx < HPC * D; idx += DEC_CWARPS * 32) {
            const int h = idx / D, e = idx - h * D;
            const size_t row = (size_t)pc.id * HPC + h;
            if (bad) {
                if (e == 0) {
                    p.part_ml[row * 2] = -INFINITY;
                    p.part_ml[row * 2 + 1] = -1.0f;
                }
                continue;
            }
            p.part_o[row * D + e] = sm.obuf[h][e];
            if (e == 0) {
                float M = -INFINITY;
#pragma unroll
                for (int ww = 0; ww < DEC_CWARPS; ww++)
                    M = fmaxf(M, sm.merge_m[ww][h]);
                float l = 0.f;
#pragma unroll
                for (int ww = 0; ww < DEC_CWARPS; ww++) {
                    const float mw = sm.merge_m[ww][h];
                    if (mw != -INFINITY)
                        l += sm.merge_l[ww][h] * exp2f(mw - M);
                }
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

__device__ __forceinline__ float gated_elem(float o, bf16 g)
{
    return o * (1.0f / (1.0f + __expf(-__bfloat162float(g))));
}

// 2^x on the MUFU unit (relative error ~2^-22; flushes subnormal results to
// zero, far below the probabilities' 1e-4 absolute bound).
__device__ __forceinline__ float ex2_approx(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Probability of key j from its raw log2-domain score (0 before the window).
__device__ __forceinline__ float prob_of(float raw, int j, int kf, float M, float inv_l)
{
    return j < kf ? 0.f : ex2_approx(raw - M) * inv_l;
}

// Combine pass: one CTA per (sequence, query head).  The sequence length and
// the stream's piece span are loaded together; then one thread requests the
// row's raw scores as bulk copies into shared memory (two buffers of `half`
// 16-byte groups, refilled in turn for long rows) while the warps load every
// piece's (max, sum) and the first pieces' output rows; no registers are
// spent on loads in flight, so many CTAs share an SM (six, held there by the
// two 16 KB buffers).  128 threads: 256-thread CTAs took 1% longer per
// decode call.
constexpr int kCombThreads = 128;
constexpr int kCombMaxHalf = 1024;  // 16-byte groups per buffer (4096 keys)

template <int D>
__global__ void __launch_bounds__(kCombThreads) decode_combine_kernel(const DecodeParams p,
                                                                      const int half)
{
    extern __shared__ __align__(16) float4 sbuf[];  // [2][half]
    __shared__ uint64_t bar[2];
    constexpr int NT = kCombThreads;
    constexpr int PO = 4;  // pieces' output elements requested with the scores
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
    }
    __syncthreads();
    grid_dependency_wait();
    grid_dependents_launch();
    const int bh = blockIdx.x;
    const int b = bh / p.H;
    const int h = bh - b * p.H;
    const int hpc = p.group / p.head_chunks;
    const int kvh = h / p.group, r = h - kvh * p.group;
    const int stream = (b * p.KV + kvh) * p.head_chunks + r / hpc;
    const int n = __ldg(p.kv_lens + b);
    const int first = p.piece_span[2 * stream], last = p.piece_span[2 * stream + 1];
    bf16 *out = p.out + (size_t)bh * D;
    auto zero_out = [&]() {
        for (int e = threadIdx.x; e < D; e += NT)
            out[e] = __float2bfloat16_rn(0.f);
    };
    if (n < 0 || (!(p.flags & NA_RING_CACHE) && n > p.capacity) || n > p.max_kv_len) {
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_CAPACITY);
        zero_out();
        return;
    }
    if (n == 0) {
        zero_out();
        return;
    }
    if (first < 0 || last < first || last >= p.max_pieces) {  // the split pass gave up
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
        zero_out();
        return;
    }
    // Pieces of this head's stream: ids first..last, HPC heads per row group.
    const int ns = last - first + 1;
    const size_t row0 = (size_t)first * hpc + (r % hpc);
    const float *ml = p.part_ml + row0 * 2;
    const float *po = p.part_o + row0 * D;

    // The row is walked as a scalar head up to its first 16-byte boundary,
    // 16-byte groups of four keys (through shared memory), and a scalar tail.
    float *pr = p.probs ? p.probs + (size_t)bh * p.probs_stride : nullptr;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(pr);
    const int pre = (addr & 3) ? n : min(n, (int)(((16 - (addr & 15)) & 15) >> 2));
    const int n4 = pr ? (n - pre) >> 2 : 0;
    float4 *pr4 = reinterpret_cast<float4 *>(pr + pre);
    const int nchunks = (n4 + half - 1) / half;
    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int c) {  // one thread: chunk c of the row into buffer c % 2
        const int i0 = c * half, cnt = min(half, n4 - i0);
        mbar_arrive_expect_tx(&bar[c & 1], (uint32_t)cnt * 16u);
        bulk_copy_g2s(sbuf + (c & 1) * half, pr4 + i0, (uint32_t)cnt * 16u, &bar[c & 1], policy);
    };
    int issued = min(nchunks, 2), waited = 0;
    if (threadIdx.x == 0)
        for (int c = 0; c < issued; c++)
            issue(c);
    // Copies still in flight land before the CTA exits (one thread waits).
    auto drain = [&]() {
        if (threadIdx.x == 0)
            for (int c = waited; c < issued; c++)
                if (!mbar_wait_bounded(&bar[c & 1], (c >> 1) & 1))
                    na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
    };

    const int lane = threadIdx.x & 31;
    float m0, l0;
    merge_lane_piece(ml, hpc, ns, lane, m0, l0);
    const int e0 = threadIdx.x;  // output element (threads below D)
    float xo[PO], mo[PO];
#pragma unroll
    for (int u = 0; u < PO; u++) {
        xo[u] = 0.f;
        mo[u] = -INFINITY;
        if (e0 < D && u < ns) {
            mo[u] = ml[2 * hpc * u];
            xo[u] = po[(size_t)u * hpc * D + e0];
        }
    }

    // Row maximum and sum over the pieces: every warp reduces them (the same
    // loads and order in every warp, so the outcome is the CTA's).
    float M, inv_l;
    if (!merge_weights_from(m0, l0, ml, hpc, ns, lane, M, inv_l)) {  // a split-pass wait gave up
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
        zero_out();
        drain();
        return;
    }

    if (e0 < D) {  // pieces' rows weighted by 2^(m_s - M), added in piece order
        float o = 0.f;
#pragma unroll
        for (int u = 0; u < PO; u++)
            if (mo[u] != -INFINITY)
                o += xo[u] * exp2f(mo[u] - M);
        for (int s = PO; s < ns; s++) {
            const float m = ml[2 * hpc * s];
            if (m != -INFINITY)
                o += po[(size_t)s * hpc * D + e0] * exp2f(m - M);
        }
        o *= inv_l;
        if ((p.flags & NA_OUT_GATE) && p.gate)
            o = gated_elem(o, p.gate[(size_t)bh * D + e0]);
        out[e0] = __float2bfloat16_rn(o);
    }
    if (pr) {
        // keys before the window (none without one) get probability 0
        const int kf = (p.window > 0 && n > p.window) ? n - p.window : 0;
        auto prob = [&](float raw, int j) { return prob_of(raw, j, kf, M, inv_l); };
        for (int c = 0; c < nchunks; c++) {
            const bool got = mbar_wait_bounded(&bar[c & 1], (c >> 1) & 1);
            if (!__syncthreads_and(got)) {
                if (threadIdx.x == 0)
                    na_report(p.status, NA_ERR_DEVICE_TIMEOUT);
                drain();
                return;
            }
            waited = c + 1;
            const int i0 = c * half, cnt = min(half, n4 - i0);
            const float4 *src = sbuf + (c & 1) * half;
            for (int i = threadIdx.x; i < cnt; i += NT) {
                const int j = pre + 4 * (i0 + i);
                float4 y = src[i];
                y.x = prob(y.x, j);
                y.y = prob(y.y, j + 1);
                y.z = prob(y.z, j + 2);
                y.w = prob(y.w, j + 3);
                pr4[i0 + i] = y;
            }
            if (c + 2 < nchunks) {
                __syncthreads();  // every thread is done with this buffer
                if (threadIdx.x == 0)
                    issue(c + 2);
                issued = c + 3;
            }
        }
        for (int j = threadIdx.x; j < pre; j += NT)
            pr[j] = prob(pr[j], j);
        for (int j = pre + (n4 << 2) + threadIdx.x; j < n; j += NT)
            pr[j] = prob(pr[j], j);
    }
    drain();
}

template <int D, int HPC, bool CAPPED>
cudaError_t launch_split(const DecodeParams &p, cudaStream_t stream)
{
    // K and V as 2-D tensors of cache rows ((sequence, kv head, slot) x D),
    // read in boxes of DEC_TILE rows x 64 elements.
    CUtensorMap mk, mv;
    const cuuint64_t rows = (cuuint64_t)p.cache_batch * p.KV * p.capacity;
    const cuuint64_t dims[2] = {(cuuint64_t)D, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    const cuuint32_t box[2] = {64, DEC_TILE};
    if (!make_bf16_tile_map(&mk, p.cache_k, 2, dims, strides, box) ||
        !make_bf16_tile_map(&mv, p.cache_v, 2, dims, strides, box))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(DecSmem<D, HPC>) + 1024;  // + alignment slack
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
                         stream, p, mk, mv);
}

template <int D, int HPC>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t stream)
{
    cudaError_t e = p.cap_out > 0.f ? launch_split<D, HPC, true>(p, stream)
                                    : launch_split<D, HPC, false>(p, stream);
    if (e != cudaSuccess)
        return e;
    // Two shared-memory buffers that hold a row of max_kv_len keys between
    // them (up to kCombMaxHalf groups of four keys each).
    const int groups = (p.max_kv_len + 3) / 4;
    const int half = std::min(kCombMaxHalf, std::max(32, ((groups + 1) / 2 + 31) / 32 * 32));
    return launch_kernel(decode_combine_kernel<D>, dim3(p.batch * p.H), dim3(kCombThreads),
                         (size_t)2 * half * sizeof(float4), stream, p, half);
}

}  // namespace

int decode_key_tile() { return DEC_TILE; }

int decode_ctas_per_sm() { return 2; }

cudaError_t launch_decode(const DecodeParams &p, int d, int heads_per_cta, cudaStream_t stream)
{
    if (d == 128) {
        switch (heads_per_cta) {
        case 8: return launch_decode_t<128, 8>(p, stream);
        case 4: return launch_decode_t<128, 4>(p, stream);
        case 2: return launch_decode_t<128, 2>(p, stream);
        default: return launch_decode_t<128, 1>(p, stream);
        }
    }
    switch (heads_per_cta) {
    case 8: return launch_decode_t<64, 8>(p, stream);
    case 4: return launch_decode_t<64, 4>(p, stream);
    case 2: return launch_decode_t<64, 2>(p, stream);
    default: return launch_decode_t<64, 1>(p, stream);
    }
}

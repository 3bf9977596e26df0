// prefill.cu -- causal GQA attention of a chunk of new tokens against the
// per-sequence KV cache, on the sm_100-family tensor cores (tcgen05 + TMEM +
// TMA).  Semantics: cortiq-engine src/attention.rs, fn qwen_attention_batch
// (query bi of a chunk sees keys 0 .. s0 + bi: all history and the earlier
// keys of its own chunk), fn attention_head (softmax(q.k * scale) . V per row)
// and fn apply_gate (sigmoid gate on the output).
//
// One CTA owns 128 query rows of one (sequence, query head) -- the 128 lanes
// of tensor memory -- and walks the 128-key tiles of kv head h / (H / KV) that
// those rows can see (tiles wholly above the diagonal are never loaded).
// Warp roles (8 warps):
//   warp 0     TMA producer: the Q tile once, then K and V tiles into a
//              3-stage ring (128-byte swizzled, as the MMA descriptors expect);
//              the Q tile and the first three stages are issued by the thread
//              that initialises the barriers, before the CTA-wide barrier;
//   warp 1     allocates tensor memory; one lane issues S_j = Q K_j^T (SS, both
//              K-major) into one of three S buffers in tensor memory;
//   warp 2     one lane issues O += P_j V_j (TS: P read from tensor memory over
//              S_j, V MN-major).  Two issuing threads, because one thread cannot
//              keep the tensor core busy with M = N = 128 instructions (each
//              takes ~116 SM cycles to issue, measured on GB300, against ~64
//              cycles of math);
//   warps 4-7  softmax, one query row per thread (its TMEM lane): load S_j,
//              mask, online max in the log2 domain (the reference max is raised
//              only when it grows by more than 2^8, and only then is the O row
//              rescaled in tensor memory), exponentiate on the MUFU unit
//              (measured faster than moving part of the exponentials to a
//              polynomial on the FMA pipe), write P_j as bf16 over S_j, and
//              finally normalise O and stage it through the idle K ring;
//   all warps  then gate and store 16 of the staged rows each, a whole row per
//              instruction (coalesced) instead of one 16-byte piece of 32
//              different rows; warps 0-3 prefetch their gate rows at the start.
// With three S buffers the tensor core computes S_{j+1} and S_{j+2} while the
// softmax works on tile j, and PV_j runs while it prepares P_{j+1}.
//
#include <climits>
#include <cuda.h>
#include <mutex>

#include "na_internal.cuh"
#include "tc_primitives.cuh"

namespace {

constexpr int BM = 128;      // query rows per CTA (tensor-memory lanes)
constexpr int BN = 128;      // keys per tile
constexpr int STAGES = 3;    // K/V shared-memory ring depth
constexpr int NUM_S = 3;     // S/P buffers in tensor memory
constexpr int THREADS = 256; // 8 warps: producer, S issuer, PV issuer, idle, 4 softmax
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL0 = 128;  // S buffer i at columns 128 (i + 1); O at column 0

template <int D>
struct __align__(1024) TcSmem {
    static constexpr int KB = D / 64;  // 64-wide column blocks of a row
    bf16 q[KB][BM * 64];
    bf16 k[STAGES][KB][BN * 64];
    bf16 v[STAGES][KB][BN * 64];
    uint64_t q_full;
    uint64_t k_full[STAGES], k_empty[STAGES], v_full[STAGES], v_empty[STAGES];
    uint64_t s_full[NUM_S], s_free[NUM_S], p_full[NUM_S];
    uint64_t o_done[NUM_S], drain[2];  // o_done[b]: the PVs of tiles b, b + NUM_S, ...
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
constexpr size_t tc_smem_bytes()
{
    // at least ~116 KB so that a single CTA owns the SM (and its tensor memory)
    return (sizeof(TcSmem<D>) + 1024) > (116u << 10) ? sizeof(TcSmem<D>) + 1024 : (116u << 10);
}

__device__ __forceinline__ bool aborted(const int *flag) { return *(volatile const int *)flag != 0; }

__device__ __forceinline__ void set_abort(int *flag, int32_t *status)
{
    *(volatile int *)flag = 1;
    na_report(status, NA_ERR_DEVICE_TIMEOUT);
}

// A bounded wait whose outcome is only reported: the drains before exit (copies
// in flight, MMAs before tensor memory is released), where there is nothing
// left to skip.  A wait that gives up writes NA_ERR_DEVICE_TIMEOUT.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, int32_t *status)
{
    if (!mbar_wait_bounded(bar, parity))
        na_report(status, NA_ERR_DEVICE_TIMEOUT);
}

// A bounded wait whose result every lane of the warp shares: the softmax warps
// follow it with warp-collective tensor-memory loads and stores, which no lane
// may skip while others execute them.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const int *abort_flag)
{
    const bool done = mbar_wait_bounded(bar, parity) && !aborted(abort_flag);
    return __all_sync(0xffffffffu, done);
}

__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// 2^x on the MUFU unit (approximate, flushes subnormal results to zero).
__device__ __forceinline__ float ex2_mufu(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

template <int D, bool CAPPED>
__global__ void __launch_bounds__(THREADS, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v)
{
    constexpr int KB = D / 64;
    extern __shared__ uint8_t smem_raw[];
    TcSmem<D> &sm = *reinterpret_cast<TcSmem<D> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Prologue that reads no global memory: descriptor prefetch, barriers and
    // tensor memory; it may overlap the end of the previous kernel.
    if (threadIdx.x == 0) {
        tc::prefetch_tmap(&map_q);
        tc::prefetch_tmap(&map_k);
        tc::prefetch_tmap(&map_v);
        mbar_init(&sm.q_full, 1);
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&sm.k_full[s], 1);
            mbar_init(&sm.v_full[s], 1);
            mbar_init(&sm.k_empty[s], 1);
            mbar_init(&sm.v_empty[s], 1);
        }
        for (int s = 0; s < NUM_S; s++) {
            mbar_init(&sm.s_full[s], 1);
            mbar_init(&sm.s_free[s], 1);
            mbar_init(&sm.p_full[s], 4);
        }
        for (int s = 0; s < NUM_S; s++)
            mbar_init(&sm.o_done[s], 1);
        mbar_init(&sm.drain[0], 1);
        mbar_init(&sm.drain[1], 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    // The block's unit: CTAs 0 .. full_units - 1 take whole units, the rest one
    // of num_splits key ranges of a tail unit.  Units run in the order
    // (query tile, head group, sequence slot), heaviest query tiles first.
    const int idx = blockIdx.x;
    const bool in_tail = idx >= p.full_units;
    const int nsplit = in_tail ? p.num_splits : 1;
    const int tail_unit = in_tail ? (idx - p.full_units) / p.num_splits : 0;
    const int split = in_tail ? (idx - p.full_units) - tail_unit * p.num_splits : 0;
    const int unit = in_tail ? p.full_units + tail_unit : idx;
    const int hg = (unit / p.q_tiles) % p.HG;
    const int slot = unit / (p.q_tiles * p.HG);
    const int qt = p.q_tiles - 1 - (unit % p.q_tiles);  // heaviest (latest) query tiles first
    // A tile that certainly has rows -- a sequence's first, or with a single
    // sequence any tile below the host-known token count -- takes the tensor
    // memory before the wait and issues its first copies speculatively.
    // Other tiles may be empty padding; they check first and leave at once.
    const bool eager = p.batch == 1 && p.window == 0 && qt * p.tile_tokens < p.total_tokens;
    if (eager && warp == 1)
        tc::tmem_alloc(&sm.tmem_base, TMEM_COLS);
    grid_dependency_wait();
    grid_dependents_launch();

    // ------------------------------------------------------------ the tile --
    // The 128 rows are tile_tokens tokens x pack query heads of one kv group,
    // token-major: row r is token r >> pack_shift, head h0 + (r & (pack - 1)).
    const int pack_shift = __ffs(p.pack) - 1;
    const int h0 = hg * p.pack;
    const int kvh = h0 / p.group;
    const int r0 = qt * p.tile_tokens;  // first token of the tile within the sequence
    const int split_off = nsplit > 1 ? split * p.split_len : 0;
    // The sequence this block serves.  With several sequences (up to 32) the
    // slots go to sequences in order of decreasing end position (prior + new
    // tokens), so the longest tiles start first (list scheduling of this
    // one-CTA-per-SM grid: measured ~10% shorter on mixed lengths).  The
    // bounds of every sequence come in the same round of loads.
    int b = slot, tok0, n_new, prior;
    if (p.batch > 1 && p.batch <= 32) {
        int c0 = 0, c1 = 0, pl = 0, key = -1;
        if (lane < p.batch) {
            c0 = __ldg(p.cu_seqlens + lane);
            c1 = __ldg(p.cu_seqlens + lane + 1);
            pl = __ldg(p.cache_lens + lane);
            key = pl + (c1 - c0);
        }
        int rank = 0;
        for (int j = 0; j < p.batch; j++) {
            const int kj = __shfl_sync(0xffffffffu, key, j);
            rank += (kj > key) || (kj == key && j < lane);
        }
        const unsigned m = __ballot_sync(0xffffffffu, lane < p.batch && rank == slot);
        const int src = __ffs(m) - 1;  // ranks are a permutation of 0 .. batch - 1
        b = src;
        tok0 = __shfl_sync(0xffffffffu, c0, src);
        n_new = __shfl_sync(0xffffffffu, c1, src) - tok0;
        prior = __shfl_sync(0xffffffffu, pl, src);
    }
    const int spec_row = (b * p.KV + kvh) * p.capacity + split_off;  // tile 0 without a window
    // K/V tiles that no other CTA of the call reads (one query tile holding
    // every query head of its kv group) are loaded first in line for L2
    // eviction, so streaming them does not push out lines worth keeping.
    const bool read_once = p.kv_read_once != 0;
    const uint64_t kv_policy = l2_policy_evict_first();
    auto load_kv = [&](void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
        if (read_once)
            tc::tma_load_2d_hint(dst, map, x, y, bar, kv_policy);
        else
            tc::tma_load_2d(dst, map, x, y, bar);
    };
    // With a single sequence the first K and V tiles depend only on the block,
    // and its tokens start at row 0: those copies are issued before the
    // sequence bounds arrive, overlapping that round trip (a CTA that turns out
    // to have no work waits for them before it exits).
    const bool early_q = eager;
    if (eager && threadIdx.x == 0) {
        mbar_arrive_expect_tx(&sm.q_full, KB * BM * 128);
        for (int kb = 0; kb < KB; kb++)
            tc::tma_load_3d(sm.q[kb], &map_q, kb * 64, h0, r0, &sm.q_full);
        mbar_arrive_expect_tx(&sm.k_full[0], KB * BN * 128);
        for (int kb = 0; kb < KB; kb++)
            load_kv(sm.k[0][kb], &map_k, kb * 64, spec_row, &sm.k_full[0]);
        mbar_arrive_expect_tx(&sm.v_full[0], KB * BN * 128);
        for (int kb = 0; kb < KB; kb++)
            load_kv(sm.v[0][kb], &map_v, kb * 64, spec_row, &sm.v_full[0]);
    }
    if (!(p.batch > 1 && p.batch <= 32)) {
        tok0 = __ldg(p.cu_seqlens + b);
        n_new = __ldg(p.cu_seqlens + b + 1) - tok0;
        prior = __ldg(p.cache_lens + b);
    }
    const int rows_tok = min(p.tile_tokens, n_new - r0);
    const int rows = rows_tok << pack_shift;  // valid tensor-memory rows
    const int pos_lo = prior + r0, pos_hi = prior + r0 + rows_tok - 1;
    // Keys the tile can see: from the key tile holding the first row's window
    // start (0 without a window) to the last row; splits cut that range.
    const int win_tile = p.window > 0 ? max(0, pos_lo - p.window + 1) / BN * BN : 0;
    const int k_begin = win_tile + split_off;
    // Cache row of key tile j: with a ring the key position wraps at the
    // capacity (a multiple of the key tile, so a tile never straddles the end).
    const bool ring = (p.flags & NA_RING_CACHE) != 0;
    const int kv_row0 = (b * p.KV + kvh) * p.capacity;
    auto tile_row = [&](int j) {
        const int k = k_begin + j * BN;
        return kv_row0 + (ring ? k % p.capacity : k);
    };
    int k_end = pos_hi + 1;
    if (nsplit > 1)
        k_end = min(k_end, k_begin + p.split_len);
    bool run = true;  // uniform over the CTA
    // A sequence must lie inside the call's tokens (cu_seqlens within
    // [0, total_tokens]): its rows are read from Q and written to out.
    if (n_new > p.max_new_len || (b == 0 && tok0 != 0) || tok0 < 0 ||
        (long long)tok0 + n_new > p.total_tokens) {
        if (qt == 0 && hg == 0 && split == 0 && threadIdx.x == 0)
            na_report(p.status, NA_ERR_INVALID_ARG);
        run = false;
    } else if (r0 >= n_new) {
        run = false;
    } else if (prior < 0 || (!ring && pos_hi >= p.capacity) || pos_hi >= p.max_total_len) {
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_CAPACITY);
        run = false;
    } else if (k_begin >= k_end) {
        run = false;
    }
    if (!run) {
        if (eager) {  // let the early copies land, give the tensor memory back
            if (threadIdx.x == 0) {
                if (early_q)
                    drain_wait(&sm.q_full, 0, p.status);
                drain_wait(&sm.k_full[0], 0, p.status);
                drain_wait(&sm.v_full[0], 0, p.status);
            }
            tc::fence_before_sync();
            __syncthreads();
            if (warp == 1) {
                tc::fence_after_sync();
                tc::tmem_dealloc(sm.tmem_base, TMEM_COLS);
            }
        }
        return;
    }
    if (!eager && warp == 1)
        tc::tmem_alloc(&sm.tmem_base, TMEM_COLS);
    const int n_tiles = (k_end - k_begin + BN - 1) / BN;
    const int pre = n_tiles < STAGES ? n_tiles : STAGES;  // tiles loaded before the barrier

    if (threadIdx.x == 0) {
        // The Q tile (unless already issued) and the remaining first ring
        // stages go out before the CTA-wide barrier (fresh stages need no
        // wait), so these copies overlap the tensor-memory allocation and the
        // barrier itself.
        if (!early_q) {
            mbar_arrive_expect_tx(&sm.q_full, KB * BM * 128);
            for (int kb = 0; kb < KB; kb++)
                tc::tma_load_3d(sm.q[kb], &map_q, kb * 64, h0, tok0 + r0, &sm.q_full);
        }
        for (int j = eager ? 1 : 0; j < pre; j++) {
            mbar_arrive_expect_tx(&sm.k_full[j], KB * BN * 128);
            for (int kb = 0; kb < KB; kb++)
                load_kv(sm.k[j][kb], &map_k, kb * 64, tile_row(j), &sm.k_full[j]);
            mbar_arrive_expect_tx(&sm.v_full[j], KB * BN * 128);
            for (int kb = 0; kb < KB; kb++)
                load_kv(sm.v[j][kb], &map_v, kb * 64, tile_row(j), &sm.v_full[j]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = sm.tmem_base;

    // Output rows are staged in shared memory by the softmax warps (they hold
    // the tensor-memory lanes) and then stored by all eight warps, SR rows
    // each: one warp per sub-partition storing 32 rows back to back was
    // latency-bound (~1.5 us per CTA, 3.3 us with the gate).  A warp's gate
    // words for its rows are requested early -- warps 0-3 now, the softmax
    // warps after their last tile.
    constexpr int LDS = D + 4;   // staged row stride (floats): conflict-free row writes
    constexpr int EPL = D / 32;  // elements per lane in the row stores
    constexpr int GW = D / 64;   // 32-bit words of gate per lane and row
    constexpr int SR = BM / 8;   // rows stored per warp
    float *stage = reinterpret_cast<float *>(&sm.k[0][0][0]);  // the K ring, idle by then
    const bool split_out = nsplit > 1;
    // rows of this piece in the workspace: [tail unit][split][row]
    const size_t piece_row0 = ((size_t)tail_unit * p.num_splits + split) * BM;
    const bool gated_out = !split_out && (p.flags & NA_OUT_GATE) && p.gate;
    uint32_t gq[SR][GW];
    auto load_gate = [&]() {
#pragma unroll
        for (int i = 0; i < SR; i++) {
            const int rr = warp * SR + i;
            const size_t off = ((size_t)(tok0 + r0 + (rr >> pack_shift)) * p.H + h0 +
                                (rr & (p.pack - 1))) * D + lane * 2 * GW;
            gq[i][0] = 0;
            if constexpr (GW == 2)
                gq[i][1] = 0;
            if (rr < rows) {
                if constexpr (GW == 2) {
                    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p.gate + off));
                    gq[i][0] = u.x;
                    gq[i][1] = u.y;
                } else {
                    gq[i][0] = __ldg(reinterpret_cast<const unsigned int *>(p.gate + off));
                }
            }
        }
    };
    if (warp < 4 && gated_out)
        load_gate();

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            int issued = pre;
            for (int j = pre; j < n_tiles; j++) {
                const int st = j % STAGES;
                const uint32_t par = ((j / STAGES) & 1) ^ 1;
                if (!mbar_wait_bounded(&sm.k_empty[st], par) || aborted(&sm.abort_flag)) {
                    set_abort(&sm.abort_flag, p.status);
                    break;
                }
                mbar_arrive_expect_tx(&sm.k_full[st], KB * BN * 128);
                for (int kb = 0; kb < KB; kb++)
                    load_kv(sm.k[st][kb], &map_k, kb * 64, tile_row(j), &sm.k_full[st]);
                if (!mbar_wait_bounded(&sm.v_empty[st], par) || aborted(&sm.abort_flag)) {
                    set_abort(&sm.abort_flag, p.status);
                    drain_wait(&sm.k_full[st], (j / STAGES) & 1, p.status);
                    break;
                }
                mbar_arrive_expect_tx(&sm.v_full[st], KB * BN * 128);
                for (int kb = 0; kb < KB; kb++)
                    load_kv(sm.v[st][kb], &map_v, kb * 64, tile_row(j), &sm.v_full[st]);
                issued = j + 1;
            }
            // every copy issued lands before the CTA can exit
            drain_wait(&sm.q_full, 0, p.status);
            for (int j = issued - 1; j >= 0 && j >= issued - STAGES; j--) {
                drain_wait(&sm.k_full[j % STAGES], (j / STAGES) & 1, p.status);
                drain_wait(&sm.v_full[j % STAGES], (j / STAGES) & 1, p.status);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------- S = Q K^T issue --
        if (lane == 0) {
            constexpr uint32_t idesc_s = tc::idesc_bf16_f32(BM, BN, false, false);
            // Descriptors of the Q tile and of K stage 0; a 64-wide column block
            // (BM = BN rows of 128 B) is BLK16 16-byte units, a K stage K_STAGE16.
            constexpr uint32_t BLK16 = (BM * 128) >> 4;
            constexpr uint32_t K_STAGE16 = (KB * BN * 128) >> 4;
            static_assert(BM == BN, "one column-block stride for Q and K");
            const uint64_t qd0 = tc::desc_kmajor_sw128(smem_addr(sm.q[0]));
            const uint64_t kd0 = tc::desc_kmajor_sw128(smem_addr(sm.k[0][0]));
            bool ok = mbar_wait_bounded(&sm.q_full, 0);
            bool any = false;
            for (int j = 0; ok && j < n_tiles; j++) {
                const int st = j % STAGES, sb = j % NUM_S;
                ok = mbar_wait_bounded(&sm.k_full[st], (j / STAGES) & 1);
                if (ok && j >= NUM_S)
                    ok = mbar_wait_bounded(&sm.s_free[sb], ((j / NUM_S) - 1) & 1);
                if (!ok || aborted(&sm.abort_flag))
                    break;
                tc::fence_after_sync();
                const uint32_t s_t = tmem + S_COL0 * (sb + 1);
                const uint64_t kd = kd0 + (uint64_t)(st * K_STAGE16);
#pragma unroll
                for (int k = 0; k < D / 16; k++) {  // descriptor start addresses advance in 16-byte units
                    const uint32_t off = (k >> 2) * BLK16 + (k & 3) * 2;
                    tc::mma_ss(s_t, qd0 + off, kd + off, idesc_s, k > 0);
                }
                tc::mma_commit(&sm.s_full[sb]);
                tc::mma_commit(&sm.k_empty[st]);
                any = true;
            }
            if (!ok)
                set_abort(&sm.abort_flag, p.status);
            if (any) {  // all issued MMAs complete before tensor memory is released
                tc::mma_commit(&sm.drain[0]);
                drain_wait(&sm.drain[0], 0, p.status);
            }
        }
    } else if (warp == 2) {
        // --------------------------------------------------- O += P V issue --
        if (lane == 0) {
            constexpr uint32_t idesc_o = tc::idesc_bf16_f32(BM, D, false, true);
            constexpr uint32_t V_STAGE16 = (KB * BN * 128) >> 4;  // a V stage in 16-byte units
            const uint64_t vd0 = tc::desc_mnmajor_sw128(smem_addr(sm.v[0][0]), BN * 128);
            bool ok = true, any = false;
            for (int j = 0; ok && j < n_tiles; j++) {
                const int st = j % STAGES, sb = j % NUM_S;
                ok = mbar_wait_bounded(&sm.p_full[sb], (j / NUM_S) & 1);
                if (ok)
                    ok = mbar_wait_bounded(&sm.v_full[st], (j / STAGES) & 1);
                if (!ok || aborted(&sm.abort_flag))
                    break;
                tc::fence_after_sync();
                const uint32_t p_t = tmem + S_COL0 * (sb + 1);
                const uint64_t vd = vd0 + (uint64_t)(st * V_STAGE16);
#pragma unroll
                for (int k = 0; k < BN / 16; k++)  // 16 keys = 16 rows of 128 B per step
                    tc::mma_ts(tmem, p_t + k * 8, vd + (uint64_t)(k * 128), idesc_o, j > 0 || k > 0);
                tc::mma_commit(&sm.s_free[sb]);
                tc::mma_commit(&sm.v_empty[st]);
                tc::mma_commit(&sm.o_done[sb]);
                any = true;
            }
            if (!ok)
                set_abort(&sm.abort_flag, p.status);
            if (any) {
                tc::mma_commit(&sm.drain[1]);
                drain_wait(&sm.drain[1], 0, p.status);
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------- softmax --
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // query row == TMEM lane
        const int row_pos = pos_lo + (r >> pack_shift);
        const int row_lo = p.window > 0 ? row_pos - p.window + 1 : INT_MIN;  // first visible key
        constexpr bool capped = CAPPED;
        // soft-capped scores, kept in the raw score's units so the rest of the
        // softmax is unchanged: s' = (c / scale) tanh(s scale / c), with
        // tanh(y) = 1 - 2 / (e^(2y) + 1)
        const float cap_in = capped ? 2.0f * p.scale_log2 / p.softcap : 0.f;
        const float cap_out = capped ? p.softcap * NA_LOG2E / p.scale_log2 : 0.f;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t o_t = tmem + lane_off;
        const float sl2 = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; j++) {
            const int sb = j % NUM_S;
            const int j0 = k_begin + j * BN;
            const uint32_t s_t = tmem + S_COL0 * (sb + 1) + lane_off;
            if (!warp_wait(&sm.s_full[sb], (j / NUM_S) & 1, &sm.abort_flag)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; c++)
                tc::tmem_ld32(s_t + c * 32, sr[c]);
            tc::tmem_wait_ld();

            if constexpr (capped) {
#pragma unroll
                for (int c = 0; c < 4; c++)
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        const float e = ex2_mufu(__uint_as_float(sr[c][i]) * cap_in);
                        sr[c][i] = __float_as_uint(cap_out * (1.0f - __fdividef(2.0f, e + 1.0f)));
                    }
            }
            const bool need_mask = (j0 + BN - 1 > pos_lo) || (j0 + BN > k_end) || (j0 < row_lo);
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < 4; c++)
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        const int key = j0 + c * 32 + i;
                        if (key > row_pos || key >= k_end || key < row_lo)
                            sr[c][i] = __float_as_uint(-INFINITY);
                    }
            }
            // row maximum: four independent chains of 3-input max
            float mxa = -INFINITY, mxb = -INFINITY, mxc = -INFINITY, mxd = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; c++)
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    mxa = max3f(mxa, __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
                    mxb = max3f(mxb, __uint_as_float(sr[c][i + 2]), __uint_as_float(sr[c][i + 3]));
                    mxc = max3f(mxc, __uint_as_float(sr[c][i + 4]), __uint_as_float(sr[c][i + 5]));
                    mxd = max3f(mxd, __uint_as_float(sr[c][i + 6]), __uint_as_float(sr[c][i + 7]));
                }
            const float mx = max3f(mxa, mxb, fmaxf(mxc, mxd));
            const float mxs = mx * sl2;
            float alpha = 1.f;
            bool corr = false;
            if (mxs > m_ref + 8.0f) {
                alpha = (m_ref == -INFINITY) ? 0.f : ex2_mufu(m_ref - mxs);
                corr = (m_ref != -INFINITY);
                m_ref = mxs;
            }
            const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
            const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(neg_m, neg_m);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const float2 x = __ffma2_rn(
                        make_float2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])),
                        sc2, nm2);
                    const float2 pp = make_float2(ex2_mufu(x.x), ex2_mufu(x.y));
                    acc[i & 3] = __fadd2_rn(acc[i & 3], pp);
                    pk[i] = pack_bf16x2(pp.x, pp.y);
                }
                tc::tmem_st16(s_t + c * 16, pk);
            }
            const float2 acc01 = __fadd2_rn(acc[0], acc[1]), acc23 = __fadd2_rn(acc[2], acc[3]);
            const float rs = (acc01.x + acc01.y) + (acc23.x + acc23.y);
            tc::tmem_wait_st();

            if (j0 + BN > k_end) {
                // Key rows past the valid range hold whatever the cache has there;
                // zero them so P * V sees no non-finite values.
                const int st = j % STAGES;
                if (!warp_wait(&sm.v_full[st], (j / STAGES) & 1, &sm.abort_flag)) {
                    ok = false;
                    break;
                }
                if (r >= k_end - j0) {
#pragma unroll
                    for (int kb = 0; kb < KB; kb++) {
                        uint4 *row = reinterpret_cast<uint4 *>(sm.v[st][kb] + r * 64);
#pragma unroll
                        for (int c = 0; c < 8; c++)
                            row[c] = make_uint4(0, 0, 0, 0);
                    }
                }
                tc::fence_proxy_async_smem();
            }
            // O is touched here only to rescale it (rare), and then PV(j-1) must
            // have landed.  PV(j) commits to o_done[j % NUM_S], so a wait there is
            // exact however rarely the softmax looks: the barrier's previous
            // phase, PV(j-1-NUM_S), completed before S(j-1) could be issued (its
            // S buffer had to be free), and its next one, PV(j-1+NUM_S), needs a
            // P this warp has not written yet.  Waiting for PV(j-1) on every tile
            // kept PV(j) from being queued behind it.
            if (j >= 1 && __any_sync(0xffffffffu, corr)) {
                if (!warp_wait(&sm.o_done[(j - 1) % NUM_S], ((j - 1) / NUM_S) & 1, &sm.abort_flag)) {
                    ok = false;
                    break;
                }
                // rescale this warp's O rows (PV(j-1) has landed)
                tc::fence_after_sync();
                const float a = corr ? alpha : 1.f;
#pragma unroll
                for (int c = 0; c < D / 32; c++) {
                    uint32_t o[32];
                    tc::tmem_ld32(o_t + c * 32, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                    tc::tmem_st32(o_t + c * 32, o);
                }
                tc::tmem_wait_st();
            }
            l = l * alpha + rs;
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.p_full[sb]);
        }
        // This warp's gate rows, requested now so their latency overlaps the
        // last P V product.
        if (ok && gated_out)
            load_gate();
        if (!ok) {
            if (lane == 0)
                set_abort(&sm.abort_flag, p.status);
        } else if (warp_wait(&sm.o_done[(n_tiles - 1) % NUM_S], ((n_tiles - 1) / NUM_S) & 1,
                             &sm.abort_flag)) {
            // ---------------------------------------------------- epilogue --
            // Each thread writes its O row (normalised unless this is a split
            // partial) into the idle K ring, rows padded by 16 bytes so the
            // row-per-thread writes are bank-conflict free; then each warp
            // stores its 32 rows one row per instruction, coalesced.
            tc::fence_after_sync();
            const float scale = split_out ? 1.0f : (l > 0.f ? 1.0f / l : 0.f);
            {
                uint32_t o[D / 32][32];  // the whole row in one round of loads
#pragma unroll
                for (int c = 0; c < D / 32; c++)
                    tc::tmem_ld32(o_t + c * 32, o[c]);
                tc::tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < D / 32; c++) {
                    float4 *row4 = reinterpret_cast<float4 *>(stage + r * LDS + c * 32);
#pragma unroll
                    for (int q = 0; q < 8; q++)
                        row4[q] = make_float4(__uint_as_float(o[c][4 * q]) * scale,
                                              __uint_as_float(o[c][4 * q + 1]) * scale,
                                              __uint_as_float(o[c][4 * q + 2]) * scale,
                                              __uint_as_float(o[c][4 * q + 3]) * scale);
                }
            }
            if (split_out && r < rows) {
                p.part_ml[(piece_row0 + r) * 2] = m_ref;
                p.part_ml[(piece_row0 + r) * 2 + 1] = l;
            }
        } else if (lane == 0) {
            set_abort(&sm.abort_flag, p.status);
        }
    }

    tc::fence_before_sync();
    __syncthreads();  // the staged rows are complete (unless a wait gave up)
    if (!aborted(&sm.abort_flag)) {
        // Lanes across a row, one row per step, this warp's SR rows.
#pragma unroll
        for (int i = 0; i < SR; i++) {
            const int rr = warp * SR + i;
            if (rr >= rows)
                break;
            const float *src = stage + rr * LDS + lane * EPL;
            float v[EPL];
            if constexpr (EPL == 4) {
                const float4 x = *reinterpret_cast<const float4 *>(src);
                v[0] = x.x;
                v[1] = x.y;
                v[2] = x.z;
                v[3] = x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2 *>(src);
                v[0] = x.x;
                v[1] = x.y;
            }
            if (split_out) {
                float *dst = p.part_o + (piece_row0 + rr) * D + lane * EPL;
                if constexpr (EPL == 4)
                    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                else
                    *reinterpret_cast<float2 *>(dst) = make_float2(v[0], v[1]);
                continue;
            }
            if (gated_out) {
#pragma unroll
                for (int e = 0; e < EPL; e += 2) {
                    const float g0 = __uint_as_float(gq[i][e / 2] << 16);
                    const float g1 = __uint_as_float(gq[i][e / 2] & 0xffff0000u);
                    v[e] *= __fdividef(1.0f, 1.0f + __expf(-g0));
                    v[e + 1] *= __fdividef(1.0f, 1.0f + __expf(-g1));
                }
            }
            uint32_t pk[EPL / 2];
#pragma unroll
            for (int e = 0; e < EPL; e += 2)
                pk[e / 2] = pack_bf16x2(v[e], v[e + 1]);
            const size_t tok = (size_t)(tok0 + r0 + (rr >> pack_shift));
            const int h = h0 + (rr & (p.pack - 1));
            const size_t off = (tok * p.H + h) * D + lane * EPL;
            if constexpr (EPL == 4)
                *reinterpret_cast<uint2 *>(p.out + off) = make_uint2(pk[0], pk[1]);
            else
                *reinterpret_cast<uint32_t *>(p.out + off) = pk[0];
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// The sequence that grid slot `slot` serves, and its bounds: with 2 to 32
// sequences the slots go to sequences in order of decreasing end position
// (prior + new tokens), as in the attention pass; otherwise slot b is
// sequence b.  Called by a full warp; every lane gets the same values.
__device__ __forceinline__ void slot_sequence(const PrefillParams &p, int slot, int lane, int &b,
                                              int &tok0, int &n_new, int &prior)
{
    if (p.batch > 1 && p.batch <= 32) {
        int c0 = 0, c1 = 0, pl = 0, key = -1;
        if (lane < p.batch) {
            c0 = __ldg(p.cu_seqlens + lane);
            c1 = __ldg(p.cu_seqlens + lane + 1);
            pl = __ldg(p.cache_lens + lane);
            key = pl + (c1 - c0);
        }
        int rank = 0;
        for (int j = 0; j < p.batch; j++) {
            const int kj = __shfl_sync(0xffffffffu, key, j);
            rank += (kj > key) || (kj == key && j < lane);
        }
        const unsigned m = __ballot_sync(0xffffffffu, lane < p.batch && rank == slot);
        const int src = __ffs(m) - 1;
        b = src;
        tok0 = __shfl_sync(0xffffffffu, c0, src);
        n_new = __shfl_sync(0xffffffffu, c1, src) - tok0;
        prior = __shfl_sync(0xffffffffu, pl, src);
        return;
    }
    b = slot;
    tok0 = __ldg(p.cu_seqlens + b);
    n_new = __ldg(p.cu_seqlens + b + 1) - tok0;
    prior = __ldg(p.cache_lens + b);
}

// Merge pass of the cut (tail) units: CTA (u, g) merges rows 8 g .. 8 g + 7
// of tail unit u, one warp per row.  Lane s loads piece s's (max, sum) (one
// round), the row's M and L come from warp reductions, then each lane loads
// its D/32 output elements of every piece's row, four pieces in flight at a
// time, weights them by 2^(m_s - M) in piece order, normalises and gates.
constexpr int kMergeRows = 8;

template <int D>
__global__ void __launch_bounds__(256) prefill_combine_kernel(const PrefillParams p)
{
    constexpr int EPL = D / 32;  // output elements per lane
    grid_dependency_wait();
    grid_dependents_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned FULL = 0xffffffffu;
    const int tu = blockIdx.x;
    const int r = blockIdx.y * kMergeRows + warp;            // the warp's row of the unit
    const size_t row0 = (size_t)tu * p.num_splits * BM + r;  // piece s at row0 + s BM
    // The pieces' (max, sum) (lane s: piece s) and rows of the first four
    // pieces are requested at once, in parallel with the sequence bounds: one
    // round trip instead of three dependent ones.  Pieces past the row's last
    // one are read but never used (their slots hold other calls' rows).
    const float2 *ml = reinterpret_cast<const float2 *>(p.part_ml);
    float2 ml_pre = make_float2(-INFINITY, 0.f);
    if (lane < p.num_splits)
        ml_pre = ml[row0 + (size_t)lane * BM];
    auto load_row = [&](int s, float (&v)[EPL]) {
        const float *src = p.part_o + (row0 + (size_t)s * BM) * D + lane * EPL;
        if constexpr (EPL == 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src);
            v[0] = x.x;
            v[1] = x.y;
            v[2] = x.z;
            v[3] = x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2 *>(src);
            v[0] = x.x;
            v[1] = x.y;
        }
    };
    float pre[4][EPL];
#pragma unroll
    for (int u = 0; u < 4; u++)
        if (u < p.num_splits)
            load_row(u, pre[u]);
    const int unit = p.full_units + tu;
    const int hg = (unit / p.q_tiles) % p.HG;
    const int slot = unit / (p.q_tiles * p.HG);
    const int qt = p.q_tiles - 1 - (unit % p.q_tiles);
    int b, tok0, n_new, prior;
    slot_sequence(p, slot, lane, b, tok0, n_new, prior);
    const int r0 = qt * p.tile_tokens;
    const bool ring = (p.flags & NA_RING_CACHE) != 0;
    if (n_new > p.max_new_len || (b == 0 && tok0 != 0) || tok0 < 0 ||
        (long long)tok0 + n_new > p.total_tokens || r0 >= n_new)
        return;  // invalid bounds were reported by the attention pass
    const int rows_tok = min(p.tile_tokens, n_new - r0);
    const int pos_lo = prior + r0, pos_hi = pos_lo + rows_tok - 1;
    if (prior < 0 || (!ring && pos_hi >= p.capacity) || pos_hi >= p.max_total_len)
        return;
    const int pack_shift = __ffs(p.pack) - 1;
    if (r >= (rows_tok << pack_shift))
        return;
    const size_t out_row = (size_t)(tok0 + r0 + (r >> pack_shift)) * p.H + hg * p.pack +
                           (r & (p.pack - 1));
    uint32_t gw[EPL / 2];  // gate words, requested before the merge arithmetic
    const bool gated = (p.flags & NA_OUT_GATE) && p.gate;
    if (gated) {
        const bf16 *gt = p.gate + out_row * D + lane * EPL;
        if constexpr (EPL == 4) {
            const uint2 u = __ldg(reinterpret_cast<const uint2 *>(gt));
            gw[0] = u.x;
            gw[1] = u.y;
        } else {
            gw[0] = __ldg(reinterpret_cast<const unsigned int *>(gt));
        }
    }
    // pieces with keys: the splits start at the key tile holding the first
    // row's window start (0 without a window), split_len keys apart
    const int win_tile = p.window > 0 ? max(0, pos_lo - p.window + 1) / BN * BN : 0;
    const int ns = min(p.num_splits, (pos_hi - win_tile) / p.split_len + 1);
    float M = -INFINITY;
    for (int s0 = 0; s0 < ns; s0 += 32)
        if (s0 + lane < ns)
            M = fmaxf(M, s0 == 0 ? ml_pre.x : ml[row0 + (size_t)(s0 + lane) * BM].x);
#pragma unroll
    for (int o = 16; o; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; e++)
        acc[e] = 0.f;
    float L = 0.f;
    for (int s0 = 0; s0 < ns; s0 += 32) {
        float w = 0.f;  // this lane's piece weight 2^(m - M)
        if (s0 + lane < ns) {
            const float2 v = s0 == 0 ? ml_pre : ml[row0 + (size_t)(s0 + lane) * BM];
            if (v.x != -INFINITY) {
                w = exp2f(v.x - M);
                L = fmaf(v.y, w, L);
            }
        }
        const int n = min(32, ns - s0);
        for (int s = 0; s < n; s += 4) {
            float v[4][EPL];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                if (s0 + s == 0) {
#pragma unroll
                    for (int e = 0; e < EPL; e++)
                        v[u][e] = pre[u][e];
                } else if (s + u < n) {
                    load_row(s0 + s + u, v[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const float ws = __shfl_sync(FULL, w, min(s + u, n - 1));
                if (s + u < n) {
#pragma unroll
                    for (int e = 0; e < EPL; e++)
                        acc[e] = fmaf(v[u][e], ws, acc[e]);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1)
        L += __shfl_xor_sync(FULL, L, o);
    const float inv = L > 0.f ? 1.0f / L : 0.f;
    bf16 *dst = p.out + out_row * D + lane * EPL;
    float g[EPL];
#pragma unroll
    for (int e = 0; e < EPL; e++)
        g[e] = 1.0f;
    if (gated) {
#pragma unroll
        for (int e = 0; e < EPL; e += 2) {
            g[e] = __fdividef(1.0f, 1.0f + __expf(-__uint_as_float(gw[e / 2] << 16)));
            g[e + 1] = __fdividef(1.0f, 1.0f + __expf(-__uint_as_float(gw[e / 2] & 0xffff0000u)));
        }
    }
    uint32_t packed[EPL / 2];
#pragma unroll
    for (int e = 0; e < EPL; e += 2)
        packed[e / 2] = pack_bf16x2(acc[e] * inv * g[e], acc[e + 1] * inv * g[e + 1]);
    if constexpr (EPL == 4)
        *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
    else
        *reinterpret_cast<uint32_t *>(dst) = packed[0];
}

template <int D>
cudaError_t launch_prefill_t(const PrefillParams &p, int total_tokens, int cache_batch,
                             cudaStream_t stream)
{
    CUtensorMap mq, mk, mv;
    {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.H, (cuuint64_t)total_tokens};
        const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.H * D * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)p.pack, (cuuint32_t)p.tile_tokens};
        if (!make_bf16_tile_map(&mq, p.q, 3, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t rows = (cuuint64_t)cache_batch * p.KV * p.capacity;
        const cuuint64_t dims[2] = {(cuuint64_t)D, rows};
        const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
        const cuuint32_t box[2] = {64, BN};
        if (!make_bf16_tile_map(&mk, p.cache_k, 2, dims, strides, box) ||
            !make_bf16_tile_map(&mv, p.cache_v, 2, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    const size_t smem = tc_smem_bytes<D>();
    static std::atomic<unsigned long long> configured{0};
    cudaError_t e = once_per_device(configured, [smem] {
        cudaError_t r = cudaFuncSetAttribute(prefill_tc_kernel<D, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(prefill_tc_kernel<D, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        return r;
    });
    if (e != cudaSuccess)
        return e;
    const dim3 grid(p.full_units + p.tail_units * p.num_splits);
    e = p.softcap > 0.f ? launch_kernel(prefill_tc_kernel<D, true>, grid, dim3(THREADS), smem,
                                        stream, p, mq, mk, mv)
                        : launch_kernel(prefill_tc_kernel<D, false>, grid, dim3(THREADS), smem,
                                        stream, p, mq, mk, mv);
    if (e != cudaSuccess || p.num_splits == 1)
        return e;
    return launch_kernel(prefill_combine_kernel<D>, dim3(p.tail_units, BM / kMergeRows), dim3(256),
                         0, stream, p);
}

}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
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

// bf16 tensor map with 64-element (128-byte) inner boxes and 128-byte swizzle.
bool make_bf16_tile_map(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
              const cuuint64_t *strides_bytes, const cuuint32_t *box)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base),
              dims, strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int prefill_key_tile() { return BN; }
int prefill_q_tile() { return BM; }

cudaError_t launch_prefill(const PrefillParams &p, int d, int total_tokens, int cache_batch,
                           cudaStream_t stream)
{
    if (d == 128)
        return launch_prefill_t<128>(p, total_tokens, cache_batch, stream);
    return launch_prefill_t<64>(p, total_tokens, cache_batch, stream);
}

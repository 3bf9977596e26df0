// prefill.cu -- causal GQA attention of a chunk of new tokens against the
// per-sequence KV cache (cortiq-engine src/attention.rs, fn
// qwen_attention_batch: query bi of a chunk sees keys 0 .. s0 + bi, i.e. all
// history and the earlier keys of its own chunk; fn attention_head for the
// softmax(q.k * scale) . V of each row; fn apply_gate for the sigmoid gate).
//
// Flash-attention tiling: a CTA owns 64 query rows of one (sequence, query
// head) and walks the key tiles of kv head h / (H / KV) that its rows can see,
// with an online softmax in fp32 (log2 domain).  Key tiles wholly above the
// diagonal are never loaded; only tiles that straddle it are masked.  When a
// launch would leave SMs idle (short chunks), the keys are split across CTAs
// and a combine pass merges the partial (max, sum, output) triples.
#include "na_internal.cuh"

namespace {

constexpr int BM = 64;       // query rows per CTA
constexpr int BN = 64;       // keys per tile
constexpr int THREADS = 128; // 4 warps x 16 rows

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_addr(p)));
}
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Element offset of 16-byte chunk `c` of row `r` in a swizzled [rows][D] tile.
template <int D>
__device__ __forceinline__ int swz(int r, int c)
{
    return r * D + ((c ^ (r & 7)) << 3);
}

template <int D>
__global__ void __launch_bounds__(THREADS, 2) prefill_kernel(const PrefillParams p)
{
    constexpr int CH = D / 8;  // 16-byte chunks per row
    extern __shared__ __align__(128) uint8_t smem_raw[];
    bf16 *sQ = reinterpret_cast<bf16 *>(smem_raw);
    bf16 *sK = sQ + BM * D;      // [2][BN][D]
    bf16 *sV = sK + 2 * BN * D;  // [2][BN][D]

    const int qt = blockIdx.x, h = blockIdx.y;
    const int b = blockIdx.z / p.num_splits, split = blockIdx.z - b * p.num_splits;
    const int tok0 = __ldg(p.cu_seqlens + b);
    const int n_new = __ldg(p.cu_seqlens + b + 1) - tok0;
    const int r0 = qt * BM;
    if (n_new > p.max_new_len) {
        if (qt == 0 && h == 0 && threadIdx.x == 0)
            na_report(p.status, NA_ERR_INVALID_ARG);
        return;
    }
    if (r0 >= n_new)
        return;
    const int prior = __ldg(p.cache_lens + b);
    const int rows = min(BM, n_new - r0);
    const int pos_lo = prior + r0, pos_hi = prior + r0 + rows - 1;
    if (prior < 0 || pos_hi >= p.capacity || pos_hi >= p.max_total_len) {
        if (threadIdx.x == 0)
            na_report(p.status, NA_ERR_CAPACITY);
        return;
    }
    int k_begin = 0, k_end = pos_hi + 1;
    if (p.num_splits > 1) {
        k_begin = split * p.split_len;
        k_end = min(k_end, k_begin + p.split_len);
    }
    if (k_begin >= k_end)
        return;

    const int kvh = h / p.group;
    const size_t cap = (size_t)p.capacity;
    const bf16 *kbase = p.cache_k + ((size_t)b * p.KV + kvh) * cap * D;
    const bf16 *vbase = p.cache_v + ((size_t)b * p.KV + kvh) * cap * D;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Q tile (rows past the chunk are zero-filled).
    for (int c = tid; c < BM * CH; c += THREADS) {
        const int r = c / CH, ch = c - r * CH;
        const bool valid = r < rows;
        const bf16 *src = p.q + ((size_t)(tok0 + r0 + (valid ? r : 0)) * p.H + h) * D + ch * 8;
        cp_async16(sQ + swz<D>(r, ch), src, valid);
    }
    auto load_kv = [&](int tile, int buf) {
        const int j0 = tile * BN;
        for (int c = tid; c < BN * CH; c += THREADS) {
            const int r = c / CH, ch = c - r * CH;
            const int j = j0 + r;
            const bool valid = j < k_end;
            const size_t off = (size_t)(valid ? j : 0) * D + ch * 8;
            cp_async16(sK + buf * BN * D + swz<D>(r, ch), kbase + off, valid);
            cp_async16(sV + buf * BN * D + swz<D>(r, ch), vbase + off, valid);
        }
    };
    const int t_first = k_begin / BN, t_last = (k_end - 1) / BN;
    load_kv(t_first, 0);
    cp_async_commit();

    const int g = lane >> 2, tq = lane & 3;
    const int wrow = warp * 16;  // first row of this warp within the tile
    const int pos0 = pos_lo + wrow + g, pos1 = pos0 + 8;

    uint32_t qf[D / 16][4];
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; i++)
        o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int tile = t_first; tile <= t_last; tile++) {
        const int buf = (tile - t_first) & 1;
        if (tile < t_last) {
            load_kv(tile + 1, buf ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (tile == t_first) {
#pragma unroll
            for (int kk = 0; kk < D / 16; kk++) {
                const int r = wrow + (lane & 7) + ((lane >> 3) & 1) * 8;
                ldsm_x4(qf[kk], sQ + swz<D>(r, kk * 2 + (lane >> 4)));
            }
        }
        const bf16 *kt = sK + buf * BN * D;
        const bf16 *vt = sV + buf * BN * D;

        float s[BN / 8][4];
#pragma unroll
        for (int i = 0; i < BN / 8; i++)
            s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
#pragma unroll
            for (int np = 0; np < BN / 16; np++) {
                uint32_t bfr[4];
                const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
                ldsm_x4(bfr, kt + swz<D>(r, kk * 2 + ((lane >> 3) & 1)));
                mma_bf16_16816(s[2 * np], qf[kk], bfr[0], bfr[1]);
                mma_bf16_16816(s[2 * np + 1], qf[kk], bfr[2], bfr[3]);
            }
        }
        const int j0 = tile * BN;
        const bool need_mask = (j0 + BN - 1 > pos_lo) || (j0 + BN > k_end) || (j0 < k_begin);
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < BN / 8; nt++) {
#pragma unroll
            for (int e = 0; e < 2; e++) {
                float v0 = s[nt][e] * p.scale_log2, v1 = s[nt][2 + e] * p.scale_log2;
                if (need_mask) {
                    const int j = j0 + nt * 8 + 2 * tq + e;
                    const bool kin = j >= k_begin && j < k_end;
                    if (!kin || j > pos0)
                        v0 = -INFINITY;
                    if (!kin || j > pos1)
                        v1 = -INFINITY;
                }
                s[nt][e] = v0;
                s[nt][2 + e] = v1;
                mx0 = fmaxf(mx0, v0);
                mx1 = fmaxf(mx1, v1);
            }
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
        const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
        const float a0 = exp2f(m0 - ref0), a1 = exp2f(m1 - ref1);  // 0 when m was -inf
        m0 = mn0;
        m1 = mn1;
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < BN / 8; nt++) {
            s[nt][0] = exp2f(s[nt][0] - ref0);
            s[nt][1] = exp2f(s[nt][1] - ref0);
            s[nt][2] = exp2f(s[nt][2] - ref1);
            s[nt][3] = exp2f(s[nt][3] - ref1);
            rs0 += s[nt][0] + s[nt][1];
            rs1 += s[nt][2] + s[nt][3];
        }
        l0 = l0 * a0 + rs0;
        l1 = l1 * a1 + rs1;
#pragma unroll
        for (int i = 0; i < D / 8; i++) {
            o[i][0] *= a0;
            o[i][1] *= a0;
            o[i][2] *= a1;
            o[i][3] *= a1;
        }
#pragma unroll
        for (int kk = 0; kk < BN / 16; kk++) {
            uint32_t a[4];
            a[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
            a[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
            a[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            a[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int dp = 0; dp < D / 16; dp++) {
                uint32_t bfr[4];
                const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                ldsm_x4_t(bfr, vt + swz<D>(r, dp * 2 + (lane >> 4)));
                mma_bf16_16816(o[2 * dp], a, bfr[0], bfr[1]);
                mma_bf16_16816(o[2 * dp + 1], a, bfr[2], bfr[3]);
            }
        }
        __syncthreads();
    }

    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

    const int rr0 = wrow + g, rr1 = rr0 + 8;  // rows within the tile
#pragma unroll
    for (int half = 0; half < 2; half++) {
        const int rr = half ? rr1 : rr0;
        if (rr >= rows)
            continue;
        const size_t t = (size_t)(tok0 + r0 + rr);
        const float l = half ? l1 : l0;
        const float m = half ? m1 : m0;
        if (p.num_splits == 1) {
            const float inv = 1.0f / l;
            bf16 *dst = p.out + (t * p.H + h) * D;
            const bf16 *gt = ((p.flags & NA_OUT_GATE) && p.gate) ? p.gate + (t * p.H + h) * D : nullptr;
#pragma unroll
            for (int nt = 0; nt < D / 8; nt++) {
                const int col = nt * 8 + 2 * tq;
                float x0 = o[nt][2 * half] * inv, x1 = o[nt][2 * half + 1] * inv;
                if (gt) {
                    const __nv_bfloat162 gg = *reinterpret_cast<const __nv_bfloat162 *>(gt + col);
                    x0 *= 1.0f / (1.0f + __expf(-__bfloat162float(gg.x)));
                    x1 *= 1.0f / (1.0f + __expf(-__bfloat162float(gg.y)));
                }
                *reinterpret_cast<uint32_t *>(dst + col) = pack_bf16x2(x0, x1);
            }
        } else {
            const size_t row = (t * p.H + h) * p.num_splits + split;
            float *dst = p.part_o + row * D;
#pragma unroll
            for (int nt = 0; nt < D / 8; nt++) {
                const int col = nt * 8 + 2 * tq;
                *reinterpret_cast<float2 *>(dst + col) =
                    make_float2(o[nt][2 * half], o[nt][2 * half + 1]);
            }
            if (tq == 0) {
                p.part_ml[row * 2] = m;
                p.part_ml[row * 2 + 1] = l;
            }
        }
    }
}

// Merge the KV splits of each (token, head) row: one warp per row.
template <int D>
__global__ void __launch_bounds__(256) prefill_combine_kernel(const PrefillParams p, int total_tokens)
{
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= total_tokens * p.H)
        return;
    const int t = row / p.H;
    int lo = 0, hi = p.batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.cu_seqlens + mid) <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int pos = __ldg(p.cache_lens + lo) + (t - __ldg(p.cu_seqlens + lo));
    if (pos < 0 || pos >= p.capacity)
        return;  // reported by the split pass
    const int ns = min(p.num_splits, pos / p.split_len + 1);
    const float *ml = p.part_ml + (size_t)row * p.num_splits * 2;
    float M = -INFINITY;
    for (int s = 0; s < ns; s++)
        M = fmaxf(M, ml[2 * s]);
    float L = 0.f;
    for (int s = 0; s < ns; s++)
        L += ml[2 * s + 1] * exp2f(ml[2 * s] - M);
    const float inv = 1.0f / L;
    const float *po = p.part_o + (size_t)row * p.num_splits * D;
    bf16 *dst = p.out + (size_t)row * D;
    const bf16 *gt = ((p.flags & NA_OUT_GATE) && p.gate) ? p.gate + (size_t)row * D : nullptr;
    for (int e = lane; e < D; e += 32) {
        float o = 0.f;
        for (int s = 0; s < ns; s++)
            o += po[(size_t)s * D + e] * exp2f(ml[2 * s] - M);
        o *= inv;
        if (gt)
            o *= 1.0f / (1.0f + __expf(-__bfloat162float(gt[e])));
        dst[e] = __float2bfloat16_rn(o);
    }
}

template <int D>
cudaError_t launch_prefill_t(const PrefillParams &p, int total_tokens, cudaStream_t stream)
{
    const size_t smem = (size_t)(BM + 4 * BN) * D * sizeof(bf16);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        configured = true;
    }
    dim3 grid(p.q_tiles, p.H, p.batch * p.num_splits);
    prefill_kernel<D><<<grid, THREADS, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.num_splits == 1)
        return e;
    const int rows = total_tokens * p.H;
    prefill_combine_kernel<D><<<(rows + 7) / 8, 256, 0, stream>>>(p, total_tokens);
    return cudaGetLastError();
}

}  // namespace

int prefill_key_tile() { return BN; }
int prefill_q_tile() { return BM; }

cudaError_t launch_prefill(const PrefillParams &p, int d, int total_tokens, cudaStream_t stream)
{
    if (d == 128)
        return launch_prefill_t<128>(p, total_tokens, stream);
    return launch_prefill_t<64>(p, total_tokens, stream);
}

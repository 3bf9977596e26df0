/*
 * na_oracle.c -- reference oracle for RoPE-rotated causal GQA attention over a
 * per-sequence KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU statement of what the GPU library computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or constant with the CUDA library, and the CUDA library
 * never calls it.
 *
 * Arithmetic: IEEE double throughout, one thread, no SIMD, no reordering
 * beyond the loops written here.  Inputs that the GPU path reads as bf16 are
 * handed in as doubles holding exactly those bf16 values.
 *
 * Sources (docs.rs source pages; "cortiq" = cortiq-engine 0.5.39
 * src/attention.rs, "needle" = needle-core 0.3.1 src/v2/batch.rs):
 *   - RoPE inverse frequencies:       cortiq, fn rope_inv_freq
 *   - YaRN inverse frequencies:       cortiq, fn yarn_inv_freq
 *   - half-split rotation with scale: cortiq, fn rope_rotate_scaled
 *   - partial rotary:                 cortiq, fn finish_projection ("Partial RoPE")
 *   - per-head qk RMSNorm (2 styles): cortiq, fn rmsnorm_head
 *   - scale-less V-norm:              cortiq, fn vnorm_head
 *   - append-before-attend, causal:   needle, module doc "What has to stay
 *                                     sequential"; cortiq, fn qwen_attention_batch
 *                                     (portable batched attend, lim = s0 + bi + 1)
 *   - softmax(q.k * scale) . V:       cortiq, fn attention_head
 *   - GQA head mapping kv = h/(H/KV): needle, fn batch_attention; cortiq,
 *                                     fn attend_all_heads
 *   - sigmoid output gate:            cortiq, fn apply_gate
 *   - decode with per-key probs:      cortiq, fn attention_head (returned probs),
 *                                     fn qwen_attention_core (append then attend)
 *   - ring cache (slot = pos mod cap): needle, fn batch_attention (the
 *                                     per-position write-and-attend loop over a
 *                                     ring of kv_window positions)
 *
 * Readings where the pages leave a choice (each one is listed with its reason
 * in the design notes of this repository):
 *   - inverse frequencies, angles, sin and cos are taken in double (the pages
 *     use f32; the mathematical definition has no rounding);
 *   - the exponent denominator of the frequencies is the rotary dimension;
 *   - the attention output skips no small probability (the pages skip |p| <
 *     1e-12 in one CPU loop; the definition sums every key);
 *   - an empty key set gives a zero output and writes no probabilities.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#define ORACLE_PI 3.14159265358979323846

/* Flag bits of the attention configuration (same meaning as the library's). */
#define ORACLE_QK_NORM 1
#define ORACLE_QK_NORM_ZERO_CENTERED 2
#define ORACLE_V_NORM 4
#define ORACLE_OUT_GATE 8
#define ORACLE_RING_CACHE 16

/* ---------------------------------------------------------------- RoPE --- */

/* cortiq fn rope_inv_freq: inv_freq[i] = 1 / base^(2 i / rd), i < rd/2. */
void oracle_rope_inv_freq(int rd, double base, double *inv_freq)
{
    for (int i = 0; i < rd / 2; i++)
        inv_freq[i] = 1.0 / pow(base, 2.0 * (double)i / (double)rd);
}

/* cortiq fn yarn_inv_freq, inner closure correction_dim: the dimension index
 * at which the wavelength equals orig/rotations full turns. */
static double yarn_correction_dim(int rd, double base, int orig_max_pos, double rotations)
{
    return ((double)rd * log((double)orig_max_pos / (rotations * 2.0 * ORACLE_PI)))
           / (2.0 * log(base));
}

/* cortiq fn yarn_inv_freq: frequencies below `low` keep the original value
 * (extrapolation), above `high` are divided by `factor` (interpolation), and a
 * linear ramp in the index mixes the two in between.  `rd` is the rotary
 * dimension.  Writes rd/2 values; also returns low and high if asked. */
void oracle_yarn_inv_freq(int rd, double base, double factor, int orig_max_pos,
                          double beta_fast, double beta_slow, double *inv_freq,
                          int *low_out, int *high_out)
{
    int half = rd / 2;
    double lo = floor(yarn_correction_dim(rd, base, orig_max_pos, beta_fast));
    if (lo < 0.0)
        lo = 0.0;
    double hi = ceil(yarn_correction_dim(rd, base, orig_max_pos, beta_slow));
    double hi_cap = (double)(half > 0 ? half - 1 : 0);
    if (hi < 0.0)
        hi = 0.0;
    if (hi > hi_cap)
        hi = hi_cap;
    int low = (int)lo, high = (int)hi;
    int span = high > low ? high - low : 0; /* saturating subtraction */
    double denom = (double)(span > 1 ? span : 1);
    for (int i = 0; i < half; i++) {
        double extrap = 1.0 / pow(base, 2.0 * (double)i / (double)rd);
        double interp = extrap / factor;
        int num = i > low ? i - low : 0; /* saturating subtraction */
        double ramp = (double)num / denom;
        if (ramp < 0.0)
            ramp = 0.0;
        if (ramp > 1.0)
            ramp = 1.0;
        double extrapolation = 1.0 - ramp;
        inv_freq[i] = interp * (1.0 - extrapolation) + extrap * extrapolation;
    }
    if (low_out)
        *low_out = low;
    if (high_out)
        *high_out = high;
}

/* Attention factor multiplied onto cos and sin.  A positive value is used as
 * given.  Otherwise: 1 without YaRN; with YaRN the YaRN paper's
 * 0.1 ln(factor) + 1 (the pages carry the multiplier, cortiq field rope_scale,
 * but do not print its formula). */
double oracle_rope_attn_factor(int yarn, double factor, double attn_factor)
{
    if (attn_factor > 0.0)
        return attn_factor;
    if (yarn && factor > 1.0)
        return 0.1 * log(factor) + 1.0;
    return 1.0;
}

/* cortiq fn rope_rotate_scaled: half-split pairs (x[i], x[i + rd/2]) turned
 * by angle pos * inv_freq[i]; both outputs multiplied by `scale`.  Dimensions
 * at and above rd are left alone (partial rotary). */
void oracle_rope_rotate(double *x, int rd, int64_t pos, const double *inv_freq, double scale)
{
    int half = rd / 2;
    for (int i = 0; i < half; i++) {
        double angle = (double)pos * inv_freq[i];
        double c = cos(angle), s = sin(angle);
        double x0 = x[i], x1 = x[i + half];
        x[i] = (x0 * c - x1 * s) * scale;
        x[i + half] = (x0 * s + x1 * c) * scale;
    }
}

/* ------------------------------------------------------------- norms --- */

/* cortiq fn rmsnorm_head: x <- x / sqrt(mean(x^2) + eps) * w   (Qwen style)
 *                      or x <- x / sqrt(mean(x^2) + eps) * (1 + w) (zero-centred). */
void oracle_rmsnorm_head(double *x, const double *w, int d, double eps, int zero_centered)
{
    double ss = 0.0;
    for (int i = 0; i < d; i++)
        ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)d + eps);
    for (int i = 0; i < d; i++)
        x[i] = x[i] * inv * (zero_centered ? 1.0 + w[i] : w[i]);
}

/* cortiq fn vnorm_head: x <- x / sqrt(mean(x^2) + eps), no weight. */
void oracle_vnorm_head(double *x, int d, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < d; i++)
        ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss / (double)d + eps);
    for (int i = 0; i < d; i++)
        x[i] *= inv;
}

/* ------------------------------------------------- rope + cache append --- */

/* Which packed sequence owns token t (cu_seqlens is non-decreasing). */
static int owner_of(int batch, const int *cu_seqlens, int t)
{
    for (int b = 0; b < batch; b++)
        if (t >= cu_seqlens[b] && t < cu_seqlens[b + 1])
            return b;
    return -1;
}

static size_t cache_index(int b, int kvh, int slot, int KV, int capacity, int d)
{
    return (((size_t)b * KV + kvh) * (size_t)capacity + (size_t)slot) * (size_t)d;
}

/* Ring cache (needle fn batch_attention: the cache of a windowed layer is a
 * ring that each new position overwrites in turn): position pos lives in slot
 * pos mod capacity, so the ring holds the newest `capacity` positions. */
int oracle_ring_slot(int64_t pos, int capacity)
{
    return (int)(pos % (int64_t)capacity);
}

/* Slot of position pos: the position itself, or its ring slot. */
static int slot_of(int flags, int64_t pos, int capacity)
{
    return (flags & ORACLE_RING_CACHE) ? oracle_ring_slot(pos, capacity) : (int)pos;
}

/* Per new token (cortiq fn finish_projection, then cache append):
 *   pos = cache_lens[b] + (t - cu_seqlens[b]);
 *   q, k: optional per-head RMSNorm, then RoPE on the first rd dims;
 *   v: optional scale-less V-norm;
 *   q_out[t] <- q;  cache_k[b][kvh][slot] <- k;  cache_v[b][kvh][slot] <- v,
 * slot = pos, or pos mod capacity with a ring cache (ORACLE_RING_CACHE).
 * Tensors: q, q_out [T][H][d]; k, v [T][KV][d]; caches [B][KV][capacity][d].
 * Returns 0, or -1 when a position does not fit a linear cache (nothing past
 * that token is written). */
int oracle_rope_append(int H, int KV, int d, int rd, int flags, double eps,
                       const double *inv_freq, double rope_scale, int batch,
                       const int *cu_seqlens, const int *cache_lens, const double *q,
                       const double *k, const double *v, const double *q_norm_w,
                       const double *k_norm_w, double *q_out, double *cache_k,
                       double *cache_v, int capacity)
{
    int zc = (flags & ORACLE_QK_NORM_ZERO_CENTERED) != 0;
    for (int b = 0; b < batch; b++) {
        for (int t = cu_seqlens[b]; t < cu_seqlens[b + 1]; t++) {
            int pos = cache_lens[b] + (t - cu_seqlens[b]);
            if (pos < 0 || (!(flags & ORACLE_RING_CACHE) && pos >= capacity))
                return -1;
            int slot = slot_of(flags, pos, capacity);
            for (int h = 0; h < H; h++) {
                double *x = q_out + ((size_t)t * H + h) * d;
                for (int i = 0; i < d; i++)
                    x[i] = q[((size_t)t * H + h) * d + i];
                if (flags & ORACLE_QK_NORM)
                    oracle_rmsnorm_head(x, q_norm_w, d, eps, zc);
                oracle_rope_rotate(x, rd, pos, inv_freq, rope_scale);
            }
            for (int g = 0; g < KV; g++) {
                double *kx = cache_k + cache_index(b, g, slot, KV, capacity, d);
                double *vx = cache_v + cache_index(b, g, slot, KV, capacity, d);
                for (int i = 0; i < d; i++) {
                    kx[i] = k[((size_t)t * KV + g) * d + i];
                    vx[i] = v[((size_t)t * KV + g) * d + i];
                }
                if (flags & ORACLE_QK_NORM)
                    oracle_rmsnorm_head(kx, k_norm_w, d, eps, zc);
                oracle_rope_rotate(kx, rd, pos, inv_freq, rope_scale);
                if (flags & ORACLE_V_NORM)
                    oracle_vnorm_head(vx, d, eps);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------ attend --- */

/* cortiq fn attention_head, one query against keys [first, n) of one KV head:
 *   s_j = scale * q.k_j, replaced by c * tanh(s_j / c) when softcap c > 0
 *   (QwenAttnCfg.softcap, the Gemma-2 soft cap on attention logits, applied
 *   ahead of the softmax);  p_j = exp(s_j - max s) / sum;  o = sum_j p_j v_j.
 * Keys before `first` are outside a sliding window (QwenAttnCfg.window, fn
 * attend_all_heads: first = stored - window) and get probability 0.
 * Key j is read from slot j, or j mod capacity with a ring cache.
 * `scores` is scratch of length n; when `probs` is non-NULL it receives p_j
 * for j < n.  n == 0 leaves o at zero and writes no probabilities. */
static void attend_one(const double *q, const double *keys, const double *vals, int n, int first,
                       int d, double scale, double softcap, int flags, int capacity,
                       double *scores, double *o, double *probs)
{
    for (int i = 0; i < d; i++)
        o[i] = 0.0;
    if (n <= 0)
        return;
    if (first < 0)
        first = 0;
    double m = -INFINITY;
    for (int j = first; j < n; j++) {
        size_t kj = (size_t)slot_of(flags, j, capacity) * (size_t)d;
        double s = 0.0;
        for (int i = 0; i < d; i++)
            s += q[i] * keys[kj + i];
        s *= scale;
        if (softcap > 0.0)
            s = softcap * tanh(s / softcap);
        scores[j] = s;
        if (scores[j] > m)
            m = scores[j];
    }
    double sum = 0.0;
    for (int j = first; j < n; j++) {
        scores[j] = exp(scores[j] - m);
        sum += scores[j];
    }
    if (probs)
        for (int j = 0; j < first; j++)
            probs[j] = 0.0;
    for (int j = first; j < n; j++) {
        double p = scores[j] / sum;
        if (probs)
            probs[j] = p;
        size_t vj = (size_t)slot_of(flags, j, capacity) * (size_t)d;
        for (int i = 0; i < d; i++)
            o[i] += p * vals[vj + i];
    }
}

/* Grow the score scratch to at least n entries (a ring's positions may run
 * past its capacity).  Returns 0, or -1 when out of memory. */
static int grow_scores(double **scores, size_t *size, int n)
{
    if ((size_t)n <= *size)
        return 0;
    double *p = (double *)realloc(*scores, sizeof(double) * (size_t)n);
    if (!p)
        return -1;
    *scores = p;
    *size = (size_t)n;
    return 0;
}

/* cortiq fn apply_gate: o <- o * sigmoid(g). */
static void apply_gate(double *o, const double *g, int d)
{
    for (int i = 0; i < d; i++)
        o[i] *= 1.0 / (1.0 + exp(-g[i]));
}

/* Causal chunked prefill attention (needle "What has to stay sequential";
 * cortiq fn qwen_attention_batch, portable attend): the chunk's keys are
 * already in the cache; new token t of sequence b sits at
 * pos = cache_lens[b] + (t - cu_seqlens[b]) and attends keys 0..pos
 * inclusive of its own KV head kvh = h / (H / KV) -- only the last `window`
 * of them when window > 0 -- with scores soft-capped when softcap > 0.
 * Computed for the listed token indices only: out[r][h][d] for rows[r].
 * With a ring cache (ORACLE_RING_CACHE, window > 0) the whole chunk is in the
 * ring before any row attends, so a row's window must not reach a slot that a
 * later token of its chunk overwrote: capacity >= window + (last new position
 * of the sequence - pos).
 * Returns 0, or -1 on a bad row, a position past a linear cache's capacity or
 * a ring too small for the row's window. */
int oracle_attend_rows(int H, int KV, int d, double scale, int flags, int batch,
                       const int *cu_seqlens, const int *cache_lens, const double *q_rot,
                       const double *cache_k, const double *cache_v, int capacity,
                       const double *gate, int nrows, const int *rows, double *out,
                       double softcap, int window)
{
    int group = H / KV;
    double *scores = NULL;
    size_t scores_size = 0;
    for (int r = 0; r < nrows; r++) {
        int t = rows[r];
        int b = owner_of(batch, cu_seqlens, t);
        if (b < 0) {
            free(scores);
            return -1;
        }
        int pos = cache_lens[b] + (t - cu_seqlens[b]);
        int bad = pos < 0;
        if (flags & ORACLE_RING_CACHE) {
            int last = cache_lens[b] + (cu_seqlens[b + 1] - cu_seqlens[b]) - 1;
            bad |= window <= 0 || (int64_t)capacity < (int64_t)window + (last - pos);
        } else {
            bad |= pos >= capacity;
        }
        if (bad || grow_scores(&scores, &scores_size, pos + 1) != 0) {
            free(scores);
            return -1;
        }
        for (int h = 0; h < H; h++) {
            int kvh = h / group;
            const double *qv = q_rot + ((size_t)t * H + h) * d;
            double *o = out + ((size_t)r * H + h) * d;
            attend_one(qv, cache_k + cache_index(b, kvh, 0, KV, capacity, d),
                       cache_v + cache_index(b, kvh, 0, KV, capacity, d), pos + 1,
                       window > 0 ? pos + 1 - window : 0, d, scale, softcap, flags, capacity,
                       scores, o, NULL);
            if ((flags & ORACLE_OUT_GATE) && gate)
                apply_gate(o, gate + ((size_t)t * H + h) * d, d);
        }
    }
    free(scores);
    return 0;
}

/* Single-token decode (cortiq fn qwen_attention_core: the current token is
 * appended first, then attends): query q[b][h] against keys [0, kv_lens[b])
 * of KV head h / (H / KV).  out [B][H][d]; probs [B][H][probs_stride] receives
 * the per-key probabilities when non-NULL.  Only the first `nrows` (b, h)
 * pairs listed in rows_bh (b * H + h) are computed when rows_bh is non-NULL;
 * otherwise all of them.  With window > 0 only the last `window` keys are
 * attended (the others get probability 0); softcap > 0 caps the scores.
 * With a ring cache (ORACLE_RING_CACHE) key j sits in slot j mod capacity and
 * the window must fit the ring (0 < window <= capacity).
 * Returns 0, or -1 when a length exceeds a linear cache's capacity or the
 * stride, or the window does not fit the ring. */
int oracle_decode(int H, int KV, int d, double scale, int flags, int batch, const double *q,
                  const double *cache_k, const double *cache_v, int capacity,
                  const int *kv_lens, const double *gate, double *out, double *probs,
                  int probs_stride, int nrows, const int *rows_bh, double softcap, int window)
{
    int group = H / KV;
    double *scores = NULL;
    size_t scores_size = 0;
    int count = rows_bh ? nrows : batch * H;
    for (int r = 0; r < count; r++) {
        int bh = rows_bh ? rows_bh[r] : r;
        int b = bh / H, h = bh % H;
        int n = kv_lens[b];
        int ring = (flags & ORACLE_RING_CACHE) != 0;
        if (n < 0 || (!ring && n > capacity) || (ring && (window <= 0 || window > capacity)) ||
            (probs && n > probs_stride) || grow_scores(&scores, &scores_size, n) != 0) {
            free(scores);
            return -1;
        }
        int kvh = h / group;
        double *o = out + ((size_t)b * H + h) * d;
        attend_one(q + ((size_t)b * H + h) * d, cache_k + cache_index(b, kvh, 0, KV, capacity, d),
                   cache_v + cache_index(b, kvh, 0, KV, capacity, d), n,
                   window > 0 ? n - window : 0, d, scale, softcap, flags, capacity, scores, o,
                   probs ? probs + ((size_t)b * H + h) * (size_t)probs_stride : NULL);
        if ((flags & ORACLE_OUT_GATE) && gate && n > 0)
            apply_gate(o, gate + ((size_t)b * H + h) * d, d);
    }
    free(scores);
    return 0;
}

/* Born-rule importance of one decode step (cortiq fn qwen_attention_core: each
 * head's probabilities are summed into `imp`, which cache.accumulate_imp adds
 * to the position's running importance; fn attend_all_heads returns the same
 * sum): imp[b][j] = sum over the H query heads of probs[b][h][j], for
 * j < kv_lens[b]; with accumulate the sum is added to what imp holds.  Keys
 * past kv_lens[b] are left untouched. */
void oracle_decode_importance(int H, int batch, const double *probs, int probs_stride,
                              const int *kv_lens, double *imp, int imp_stride, int accumulate)
{
    for (int b = 0; b < batch; b++) {
        int n = kv_lens[b];
        for (int j = 0; j < n; j++) {
            double s = 0.0;
            for (int h = 0; h < H; h++)
                s += probs[((size_t)b * H + h) * (size_t)probs_stride + j];
            double *dst = imp + (size_t)b * imp_stride + j;
            *dst = accumulate ? *dst + s : s;
        }
    }
}

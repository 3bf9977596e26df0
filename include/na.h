/*
 * na.h -- C ABI of the GB300 (sm_103a) library for RoPE-rotated causal
 * grouped-query attention over a per-sequence KV cache.
 *
 * The operation comes from two docs.rs source pages:
 *   [cortiq]  cortiq-engine 0.5.39 src/attention.rs
 *   [needle]  needle-core 0.3.1 src/v2/batch.rs
 *
 * Conventions shared by every entry point
 *   - bf16 means IEEE bfloat16 stored as 16-bit words, little-endian.
 *   - Token-packed tensors hold the new tokens of all sequences back to back
 *     (varlen packing): token t belongs to sequence b when
 *     cu_seqlens[b] <= t < cu_seqlens[b+1].
 *   - The KV cache is head-major, one slot per absolute position:
 *     k[b][kv_head][slot][head_dim] (same for v), slot = position
 *     (position % capacity with NA_RING_CACHE).
 *   - Every pointer argument is DEVICE memory unless its comment says HOST.
 *     Configuration structs are HOST memory and are read only during the call.
 *   - Ownership: the caller allocates and frees every buffer (including the
 *     workspace).  The library allocates no device memory, never synchronises
 *     the host with the device, and enqueues all work on `stream`
 *     (a cudaStream_t; NULL is the legacy default stream).
 *   - Threads: calls may come from several host threads at once, each with its
 *     own buffers, workspace and stream (na_attn_decode_static_ws excepted: its
 *     calls share one scratch array).  Work goes to the calling thread's current
 *     device, whose primary context the library makes current on that thread.
 *   - Errors: a negative na_status is returned when host-side validation fails;
 *     nothing is enqueued in that case.  Conditions only the device can see
 *     (a position past the cache capacity, an internal wait that timed out) are
 *     reported by writing a nonzero na_status value into *status (a device
 *     int32, may be NULL to skip reporting); the affected tile is skipped and the
 *     kernel returns normally.  The library never clears *status: the caller
 *     zeroes it and reads it when convenient.
 *   - Alignment: q, k, v, q_out, gate, out and the cache base pointers must be
 *     16-byte aligned, contiguous, with head_dim a multiple of 8.
 */
#ifndef NA_H
#define NA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum na_status {
    NA_OK = 0,
    NA_ERR_INVALID_ARG = -1,   /* null pointer, bad size, num_heads % num_kv_heads != 0, ... */
    NA_ERR_UNSUPPORTED = -2,   /* a shape or option this build does not implement */
    NA_ERR_CAPACITY = -3,      /* a position does not fit the cache / probability stride */
    NA_ERR_WORKSPACE = -4,     /* workspace missing or smaller than required */
    NA_ERR_CUDA = -5,          /* a CUDA runtime call (launch, attribute) failed */
    NA_ERR_DEVICE_TIMEOUT = -6 /* device only: a bounded wait inside a kernel gave up */
} na_status;

/* Option flags (na_attn_cfg.flags). */
#define NA_QK_NORM 1u                 /* per-head RMSNorm of q and k before RoPE [cortiq fn rmsnorm_head] */
#define NA_QK_NORM_ZERO_CENTERED 2u   /* with NA_QK_NORM: multiply by (1 + w) instead of w */
#define NA_V_NORM 4u                  /* scale-less RMS of v before it enters the cache [cortiq fn vnorm_head] */
#define NA_OUT_GATE 8u                /* out *= sigmoid(gate) after attention [cortiq fn apply_gate] */
#define NA_RING_CACHE 16u             /* the cache is a ring: position pos lives in slot pos % capacity
                                         (needle-core batch.rs, the per-position write-and-attend loop:
                                         a ring of kv_window positions).  Needs window > 0.  The pages'
                                         ring holds exactly the window, so writes and attends must
                                         alternate; here the ring holds at least window + (new tokens
                                         per sequence) - 1 positions, so a whole chunk is written first
                                         without overwriting a key any of its rows still reads.
                                         Prefill needs capacity % 128 == 0 and capacity >= window +
                                         max_new_len - 1; decode needs capacity >= window and
                                         capacity % 64 == 0 (NA_ERR_UNSUPPORTED otherwise). */

/* One attention layer [cortiq struct QwenAttnCfg, the in-scope fields]. */
typedef struct na_attn_cfg {
    int32_t num_heads;     /* H query heads */
    int32_t num_kv_heads;  /* KV heads; H % KV == 0; query head h reads kv head h / (H / KV) */
    int32_t head_dim;      /* d: 64 or 128 */
    int32_t rotary_dim;    /* rd: even, 0 <= rd <= d; RoPE turns dims [0, rd) only */
    float sm_scale;        /* score scale; <= 0 selects 1 / sqrt(head_dim) */
    float rms_eps;         /* epsilon of the qk-norm and v-norm */
    uint32_t flags;        /* NA_* option bits */
    float softcap;         /* > 0: each scaled score s becomes softcap * tanh(s / softcap)
                              ahead of the softmax (cortiq QwenAttnCfg.softcap, the Gemma-2
                              soft cap on attention logits); 0: off */
    int32_t window;        /* > 0: a query at pos attends only keys pos - window + 1 .. pos
                              (cortiq QwenAttnCfg.window, sliding window); 0: full context */
} na_attn_cfg;

/* RoPE frequencies [cortiq fns rope_inv_freq, yarn_inv_freq, rope_rotate_scaled]. */
typedef struct na_rope_params {
    double base;          /* inv_freq[i] = base^(-2 i / rd) */
    int32_t yarn;         /* 0: plain RoPE; 1: YaRN ramp between extrapolation and interpolation */
    double factor;        /* YaRN context extension factor (> 0) */
    int32_t orig_max_pos; /* YaRN original_max_position_embeddings (> 0 when yarn) */
    double beta_fast;     /* YaRN ramp bounds in rotations */
    double beta_slow;
    double attn_factor;   /* multiplier on cos and sin; <= 0 selects 1 without YaRN and
                             0.1 ln(factor) + 1 with YaRN */
} na_rope_params;

/* Caller-owned per-sequence cache: k, v bf16 [batch][num_kv_heads][capacity][head_dim]. */
typedef struct na_kv_cache {
    void *k;
    void *v;
    int32_t batch;
    int32_t capacity;
} na_kv_cache;

/*
 * Fused qk-norm + RoPE + cache append for a chunk of new tokens.
 * [cortiq fn finish_projection (norms before RoPE, partial rotary) and
 *  fn rope_rotate_scaled; needle module doc "What has to stay sequential":
 *  the chunk's K/V are written before any of its positions attends.]
 *
 * For new token t of sequence b, pos = cache_lens[b] + (t - cu_seqlens[b]):
 *   q_out[t][h]            = RoPE(norm_q(q[t][h]), pos)         for every h
 *   cache.k[b][g][pos]     = RoPE(norm_k(k[t][g]), pos)         for every g
 *   cache.v[b][g][pos]     = vnorm(v[t][g])  (or v unchanged)
 * (slot pos % capacity instead of pos with NA_RING_CACHE).
 * RoPE turns pairs (x[i], x[i + rd/2]), i < rd/2, by pos * inv_freq[i] and
 * multiplies both outputs by the attention factor.
 * Accuracy: each stored rotated or normed value is within one bf16 ulp of the
 * exact result: the correctly rounded value unless the exact one lies within
 * ~2^-23 (relative) of a bf16 rounding boundary (about 7 values in a million);
 * V without V-norm is stored bit for bit.
 *
 *   cfg, rope     HOST structs.
 *   batch         number of sequences (>= 1, <= cache->batch).
 *   cu_seqlens    int32 [batch + 1], non-decreasing, cu_seqlens[0] == 0.
 *   cache_lens    int32 [batch]: tokens already cached (prior length).
 *   total_tokens  HOST copy of cu_seqlens[batch]; 0 is a no-op returning NA_OK.
 *   q             bf16 [total_tokens][H][d];  k, v bf16 [total_tokens][KV][d].
 *   q_norm_w, k_norm_w  bf16 [d] (shared by all heads), 16-byte aligned, required with
 *              NA_QK_NORM, else ignored.
 *   q_out         bf16 [total_tokens][H][d]: rotated queries (may not alias q).
 *   status        device int32 or NULL; a token whose pos >= capacity is skipped and
 *                 NA_ERR_CAPACITY is written.
 * The caller advances cache_lens afterwards.
 */
int na_rope_append_kv(const na_attn_cfg *cfg, const na_rope_params *rope, int32_t batch,
                      const int32_t *cu_seqlens, const int32_t *cache_lens,
                      int32_t total_tokens, const void *q, const void *k, const void *v,
                      const void *q_norm_w, const void *k_norm_w, void *q_out,
                      const na_kv_cache *cache, int32_t *status, void *stream);

/*
 * Causal GQA attention of a chunk of new tokens against the cache.
 * [cortiq fn qwen_attention_batch, portable batched attend: query bi of the
 *  chunk sees keys 0 .. s0 + bi; fn attention_head: softmax(q.k * scale) . V;
 *  fn apply_gate; needle fn batch_attention.]
 *
 * The chunk's keys must already be in the cache (na_rope_append_kv first).
 * New token t of sequence b at pos = cache_lens[b] + (t - cu_seqlens[b]) and
 * query head h attends keys 0 .. pos of kv head h / (H / KV):
 *   out[t][h] = sum_j softmax_j(scale * q_rot[t][h] . k_j) v_j   (* sigmoid(gate[t][h]))
 * With cfg->window > 0 only keys pos - window + 1 .. pos are attended; with
 * cfg->softcap > 0 each scaled score is capped before the softmax.  Chunks of a
 * few tokens per sequence (the drafted tokens of a speculative verify) are
 * valid chunks: each attends the cache plus its own earlier tokens.
 * Arithmetic: Q.K and P.V on bf16 tensor cores with fp32 accumulation, the
 * softmax in fp32 with P rounded to bf16 for the P.V product; with unit-scale
 * inputs the output is within 2e-2 (max-abs) and 5e-3 (relative L2) of the
 * exact result.
 *
 *   cu_seqlens    int32 [batch + 1], non-decreasing, cu_seqlens[0] == 0.
 *   cache_lens    int32 [batch]: prior lengths (the same values given to na_rope_append_kv).
 *   total_tokens  HOST copy of cu_seqlens[batch]; 0 is a no-op returning NA_OK.
 *   max_new_len   HOST upper bound of cu_seqlens[b+1] - cu_seqlens[b].
 *   max_total_len HOST upper bound of cache_lens[b] + new length; <= capacity unless
 *                 NA_RING_CACHE (then positions wrap; see that flag for its capacity rules).
 *   q_rot         bf16 [total_tokens][H][d] (q_out of na_rope_append_kv).
 *   gate          bf16 [total_tokens][H][d], required with NA_OUT_GATE, else ignored.
 *   out           bf16 [total_tokens][H][d].
 *   workspace     device scratch of at least na_prefill_workspace_size() bytes
 *                 (NULL allowed when that size is 0).
 *   status        device int32 or NULL: NA_ERR_INVALID_ARG when a new length exceeds
 *                 max_new_len or cu_seqlens[0] != 0, NA_ERR_CAPACITY when a position
 *                 reaches max_total_len or the capacity (those rows are not written).
 * Errors (before anything is enqueued): NA_ERR_INVALID_ARG for null or misaligned
 * buffers and negative sizes, NA_ERR_UNSUPPORTED for a ring whose capacity is not
 * a multiple of 128 or a cache of more than 2^31 - 1 rows (batch x kv heads x
 * capacity), NA_ERR_CAPACITY when the ring cannot hold a window plus a chunk,
 * NA_ERR_WORKSPACE for a missing or short workspace.
 */
int na_attn_prefill_chunk(const na_attn_cfg *cfg, int32_t batch, const int32_t *cu_seqlens,
                          const int32_t *cache_lens, int32_t total_tokens, int32_t max_new_len,
                          int32_t max_total_len, const void *q_rot, const na_kv_cache *cache,
                          const void *gate, void *out, void *workspace, size_t ws_bytes,
                          int32_t *status, void *stream);

/*
 * Single-token decode with optional per-key probabilities.
 * [cortiq fn attention_head (returns the per-key probabilities that feed
 *  eviction scoring), fns qwen_attention_core and attend_all_heads: the current
 *  token is appended first, then each group's K/V are streamed once for all its
 *  query heads.]
 * Arithmetic: bf16 MMAs with fp32 accumulation, softmax and probabilities in
 * fp32; with unit-scale inputs the output is within 2e-2 (max-abs) of the exact
 * result and each probability within 1e-4 (measured ~1.5e-6 of its own value).
 *
 *   q_rot      bf16 [batch][H][d], already rotated (one query per sequence).
 *   kv_lens    int32 [batch]: keys to attend, current token included (0 gives a zero
 *              output and writes no probabilities).
 *   max_kv_len HOST upper bound of kv_lens; <= capacity and <= probs_stride.
 *   gate       bf16 [batch][H][d] with NA_OUT_GATE, else ignored.
 *   out        bf16 [batch][H][d].
 *   probs      fp32 [batch][H][probs_stride] or NULL: probs[b][h][j] = p_j for
 *              j < kv_lens[b]; entries past kv_lens[b] are not written.
 *   num_splits granularity of the key split (0 = automatic).  The keys of all
 *              sequences are cut into one equal slice per CTA of the split pass
 *              (two CTAs per SM); num_splits > 0 makes every slice at least
 *              ceil(max_kv_len / num_splits) keys long, so the longest sequence
 *              is merged from at most num_splits + 1 partial results.
 *   workspace  at least na_decode_workspace_size() bytes: partial results of
 *              every slice piece plus 8 bytes per (sequence, kv head, head
 *              chunk); its size depends on the batch and the head layout, not on
 *              the lengths.  Not read before the call writes it (any contents
 *              will do, also after a call that timed out).
 *   status     device int32 or NULL: NA_ERR_CAPACITY for a length past the
 *              capacity or max_kv_len (zero output), NA_ERR_DEVICE_TIMEOUT when
 *              a wait of the split pass gave up (the affected heads get a zero
 *              output and no probabilities).
 * Errors (before anything is enqueued): NA_ERR_INVALID_ARG for null or
 * misaligned buffers, NA_ERR_CAPACITY when max_kv_len (or, with a ring, the
 * window) exceeds the capacity or a stride, NA_ERR_UNSUPPORTED for a ring whose
 * capacity is not a multiple of 64 (keys are read in aligned 64-key tiles) or a
 * cache of more than 2^31 - 1 rows (batch x kv heads x capacity: the tensor-map
 * row coordinate is 32-bit), NA_ERR_WORKSPACE for a missing or short workspace.
 */
int na_attn_decode(const na_attn_cfg *cfg, int32_t batch, const void *q_rot,
                   const na_kv_cache *cache, const int32_t *kv_lens, int32_t max_kv_len,
                   const void *gate, void *out, float *probs, int32_t probs_stride,
                   int32_t num_splits, void *workspace, size_t ws_bytes, int32_t *status,
                   void *stream);

/*
 * na_attn_decode for callers that cannot supply a workspace.
 * (An addition of this library; the pages have no counterpart.)
 *
 * Some callers have no way to allocate device memory for the workspace: a
 * plugin inside another runtime that owns all device memory and exposes no
 * allocator, or a serving loop that may not allocate once it is running.  This
 * entry point takes the same arguments as na_attn_decode minus the workspace
 * and keeps the split partials in a fixed 20 MiB device array inside the
 * library, so the call allocates nothing.  That array exists on every GPU that
 * loads the library, for as long as the library stays loaded.
 *
 *   - Sizes whose na_decode_workspace_size() exceeds 20 MiB are rejected with
 *     NA_ERR_WORKSPACE before anything is enqueued (for 32 query heads and
 *     head_dim 128: a batch of up to about 1200 sequences, of any length).
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and keeps it; make that first call before any stream
 *     capture.  A cudaDeviceReset() of the device invalidates the kept address:
 *     do not call this entry point on a device after resetting it.
 *   - All calls share the array and it keeps the last call's contents; the
 *     decode needs nothing in it to start at zero (the split pass writes every
 *     partial result and piece span the merge pass reads, in the same call,
 *     and a piece whose wait gave up is written as a marker that the merge
 *     pass reports as NA_ERR_DEVICE_TIMEOUT, with a zero output, instead of
 *     merging).  Calls whose kernels overlap on the GPU (other streams, other
 *     host threads) race on the array: order them on one stream.
 */
int na_attn_decode_static_ws(const na_attn_cfg *cfg, int32_t batch, const void *q_rot,
                             const na_kv_cache *cache, const int32_t *kv_lens, int32_t max_kv_len,
                             const void *gate, void *out, float *probs, int32_t probs_stride,
                             int32_t num_splits, int32_t *status, void *stream);

/*
 * Born-rule importance of a decode step: the probability mass that reads each key.
 * [cortiq fn qwen_attention_core: each head's per-key probabilities are summed into
 *  `imp`, which cache.accumulate_imp adds to the position's running importance for
 *  importance-aware eviction; fn attend_all_heads returns the same sum.]
 *
 *   imp[b][j] = sum over the H query heads of probs[b][h][j]     for j < kv_lens[b]
 * or, with accumulate != 0, imp[b][j] += that sum.  Keys past kv_lens[b] are not
 * touched.  The sum is fp32 and deterministic: the heads are cut into four
 * consecutive groups, each summed in index order, and the group sums are added
 * in group order.  Both strides a multiple of 4 with 16-byte-aligned probs and
 * imp give 16-byte accesses (the fast layout); any stride is correct.
 *
 *   probs       fp32 [batch][H][probs_stride]: the probabilities na_attn_decode wrote.
 *   kv_lens     int32 [batch] (device), the same lengths given to na_attn_decode.
 *   max_kv_len  HOST upper bound of kv_lens; <= probs_stride and <= imp_stride.
 *   imp         fp32 [batch][imp_stride] (device), caller-owned.
 *   status      device int32 or NULL: NA_ERR_CAPACITY for a length past max_kv_len
 *               (that sequence is skipped).
 * Errors: NA_ERR_INVALID_ARG for null buffers or a non-positive batch,
 * NA_ERR_CAPACITY when max_kv_len exceeds a stride.
 */
int na_decode_importance(const na_attn_cfg *cfg, int32_t batch, const float *probs,
                         int32_t probs_stride, const int32_t *kv_lens, int32_t max_kv_len,
                         float *imp, int32_t imp_stride, int32_t accumulate, int32_t *status,
                         void *stream);

/* Workspace bytes (HOST out-parameter) that na_attn_prefill_chunk needs for these bounds. */
int na_prefill_workspace_size(const na_attn_cfg *cfg, int32_t batch, int32_t total_tokens,
                              int32_t max_new_len, int32_t max_total_len, size_t *bytes);

/* Workspace bytes (HOST out-parameter) that na_attn_decode needs for these bounds. */
int na_decode_workspace_size(const na_attn_cfg *cfg, int32_t batch, int32_t max_kv_len,
                             int32_t num_splits, size_t *bytes);

/*
 * Self-test of the device-side failure detection (an addition of this
 * library).  Every wait inside the library's kernels gives up after about a
 * second (2^31 SM cycles) and writes NA_ERR_DEVICE_TIMEOUT into the caller's
 * status word instead of hanging.  This call runs that same bounded wait, in a
 * one-CTA kernel, on a barrier that nothing ever completes: after about a
 * second *status holds NA_ERR_DEVICE_TIMEOUT (unless it already held an error),
 * the kernel returns normally and the context stays usable.
 *
 *   status  device int32, required.
 * Errors: NA_ERR_INVALID_ARG for a NULL status; NA_ERR_CUDA if the launch fails.
 */
int na_selftest_wait_timeout(int32_t *status, void *stream);

/* Static description of a status code (HOST string, never NULL). */
const char *na_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* NA_H */

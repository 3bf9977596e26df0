// na_api.cu -- C ABI of the attention library: argument validation, launch
// planning (tile counts, KV splits, workspace layout) and kernel launches.
// Nothing here allocates device memory or synchronises with the device.
#include <math.h>
#include <string.h>

#include <cmath>

#include "na_internal.cuh"

namespace {

constexpr uint32_t kKnownFlags =
    NA_QK_NORM | NA_QK_NORM_ZERO_CENTERED | NA_V_NORM | NA_OUT_GATE | NA_RING_CACHE;
constexpr double kPi = 3.14159265358979323846;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cfg(const na_attn_cfg *c)
{
    if (!c)
        return NA_ERR_INVALID_ARG;
    if (c->num_heads <= 0 || c->num_kv_heads <= 0 || c->num_heads % c->num_kv_heads != 0)
        return NA_ERR_INVALID_ARG;
    if (c->rotary_dim < 0 || (c->rotary_dim & 1) || c->rotary_dim > c->head_dim)
        return NA_ERR_INVALID_ARG;
    if (c->flags & ~kKnownFlags)
        return NA_ERR_INVALID_ARG;
    if (!(c->rms_eps >= 0.f))
        return NA_ERR_INVALID_ARG;
    if (!(c->softcap >= 0.f) || !std::isfinite(c->softcap) || c->window < 0)
        return NA_ERR_INVALID_ARG;
    if ((c->flags & NA_RING_CACHE) && c->window <= 0)  // a ring only makes sense with a window
        return NA_ERR_INVALID_ARG;
    if (c->head_dim != 64 && c->head_dim != 128)
        return NA_ERR_UNSUPPORTED;
    return NA_OK;
}

float score_scale_log2(const na_attn_cfg *c)
{
    const double s = c->sm_scale > 0.f ? (double)c->sm_scale : 1.0 / sqrt((double)c->head_dim);
    return (float)(s * 1.4426950408889634);
}

int check_cache(const na_kv_cache *cache, int batch)
{
    if (!cache || !cache->k || !cache->v || cache->capacity <= 0 || cache->batch < batch)
        return NA_ERR_INVALID_ARG;
    if (!aligned16(cache->k) || !aligned16(cache->v))
        return NA_ERR_INVALID_ARG;
    return NA_OK;
}

// The attention kernels address cache rows (sequence, kv head, slot) through
// tensor maps whose row coordinate is a signed 32-bit integer.
// The attention calls encode tensor maps with a driver call before they
// launch, and a driver call needs the device's context current on the calling
// thread.  The runtime binds it lazily (on a launch or a copy), so a thread
// whose first CUDA call is one of these may not have it yet: the current
// device's primary context is bound once per thread and device.
int bind_context()
{
    thread_local int bound = -1;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return NA_ERR_CUDA;
    if (dev != bound) {
        if (cudaSetDevice(dev) != cudaSuccess)
            return NA_ERR_CUDA;
        bound = dev;
    }
    return NA_OK;
}

int check_cache_rows(const na_kv_cache *cache, int kv_heads)
{
    return (long long)cache->batch * kv_heads * cache->capacity > 0x7fffffffLL ? NA_ERR_UNSUPPORTED
                                                                               : NA_OK;
}

int sm_count()
{
    // per device; an unreadable count plans for 152 SMs (the launches then
    // report the device error themselves)
    static std::atomic<int> cached[kMaxDevices];
    const int dev = current_device_index();
    if (dev >= 0) {
        const int n = cached[dev].load(std::memory_order_relaxed);
        if (n > 0)
            return n;
    }
    int d = 0, n = 0;
    if (cudaGetDevice(&d) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0)
        return 152;
    if (dev >= 0)
        cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

// RoPE inverse frequencies in double (cortiq fns rope_inv_freq / yarn_inv_freq,
// with the rotary dimension as the exponent's denominator).
void rope_frequencies(const na_rope_params *r, int rd, double *out)
{
    const int half = rd / 2;
    if (!r->yarn) {
        for (int i = 0; i < half; i++)
            out[i] = pow(r->base, -2.0 * i / rd);
        return;
    }
    auto dim_at = [&](double rotations) {
        return rd * log(r->orig_max_pos / (rotations * 2.0 * kPi)) / (2.0 * log(r->base));
    };
    const int low = (int)fmax(floor(dim_at(r->beta_fast)), 0.0);
    const int high = (int)fmin(fmax(ceil(dim_at(r->beta_slow)), 0.0), (double)(half > 0 ? half - 1 : 0));
    const double span = (double)(high > low + 1 ? high - low : 1);
    for (int i = 0; i < half; i++) {
        const double plain = pow(r->base, -2.0 * i / rd);
        double ramp = (i > low ? i - low : 0) / span;
        ramp = ramp < 0.0 ? 0.0 : (ramp > 1.0 ? 1.0 : ramp);
        // ramp 0: keep the plain frequency; ramp 1: divide it by the factor.
        out[i] = plain * (1.0 - ramp) + (plain / r->factor) * ramp;
    }
}

// Multiplier on cos and sin: given value, else 1, else YaRN's 0.1 ln(factor) + 1.
double rope_attention_factor(const na_rope_params *r)
{
    if (r->attn_factor > 0.0)
        return r->attn_factor;
    if (r->yarn && r->factor > 1.0)
        return 0.1 * log(r->factor) + 1.0;
    return 1.0;
}

int check_rope(const na_rope_params *r)
{
    if (!r || !(r->base > 1.0))
        return NA_ERR_INVALID_ARG;
    if (r->yarn && (!(r->factor > 0.0) || r->orig_max_pos <= 0 || !(r->beta_fast > 0.0) ||
                    !(r->beta_slow > 0.0)))
        return NA_ERR_INVALID_ARG;
    return NA_OK;
}

struct PrefillPlan {
    int pack, tile_tokens, q_tiles, full_units, tail_units, num_splits, split_len, grid;
    size_t ws_bytes;
};

// Units (query tile, head group, sequence) run one per CTA, at one CTA per
// SM, in the order of the grid (heaviest query tiles first within a head, the
// longest sequences first): the hardware starts each on the next free SM, and
// the units streaming the same K/V run side by side.  Only the units left over
// after the last whole wave -- or all of them when there are fewer than SMs --
// are cut into up to SMs / units equal key ranges, at least four key tiles
// each, so that the last wave keeps every SM busy (640 units of a long
// context chunk on 152 SMs left 120 SMs idle for most of a fifth wave); a
// merge pass combines the pieces of those units.
PrefillPlan plan_prefill(const na_attn_cfg *c, int batch, int total_tokens, int max_new_len,
                         int max_total_len)
{
    PrefillPlan pl{};
    const int bm = prefill_q_tile(), bn = prefill_key_tile();
    // GQA packing: a tile holds bm / group tokens of all `group` query heads
    // that share a kv head (when the group divides bm), so a sequence with few
    // new tokens fills the tile's rows instead of leaving most of them idle,
    // and each K/V tile serves the whole group.
    // A single sequence whose tokens fill whole tiles gains nothing (measured
    // 3% slower packed on 128-token chunks, group 4), so it stays unpacked.
    const int group = c->num_heads / c->num_kv_heads;
    pl.pack = (group > 1 && bm % group == 0) ? group : 1;
    if (batch == 1 && total_tokens % bm == 0)
        pl.pack = 1;
    pl.tile_tokens = bm / pl.pack;
    pl.q_tiles = (max_new_len + pl.tile_tokens - 1) / pl.tile_tokens;
    const long long units = (long long)batch * pl.q_tiles * (c->num_heads / pl.pack);
    const long long sms = sm_count();
    // With ragged lengths the unit count is only a bound (the shortest
    // sequences' trailing units are empty), so the leftover units after the
    // last whole wave are known to be real only when every sequence has
    // max_new_len new tokens.
    const bool exact = (long long)batch * max_new_len == total_tokens;
    pl.full_units = (int)(units >= sms && exact ? units - units % sms : (units >= sms ? units : 0));
    pl.tail_units = (int)(units - pl.full_units);
    // Keys one tile can see: all history, or with a sliding window at most the
    // window plus the tile's own tokens (from the key tile holding the first
    // row's window start).
    long long span = max_total_len;
    if (c->window > 0) {
        const long long w = (long long)c->window + pl.tile_tokens - 1 + bn;
        span = w < span ? w : span;
    }
    int splits = 1;
    if (pl.tail_units > 0 && span > 4 * bn) {
        splits = (int)(sms / pl.tail_units);
        const int max_by_len = (int)((span + 4 * bn - 1) / (4 * bn));
        splits = splits < max_by_len ? splits : max_by_len;
        if (splits < 1)
            splits = 1;
    }
    if (splits > 1) {
        int len = (int)((span + splits - 1) / splits);
        len = (len + bn - 1) / bn * bn;
        pl.split_len = len;
        pl.num_splits = (int)((span + len - 1) / len);
    } else {
        pl.split_len = span > 0 ? (int)span : 1;
        pl.num_splits = 1;
    }
    pl.grid = pl.full_units + pl.tail_units * pl.num_splits;
    pl.ws_bytes = pl.num_splits > 1 ? (size_t)pl.tail_units * pl.num_splits * bm *
                                          (c->head_dim + 2) * sizeof(float)
                                    : 0;
    return pl;
}

struct DecodePlan {
    int heads_per_cta, grid, min_slice, max_pieces, streams;
    size_t ws_bytes;
};

// Decode split plan.  The split pass runs a fixed grid (two CTAs per SM) and
// cuts the concatenated key streams into one equal slice per CTA (at least
// min_slice keys), so the workspace holds one partial row group per piece:
// streams + grid pieces at most, whatever the lengths.
DecodePlan plan_decode(const na_attn_cfg *c, int batch, int max_kv_len, int num_splits)
{
    DecodePlan pl{};
    const int tile = decode_key_tile();
    const int group = c->num_heads / c->num_kv_heads;
    // query heads scored together (the MMA takes up to 8): each stream of
    // K/V is read once for them
    pl.heads_per_cta = (group % 8 == 0) ? 8 : (group % 4 == 0) ? 4 : ((group % 2 == 0) ? 2 : 1);
    const int len = max_kv_len > 0 ? max_kv_len : 1;
    int min_slice = num_splits > 0 ? (len + num_splits - 1) / num_splits : 4 * tile;
    if (min_slice < 1)
        min_slice = 1;
    pl.min_slice = min_slice;
    pl.grid = decode_ctas_per_sm() * sm_count();
    pl.streams = batch * c->num_kv_heads * (group / pl.heads_per_cta);
    pl.max_pieces = pl.streams + pl.grid;
    const size_t rows = (size_t)pl.max_pieces * pl.heads_per_cta;
    pl.ws_bytes = rows * (c->head_dim + 2) * 4 + (size_t)pl.streams * 2 * 4;
    pl.ws_bytes = (pl.ws_bytes + 15) / 16 * 16;
    return pl;
}

}  // namespace

extern "C" {

const char *na_status_string(int status)
{
    switch (status) {
    case NA_OK: return "ok";
    case NA_ERR_INVALID_ARG: return "invalid argument";
    case NA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case NA_ERR_CAPACITY: return "position beyond cache capacity or probability stride";
    case NA_ERR_WORKSPACE: return "workspace missing or too small";
    case NA_ERR_CUDA: return "CUDA runtime error";
    case NA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
    }
}

int na_rope_append_kv(const na_attn_cfg *cfg, const na_rope_params *rope, int32_t batch,
                      const int32_t *cu_seqlens, const int32_t *cache_lens, int32_t total_tokens,
                      const void *q, const void *k, const void *v, const void *q_norm_w,
                      const void *k_norm_w, void *q_out, const na_kv_cache *cache, int32_t *status,
                      void *stream)
{
    int rc = check_cfg(cfg);
    if (rc != NA_OK)
        return rc;
    if ((rc = check_rope(rope)) != NA_OK)
        return rc;
    if (batch <= 0 || total_tokens < 0)
        return NA_ERR_INVALID_ARG;
    if ((rc = check_cache(cache, batch)) != NA_OK)
        return rc;
    if (total_tokens == 0)
        return NA_OK;
    if (!cu_seqlens || !cache_lens || !q || !k || !v || !q_out)
        return NA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out))
        return NA_ERR_INVALID_ARG;
    if ((cfg->flags & NA_QK_NORM) &&
        (!q_norm_w || !k_norm_w || !aligned16(q_norm_w) || !aligned16(k_norm_w)))
        return NA_ERR_INVALID_ARG;
    if (rope_append_smem_bytes(cfg->num_heads, cfg->num_kv_heads, cfg->head_dim,
                               cfg->rotary_dim) > 200 * 1024)
        return NA_ERR_UNSUPPORTED;

    double inv_freq[64];
    rope_frequencies(rope, cfg->rotary_dim, inv_freq);
    RopeAppendParams p{};
    p.H = cfg->num_heads;
    p.KV = cfg->num_kv_heads;
    p.d = cfg->head_dim;
    p.rd = cfg->rotary_dim;
    p.flags = cfg->flags;
    p.eps = cfg->rms_eps;
    p.rope_scale = (float)rope_attention_factor(rope);
    p.batch = batch;
    p.capacity = cache->capacity;
    p.total_tokens = total_tokens;
    p.cu_seqlens = cu_seqlens;
    p.cache_lens = cache_lens;
    p.q = static_cast<const bf16 *>(q);
    p.k = static_cast<const bf16 *>(k);
    p.v = static_cast<const bf16 *>(v);
    p.qw = static_cast<const bf16 *>(q_norm_w);
    p.kw = static_cast<const bf16 *>(k_norm_w);
    p.q_out = static_cast<bf16 *>(q_out);
    p.cache_k = static_cast<bf16 *>(cache->k);
    p.cache_v = static_cast<bf16 *>(cache->v);
    p.status = status;
    return launch_rope_append(p, inv_freq, cfg->rotary_dim / 2,
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? NA_OK
               : NA_ERR_CUDA;
}

int na_prefill_workspace_size(const na_attn_cfg *cfg, int32_t batch, int32_t total_tokens,
                              int32_t max_new_len, int32_t max_total_len, size_t *bytes)
{
    int rc = check_cfg(cfg);
    if (rc != NA_OK)
        return rc;
    if (!bytes || batch <= 0 || total_tokens < 0 || max_new_len < 0 || max_total_len < 0)
        return NA_ERR_INVALID_ARG;
    *bytes = plan_prefill(cfg, batch, total_tokens, max_new_len, max_total_len).ws_bytes;
    return NA_OK;
}

int na_attn_prefill_chunk(const na_attn_cfg *cfg, int32_t batch, const int32_t *cu_seqlens,
                          const int32_t *cache_lens, int32_t total_tokens, int32_t max_new_len,
                          int32_t max_total_len, const void *q_rot, const na_kv_cache *cache,
                          const void *gate, void *out, void *workspace, size_t ws_bytes,
                          int32_t *status, void *stream)
{
    int rc = check_cfg(cfg);
    if (rc != NA_OK)
        return rc;
    if (batch <= 0 || total_tokens < 0 || max_new_len < 0 || max_total_len < 0)
        return NA_ERR_INVALID_ARG;
    if ((rc = check_cache(cache, batch)) != NA_OK)
        return rc;
    if ((rc = check_cache_rows(cache, cfg->num_kv_heads)) != NA_OK)
        return rc;
    if (total_tokens == 0)
        return NA_OK;
    if (!cu_seqlens || !cache_lens || !q_rot || !out || max_new_len <= 0)
        return NA_ERR_INVALID_ARG;
    const bool ring = (cfg->flags & NA_RING_CACHE) != 0;
    if (ring) {  // tiles of 128 keys never wrap; a whole chunk fits beside its rows' windows
        if (cache->capacity % prefill_key_tile() != 0)
            return NA_ERR_UNSUPPORTED;
        if ((long long)cfg->window + max_new_len - 1 > cache->capacity)
            return NA_ERR_CAPACITY;
    } else if (max_total_len > cache->capacity) {
        return NA_ERR_CAPACITY;
    }
    if ((long long)total_tokens * cfg->num_heads * cfg->head_dim >= (1ll << 40))
        return NA_ERR_UNSUPPORTED;  // tile coordinates are 32-bit
    if (!aligned16(q_rot) || !aligned16(out))
        return NA_ERR_INVALID_ARG;
    const bool gated = (cfg->flags & NA_OUT_GATE) != 0;
    if (gated && (!gate || !aligned16(gate)))
        return NA_ERR_INVALID_ARG;
    const PrefillPlan pl = plan_prefill(cfg, batch, total_tokens, max_new_len, max_total_len);
    if (pl.ws_bytes > 0 && (!workspace || ws_bytes < pl.ws_bytes || !aligned16(workspace)))
        return NA_ERR_WORKSPACE;

    PrefillParams p{};
    p.H = cfg->num_heads;
    p.KV = cfg->num_kv_heads;
    p.group = p.H / p.KV;
    p.batch = batch;
    p.capacity = cache->capacity;
    p.scale_log2 = score_scale_log2(cfg);
    p.max_new_len = max_new_len;
    p.max_total_len = max_total_len;
    p.total_tokens = total_tokens;
    p.softcap = cfg->softcap;
    p.window = cfg->window;
    p.pack = pl.pack;
    p.tile_tokens = pl.tile_tokens;
    p.q_tiles = pl.q_tiles;
    p.HG = p.H / pl.pack;
    p.kv_read_once = (pl.q_tiles == 1 && p.HG == p.KV) ? 1 : 0;
    p.full_units = pl.full_units;
    p.tail_units = pl.tail_units;
    p.split_len = pl.split_len;
    p.num_splits = pl.num_splits;
    p.flags = cfg->flags;
    p.cu_seqlens = cu_seqlens;
    p.cache_lens = cache_lens;
    p.q = static_cast<const bf16 *>(q_rot);
    p.cache_k = static_cast<const bf16 *>(cache->k);
    p.cache_v = static_cast<const bf16 *>(cache->v);
    p.gate = gated ? static_cast<const bf16 *>(gate) : nullptr;
    p.out = static_cast<bf16 *>(out);
    if (pl.ws_bytes > 0) {
        p.part_o = static_cast<float *>(workspace);
        p.part_ml = p.part_o + (size_t)pl.tail_units * pl.num_splits * prefill_q_tile() * cfg->head_dim;
    }
    p.status = status;
    if ((rc = bind_context()) != NA_OK)
        return rc;
    return launch_prefill(p, cfg->head_dim, total_tokens, cache->batch,
                          static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? NA_OK
               : NA_ERR_CUDA;
}

int na_decode_importance(const na_attn_cfg *cfg, int32_t batch, const float *probs,
                         int32_t probs_stride, const int32_t *kv_lens, int32_t max_kv_len,
                         float *imp, int32_t imp_stride, int32_t accumulate, int32_t *status,
                         void *stream)
{
    int rc = check_cfg(cfg);
    if (rc != NA_OK)
        return rc;
    if (batch <= 0 || max_kv_len < 0 || !probs || !kv_lens || !imp)
        return NA_ERR_INVALID_ARG;
    if (max_kv_len > probs_stride || max_kv_len > imp_stride)
        return NA_ERR_CAPACITY;
    ImportanceParams p{};
    p.H = cfg->num_heads;
    p.batch = batch;
    p.max_kv_len = max_kv_len;
    p.probs_stride = probs_stride;
    p.imp_stride = imp_stride;
    p.accumulate = accumulate != 0;
    p.vector_ok = aligned16(probs) && aligned16(imp) && probs_stride % 4 == 0 && imp_stride % 4 == 0;
    p.probs = probs;
    p.kv_lens = kv_lens;
    p.imp = imp;
    p.status = status;
    if ((rc = bind_context()) != NA_OK)
        return rc;
    return launch_importance(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? NA_OK
                                                                                   : NA_ERR_CUDA;
}

int na_decode_workspace_size(const na_attn_cfg *cfg, int32_t batch, int32_t max_kv_len,
                             int32_t num_splits, size_t *bytes)
{
    int rc = check_cfg(cfg);
    if (rc != NA_OK)
        return rc;
    if (!bytes || batch <= 0 || max_kv_len < 0 || num_splits < 0)
        return NA_ERR_INVALID_ARG;
    *bytes = plan_decode(cfg, batch, max_kv_len, num_splits).ws_bytes;
    return NA_OK;
}

int na_attn_decode(const na_attn_cfg *cfg, int32_t batch, const void *q_rot,
                   const na_kv_cache *cache, const int32_t *kv_lens, int32_t max_kv_len,
                   const void *gate, void *out, float *probs, int32_t probs_stride,
                   int32_t num_splits, void *workspace, size_t ws_bytes, int32_t *status,
                   void *stream)
{
    int rc = check_cfg(cfg);
    if (rc != NA_OK)
        return rc;
    if (batch <= 0 || max_kv_len < 0 || num_splits < 0)
        return NA_ERR_INVALID_ARG;
    if ((rc = check_cache(cache, batch)) != NA_OK)
        return rc;
    if ((rc = check_cache_rows(cache, cfg->num_kv_heads)) != NA_OK)
        return rc;
    if (!q_rot || !kv_lens || !out || !aligned16(q_rot) || !aligned16(out))
        return NA_ERR_INVALID_ARG;
    if ((cfg->flags & NA_RING_CACHE) ? cfg->window > cache->capacity : max_kv_len > cache->capacity)
        return NA_ERR_CAPACITY;
    // a ring is read in whole key tiles, which must not cross its end
    if ((cfg->flags & NA_RING_CACHE) && cache->capacity % decode_key_tile() != 0)
        return NA_ERR_UNSUPPORTED;
    if (probs && probs_stride < max_kv_len)
        return NA_ERR_CAPACITY;
    const bool gated = (cfg->flags & NA_OUT_GATE) != 0;
    if (gated && !gate)
        return NA_ERR_INVALID_ARG;
    const DecodePlan pl = plan_decode(cfg, batch, max_kv_len, num_splits);
    if (!workspace || ws_bytes < pl.ws_bytes || !aligned16(workspace))
        return NA_ERR_WORKSPACE;

    DecodeParams p{};
    p.H = cfg->num_heads;
    p.KV = cfg->num_kv_heads;
    p.group = p.H / p.KV;
    p.batch = batch;
    p.capacity = cache->capacity;
    p.cache_batch = cache->batch;
    p.scale_log2 = score_scale_log2(cfg);
    p.head_chunks = p.group / pl.heads_per_cta;
    p.grid = pl.grid;
    p.min_slice = pl.min_slice;
    p.max_pieces = pl.max_pieces;
    p.max_kv_len = max_kv_len;
    p.flags = cfg->flags;
    p.window = cfg->window;
    if (cfg->softcap > 0.f) {  // scores are log2-domain: c tanh(s / c) -> tanh via 2^(2 s / c)
        p.cap_in = 2.0f / cfg->softcap;
        p.cap_out = cfg->softcap * 1.4426950408889634f;
    }
    p.q = static_cast<const bf16 *>(q_rot);
    p.cache_k = static_cast<const bf16 *>(cache->k);
    p.cache_v = static_cast<const bf16 *>(cache->v);
    p.gate = gated ? static_cast<const bf16 *>(gate) : nullptr;
    p.kv_lens = kv_lens;
    p.out = static_cast<bf16 *>(out);
    p.probs = probs;
    p.probs_stride = probs ? probs_stride : 0;
    p.part_o = static_cast<float *>(workspace);
    const size_t rows = (size_t)pl.max_pieces * pl.heads_per_cta;
    p.part_ml = p.part_o + rows * cfg->head_dim;
    p.piece_span = reinterpret_cast<int32_t *>(p.part_ml + rows * 2);
    p.status = status;
    if ((rc = bind_context()) != NA_OK)
        return rc;
    return launch_decode(p, cfg->head_dim, pl.heads_per_cta, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? NA_OK
               : NA_ERR_CUDA;
}

}  // extern "C"

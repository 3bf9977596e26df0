"""Pins that tie the oracle to something other than itself.

Each pin takes an ``Oracle`` and raises AssertionError when it disagrees with
what the pages print (worked examples under ``tests/golden/``), a closed form,
a textbook or library routine (``math.cos``, ``scipy.special.softmax``), an
invariant of the mathematics, or brute force on tiny inputs.  The same pins
run against deliberately broken copies of the oracle (tests/test_oracle_mutants.py)
to show that a plausible mistake anywhere in it fails at least one of them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import softmax as scipy_softmax

import oracle as oracle_mod

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _close(a, b, tol, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert err <= tol, f"{what}: max abs error {err} > {tol}"


# ------------------------------------------------------------------ RoPE ---

def pin_rope_page_tests(o):
    """cortiq unit tests rope_preserves_norm / rope_identity_at_position_zero."""
    g = _golden("rope_page_tests.json")
    a = g["preserves_norm"]
    inv = o.rope_inv_freq(a["head_dim"], a["base"])
    y = o.rope_rotate(np.array(a["x"]), a["head_dim"], a["position"], inv)
    assert abs(np.linalg.norm(y) - np.linalg.norm(a["x"])) < a["abs_tol"]
    b = g["identity_at_zero"]
    inv = o.rope_inv_freq(b["head_dim"], b["base"])
    y = o.rope_rotate(np.array(b["x"]), b["head_dim"], b["position"], inv)
    _close(y, b["x"], b["abs_tol"], "identity at position 0")


def pin_rope_frequency_values(o):
    """Closed forms of base^(-2i/rd): rd=4, base 1e4 gives [1, 1e-2]; rd=128,
    base 5e5 has inv_freq[32] = 5e5^(-1/2)."""
    _close(o.rope_inv_freq(4, 10000.0), [1.0, 0.01], 1e-15, "rd 4 frequencies")
    f = o.rope_inv_freq(128, 500000.0)
    assert f.shape == (64,)
    _close(f[32], 1.0 / math.sqrt(500000.0), 1e-15, "rd 128 midpoint")
    _close(f[0], 1.0, 0.0, "first frequency")


def pin_rope_closed_form_rotation(o):
    """One pair (rd 2, frequency 1): e0 at position p -> (cos p, sin p) and
    e1 -> (-sin p, cos p), checked against math.cos / math.sin."""
    inv = np.array([1.0])
    for p in (1, 2, 5, 1000, 32767):
        y = o.rope_rotate(np.array([1.0, 0.0]), 2, p, inv)
        _close(y, [math.cos(p), math.sin(p)], 1e-12, f"e0 at {p}")
        y = o.rope_rotate(np.array([0.0, 1.0]), 2, p, inv)
        _close(y, [-math.sin(p), math.cos(p)], 1e-12, f"e1 at {p}")


def pin_rope_half_split_pairing(o):
    """Half-split pairing (i, i + rd/2): a unit vector e1 of an 8-dim head
    only reaches indices 1 and 5."""
    inv = o.rope_inv_freq(8, 10000.0)
    x = np.zeros(8)
    x[1] = 1.0
    y = o.rope_rotate(x, 8, 3, inv)
    nz = set(np.nonzero(np.abs(y) > 1e-15)[0].tolist())
    assert nz == {1, 5}, f"pairing touched {sorted(nz)}"
    # the pair turns by 3 * inv_freq[1]
    _close(y[[1, 5]], [math.cos(3 * inv[1]), math.sin(3 * inv[1])], 1e-12, "pair 1")


def pin_rope_relative_position(o):
    """<R(m) q, R(n) k> depends only on m - n (full rotary)."""
    rng = np.random.default_rng(1)
    inv = o.rope_inv_freq(64, 10000.0)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for (m, n, c) in ((5, 2, 11), (100, 37, 4000), (0, 9, 123), (30000, 29000, 2767)):
        a = o.rope_rotate(q, 64, m, inv) @ o.rope_rotate(k, 64, n, inv)
        b = o.rope_rotate(q, 64, m + c, inv) @ o.rope_rotate(k, 64, n + c, inv)
        assert abs(a - b) < 1e-9, (m, n, c, a, b)


def pin_rope_composition_and_scale(o):
    """R(a) R(b) = R(a + b); the scale multiplies the norm; dims >= rd and
    rd = 0 are identity."""
    rng = np.random.default_rng(2)
    inv = o.rope_inv_freq(32, 500000.0)
    x = rng.standard_normal(48)
    _close(o.rope_rotate(o.rope_rotate(x, 32, 17, inv), 32, 40, inv),
           o.rope_rotate(x, 32, 57, inv), 1e-12, "composition")
    y = o.rope_rotate(x, 32, 9, inv, scale=1.5)
    _close(np.linalg.norm(y[:32]), 1.5 * np.linalg.norm(x[:32]), 1e-12, "scaled norm")
    _close(y[32:], x[32:], 0.0, "dims past rd")
    _close(o.rope_rotate(x, 0, 9, inv), x, 0.0, "rd 0")


def pin_yarn_page_endpoints(o):
    """cortiq unit test yarn_frequency_endpoints_match_interpolation_contract."""
    g = _golden("yarn_endpoints.json")
    f = o.yarn_inv_freq(g["rd"], g["base"], g["factor"], g["orig_max_pos"], g["beta_fast"],
                        g["beta_slow"])
    base = o.rope_inv_freq(g["rd"], g["base"])
    assert f.shape == (g["len"],)
    for c in g["checks"]:
        i = c["index"]
        assert abs(f[i] - base[i] / c["divided_by"]) < c["abs_tol"], (i, f[i], base[i])


def pin_yarn_reductions(o):
    """factor 1 is plain RoPE; for rotary 64, base 1e6, factor 4, original 8192,
    betas (32, 1): the ramp runs from index low = floor(8.59) = 8 to high =
    ceil(16.6) = 17, indices <= 8 keep the plain frequency, indices >= 17 are
    divided by 4, and index 11 sits one third up the ramp (ratio 3/4)."""
    _close(o.yarn_inv_freq(64, 1e6, 1.0, 8192, 32.0, 1.0), o.rope_inv_freq(64, 1e6), 1e-18,
           "factor 1")
    f, low, high = o.yarn_inv_freq(64, 1e6, 4.0, 8192, 32.0, 1.0, with_bounds=True)
    base = o.rope_inv_freq(64, 1e6)
    assert (low, high) == (8, 17), (low, high)
    _close(f[:9], base[:9], 1e-18, "extrapolated band")
    _close(f[17:], base[17:] / 4.0, 1e-18, "interpolated band")
    _close(f[11] / base[11], 0.75, 1e-14, "one third up the ramp")
    r = f / base
    assert np.all(np.diff(r) <= 1e-15), "ratio must fall monotonically"


def pin_yarn_attention_factor(o):
    """The multiplier on cos and sin (cortiq QwenAttnCfg.rope_scale, fn
    rope_rotate_scaled): the YaRN paper's 0.1 ln(s) + 1 at the hand-computed
    values of tests/golden/yarn_attn_factor.json; 1 without YaRN or with a
    factor <= 1; a positive value given by the caller passes unchanged.  In the
    append, the rotated dims of K come out scaled by exactly that factor (norm
    times the factor) and the other dims unchanged."""
    g = _golden("yarn_attn_factor.json")
    for c in g["values"]:
        _close(o.rope_attn_factor(True, c["factor"], 0.0), c["expected"], g["abs_tol"],
               f"factor {c['factor']}")
        _close(o.rope_attn_factor(True, c["factor"], -1.0), c["expected"], g["abs_tol"],
               "negative selects the default")
    br = g["branches"]
    _close(o.rope_attn_factor(False, 4.0, 0.0), br["no_yarn_default"], 0.0, "no yarn")
    for f in (1.0, 0.5):
        _close(o.rope_attn_factor(True, f, 0.0), br["yarn_factor_at_most_one_default"], 0.0,
               f"yarn factor {f}")
    for v in br["given_value_passes_through"]:
        _close(o.rope_attn_factor(True, 4.0, v), v, 0.0, "given value (yarn)")
        _close(o.rope_attn_factor(False, 1.0, v), v, 0.0, "given value (plain)")
    # through the append: one token, K of 16 dims with rotary 8 at position 300
    rng = np.random.default_rng(31)
    d, rd = 16, 8
    inv = o.yarn_inv_freq(rd, 1e6, 4.0, 8192, 32.0, 1.0)
    s = o.rope_attn_factor(True, 4.0, 0.0)
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    v = rng.standard_normal((1, 1, d))
    ck = np.zeros((1, 1, 400, d))
    cv = np.zeros((1, 1, 400, d))
    q_rot = o.rope_append(1, 1, d, rd, 0, 0.0, inv, s, [0, 1], [300], q, k, v, None, None, ck, cv)
    kr = ck[0, 0, 300]
    _close(np.linalg.norm(kr[:rd]), 1.1386294361119890618 * np.linalg.norm(k[0, 0, :rd]), 1e-13,
           "rotated K norm")
    _close(kr[rd:], k[0, 0, rd:], 0.0, "K dims past rd")
    _close(np.linalg.norm(q_rot[0, 0, :rd]),
           1.1386294361119890618 * np.linalg.norm(q[0, 0, :rd]), 1e-13, "rotated Q norm")


# ------------------------------------------------------------ ring cache ---

def _simulated_ring(n_positions, capacity):
    """Where a ring buffer puts positions 0, 1, ...: a write pointer that
    starts at slot 0, advances by one slot per position and wraps to 0 at the
    end (needle fn batch_attention's ring of kv_window positions)."""
    slots, ptr = [], 0
    for _ in range(n_positions):
        slots.append(ptr)
        ptr += 1
        if ptr == capacity:
            ptr = 0
    return slots


def pin_ring_slot_simulated(o):
    """The oracle's ring slot of every position equals the slot a simulated
    write pointer gives it, for rings of 1, 3, 128 and 448 slots."""
    for cap in (1, 3, 128, 448):
        sim = _simulated_ring(5 * cap + 7, cap)
        got = [o.ring_slot(p, cap) for p in range(len(sim))]
        assert got == sim, f"ring of {cap}: {got[:12]} vs {sim[:12]}"
    assert o.ring_slot(32768 * 3 + 5, 32768) == 5


def pin_ring_equals_linear_window(o):
    """With a window W, a ring cache of window + chunk - 1 slots gives the same
    chunked prefill rows and the same decode outputs and probabilities as a
    linear cache (the ring holds every key a row can see); each appended
    position lands in the simulated slot with the linear cache's value; a ring
    one slot too small for the chunk is rejected."""
    rng = np.random.default_rng(41)
    H, KV, d, rd, W = 2, 1, 8, 8, 3
    inv = o.rope_inv_freq(rd, 1e4)
    prior, new = [9, 0], [4, 3]
    R = W + max(new) - 1
    cu = [0, new[0], new[0] + new[1]]
    T = cu[-1]
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, KV, d))
    v = rng.standard_normal((T, KV, d))
    L = 16
    lin_k = rng.standard_normal((2, KV, L, d))
    lin_v = rng.standard_normal((2, KV, L, d))
    ring_k = np.full((2, KV, R, d), np.nan)
    ring_v = np.full((2, KV, R, d), np.nan)
    for b in range(2):
        sim = _simulated_ring(prior[b], R)
        for pos in range(prior[b]):
            ring_k[b, :, sim[pos]] = lin_k[b, :, pos]
            ring_v[b, :, sim[pos]] = lin_v[b, :, pos]
    q_lin = o.rope_append(H, KV, d, rd, 0, 0.0, inv, 1.0, cu, prior, q, k, v, None, None,
                          lin_k, lin_v)
    q_ring = o.rope_append(H, KV, d, rd, o_ring(o), 0.0, inv, 1.0, cu, prior, q, k, v, None, None,
                           ring_k, ring_v)
    _close(q_ring, q_lin, 0.0, "rotated q")
    for b in range(2):
        sim = _simulated_ring(prior[b] + new[b], R)
        for pos in range(prior[b], prior[b] + new[b]):
            _close(ring_k[b, :, sim[pos]], lin_k[b, :, pos], 0.0, f"ring K slot of {pos}")
            _close(ring_v[b, :, sim[pos]], lin_v[b, :, pos], 0.0, f"ring V slot of {pos}")
    rows = list(range(T))
    a = o.attend_rows(H, KV, d, 0.6, 0, cu, prior, q_lin, lin_k, lin_v, None, rows, window=W)
    b_ = o.attend_rows(H, KV, d, 0.6, o_ring(o), cu, prior, q_lin, ring_k, ring_v, None, rows,
                       window=W)
    _close(b_, a, 0.0, "ring prefill rows")
    lens = [p + n for p, n in zip(prior, new)]
    qd = rng.standard_normal((2, H, d))
    lo, lp = o.decode(H, KV, d, 0.6, 0, qd, lin_k, lin_v, lens, probs_stride=L, window=W)
    ro, rp = o.decode(H, KV, d, 0.6, o_ring(o), qd, ring_k, ring_v, lens, probs_stride=L, window=W)
    _close(ro, lo, 0.0, "ring decode out")
    _close(rp, lp, 0.0, "ring decode probs")
    small_k = np.zeros((2, KV, R - 1, d))
    try:
        o.attend_rows(H, KV, d, 0.6, o_ring(o), cu, prior, q_lin, small_k, small_k.copy(), None,
                      rows, window=W)
    except ValueError:
        pass
    else:
        raise AssertionError("a ring smaller than window + chunk - 1 must be rejected")


def o_ring(o):
    import oracle as oracle_mod
    return oracle_mod.RING_CACHE


# ----------------------------------------------------------------- norms ---

def pin_rmsnorm_values(o):
    """x = 3 everywhere, eps 7: 3 / sqrt(9 + 7) = 0.75 times the weight; unit
    RMS at eps 0; zero-centred style with w = 0 equals Qwen style with w = 1."""
    d = 8
    w = np.linspace(0.5, 2.0, d)
    _close(o.rmsnorm_head(np.full(d, 3.0), w, 7.0), 0.75 * w, 1e-15, "constant input")
    rng = np.random.default_rng(3)
    x = rng.standard_normal(128) * 5
    y = o.rmsnorm_head(x, np.ones(128), 0.0)
    _close(np.sqrt(np.mean(y * y)), 1.0, 1e-13, "unit rms")
    _close(o.rmsnorm_head(x, np.zeros(128), 0.0, zero_centered=True), y, 1e-15, "zero-centred")
    _close(o.rmsnorm_head(np.full(d, 3.0), w, 7.0, zero_centered=True), 0.75 * (1 + w), 1e-15,
           "zero-centred weights")


def pin_vnorm_values(o):
    """Scale-less V-norm: (3, 4) at eps 0 becomes (3, 4) / sqrt(12.5); a
    constant 2 vector with eps 12 becomes 2 / 4 = 0.5."""
    _close(o.vnorm_head(np.array([3.0, 4.0]), 0.0), np.array([3.0, 4.0]) / math.sqrt(12.5),
           1e-15, "(3, 4)")
    _close(o.vnorm_head(np.full(6, 2.0), 12.0), np.full(6, 0.5), 1e-15, "constant")


# ------------------------------------------------------------- attention ---

def _attend_single(o, q, keys, vals, scale, gate=None):
    """One query through attend_rows: a one-token chunk whose prior length
    places it at the last key."""
    n, d = keys.shape
    cache_k = np.zeros((1, 1, n, d))
    cache_v = np.zeros((1, 1, n, d))
    cache_k[0, 0] = keys
    cache_v[0, 0] = vals
    flags = oracle_mod.OUT_GATE if gate is not None else 0
    g = None if gate is None else gate.reshape(1, 1, d)
    out = o.attend_rows(1, 1, d, scale, flags, [0, 1], [n - 1], q.reshape(1, 1, d), cache_k,
                        cache_v, g, [0])
    return out[0, 0]


def pin_attention_page_uniform(o):
    """cortiq unit test attention_head_uniform, through both decode and prefill."""
    g = _golden("attention_head_uniform.json")
    d = g["head_dim"]
    q, k, v = np.array(g["q"]), np.array(g["k"]), np.array(g["v"])
    n = k.shape[0]
    cache_k = np.zeros((1, 1, n, d))
    cache_v = np.zeros((1, 1, n, d))
    cache_k[0, 0], cache_v[0, 0] = k, v
    out, probs = o.decode(1, 1, d, 1.0 / math.sqrt(d), 0, q.reshape(1, 1, d), cache_k, cache_v,
                          [n])
    _close(out[0, 0], g["expected_out"], g["exact_tolerance"], "uniform out")
    _close(probs[0, 0], g["expected_probs"], g["exact_tolerance"], "uniform probs")
    assert abs(probs.sum() - 1.0) < g["page_tolerance_mass"]
    _close(_attend_single(o, q, k, v, 0.5), g["expected_out"], g["exact_tolerance"], "prefill")


def pin_attention_scale_value(o):
    """d = 4, scale 1/2: q = 2 e0, keys e0 and 0 -> scores 1 and 0, so the
    first probability is e / (1 + e)."""
    q = np.array([2.0, 0, 0, 0])
    keys = np.array([[1.0, 0, 0, 0], [0, 0, 0, 0]])
    vals = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    cache_k = keys.reshape(1, 1, 2, 4).copy()
    cache_v = vals.reshape(1, 1, 2, 4).copy()
    out, probs = o.decode(1, 1, 4, 0.5, 0, q.reshape(1, 1, 4), cache_k, cache_v, [2])
    p0 = math.e / (1 + math.e)
    _close(probs[0, 0], [p0, 1 - p0], 1e-15, "probs")
    _close(out[0, 0], [p0, 1 - p0, 0, 0], 1e-15, "out")


def pin_attention_special_cases(o):
    """One key gives o = v; identical keys give the mean of V; empty key set
    gives zero output and untouched probabilities."""
    rng = np.random.default_rng(4)
    d = 16
    q = rng.standard_normal(d)
    v = rng.standard_normal((1, d))
    _close(_attend_single(o, q, rng.standard_normal((1, d)), v, 0.25), v[0], 1e-15, "one key")
    k1 = rng.standard_normal(d)
    vals = rng.standard_normal((7, d))
    _close(_attend_single(o, q, np.tile(k1, (7, 1)), vals, 0.25), vals.mean(0), 1e-14,
           "identical keys")
    cache = np.zeros((1, 1, 4, d))
    out, probs = o.decode(1, 1, d, 0.25, 0, q.reshape(1, 1, d), cache, cache, [0],
                          probs_stride=4)
    _close(out, np.zeros_like(out), 0.0, "empty out")
    _close(probs, np.zeros_like(probs), 0.0, "empty probs")


def pin_decode_vs_library_softmax(o):
    """Decode probabilities and output against scipy.special.softmax on random
    tiny inputs; probabilities sum to 1."""
    rng = np.random.default_rng(5)
    B, H, KV, d, cap = 3, 6, 2, 8, 11
    lens = [11, 1, 6]
    q = rng.standard_normal((B, H, d))
    ck = rng.standard_normal((B, KV, cap, d))
    cv = rng.standard_normal((B, KV, cap, d))
    scale = 0.3
    out, probs = o.decode(H, KV, d, scale, 0, q, ck, cv, lens, probs_stride=cap)
    for b in range(B):
        for h in range(H):
            g = h // (H // KV)
            n = lens[b]
            p = scipy_softmax(scale * ck[b, g, :n] @ q[b, h])
            _close(probs[b, h, :n], p, 1e-14, f"probs {b},{h}")
            _close(probs[b, h, n:], np.zeros(cap - n), 0.0, "probs tail")
            _close(out[b, h], p @ cv[b, g, :n], 1e-13, f"out {b},{h}")
            assert abs(probs[b, h].sum() - 1.0) < 1e-13


def _prefill(o, H, KV, d, rd, inv, rope_scale, flags, eps, cu, prior, q, k, v, qw, kw,
             cache_k, cache_v, gate, scale):
    q_rot = o.rope_append(H, KV, d, rd, flags, eps, inv, rope_scale, cu, prior, q, k, v, qw, kw,
                          cache_k, cache_v)
    rows = list(range(int(cu[-1])))
    return o.attend_rows(H, KV, d, scale, flags, cu, prior, q_rot, cache_k, cache_v, gate,
                         rows), q_rot


def pin_causal_mask_brute_force(o):
    """Whole-prompt prefill against an explicit T x T lower-triangular mask
    with scipy softmax, RoPE applied by rotating each row (brute force)."""
    rng = np.random.default_rng(6)
    H, KV, d, T = 4, 2, 8, 9
    inv = o.rope_inv_freq(d, 10000.0)
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, KV, d))
    v = rng.standard_normal((T, KV, d))
    ck = np.zeros((1, KV, T, d))
    cv = np.zeros((1, KV, T, d))
    scale = 1 / math.sqrt(d)
    out, _ = _prefill(o, H, KV, d, d, inv, 1.0, 0, 1e-6, [0, T], [0], q, k, v, None, None,
                      ck, cv, None, scale)
    mask = np.tril(np.ones((T, T), dtype=bool))
    for h in range(H):
        g = h // (H // KV)
        qr = np.stack([o.rope_rotate(q[t, h], d, t, inv) for t in range(T)])
        kr = np.stack([o.rope_rotate(k[t, g], d, t, inv) for t in range(T)])
        s = np.where(mask, scale * qr @ kr.T, -np.inf)
        p = scipy_softmax(s, axis=1)
        _close(out[:, h], p @ v[:, g], 1e-13, f"head {h}")


def pin_gqa_equals_replicated_mha(o):
    """H=4 over KV=2 equals H=4 over KV=4 with each KV head copied into its
    group (heads 0,1 -> kv 0; heads 2,3 -> kv 1)."""
    rng = np.random.default_rng(7)
    H, d, n = 4, 8, 5
    q = rng.standard_normal((1, H, d))
    ck = rng.standard_normal((1, 2, n, d))
    cv = rng.standard_normal((1, 2, n, d))
    a, pa = o.decode(H, 2, d, 0.4, 0, q, ck, cv, [n])
    ck4 = np.ascontiguousarray(np.repeat(ck, 2, axis=1))
    cv4 = np.ascontiguousarray(np.repeat(cv, 2, axis=1))
    b, pb = o.decode(H, 4, d, 0.4, 0, q, ck4, cv4, [n])
    _close(a, b, 1e-15, "gqa out")
    _close(pa, pb, 1e-15, "gqa probs")


def pin_chunked_equals_single_chunk(o):
    """needle "What has to stay sequential": a prompt in chunks of 3 gives
    the same outputs and cache as the whole prompt in one chunk (two
    sequences, qk-norm, v-norm, gate, partial rotary)."""
    rng = np.random.default_rng(8)
    H, KV, d, rd, L, B = 4, 2, 8, 4, 10, 2
    inv = o.rope_inv_freq(rd, 500.0)
    flags = oracle_mod.QK_NORM | oracle_mod.V_NORM | oracle_mod.OUT_GATE
    q = rng.standard_normal((B, L, H, d))
    k = rng.standard_normal((B, L, KV, d))
    v = rng.standard_normal((B, L, KV, d))
    gate = rng.standard_normal((B, L, H, d))
    qw, kw = rng.standard_normal(d) + 1, rng.standard_normal(d) + 1
    scale = 0.35
    ck1, cv1 = np.zeros((B, KV, L, d)), np.zeros((B, KV, L, d))
    whole, _ = _prefill(o, H, KV, d, rd, inv, 1.1, flags, 1e-5, [0, L, 2 * L], [0, 0],
                        q.reshape(-1, H, d), k.reshape(-1, KV, d), v.reshape(-1, KV, d), qw, kw,
                        ck1, cv1, gate.reshape(-1, H, d), scale)
    whole = whole.reshape(B, L, H, d)
    ck2, cv2 = np.zeros((B, KV, L, d)), np.zeros((B, KV, L, d))
    for lo in range(0, L, 3):
        hi = min(L, lo + 3)
        n = hi - lo
        part, _ = _prefill(o, H, KV, d, rd, inv, 1.1, flags, 1e-5, [0, n, 2 * n], [lo, lo],
                           q[:, lo:hi].reshape(-1, H, d), k[:, lo:hi].reshape(-1, KV, d),
                           v[:, lo:hi].reshape(-1, KV, d), qw, kw, ck2, cv2,
                           gate[:, lo:hi].reshape(-1, H, d), scale)
        _close(part.reshape(B, n, H, d), whole[:, lo:hi], 1e-13, f"chunk at {lo}")
    _close(ck1, ck2, 0.0, "cache k")
    _close(cv1, cv2, 0.0, "cache v")


def pin_decode_equals_last_prefill_row(o):
    """Decode of the token at position p equals the prefill row at p of the
    whole prompt (append then attend)."""
    rng = np.random.default_rng(9)
    H, KV, d, L = 4, 2, 8, 7
    inv = o.rope_inv_freq(d, 10000.0)
    q = rng.standard_normal((L, H, d))
    k = rng.standard_normal((L, KV, d))
    v = rng.standard_normal((L, KV, d))
    ck, cv = np.zeros((1, KV, L, d)), np.zeros((1, KV, L, d))
    out, q_rot = _prefill(o, H, KV, d, d, inv, 1.0, 0, 1e-6, [0, L], [0], q, k, v, None, None,
                          ck, cv, None, 0.3)
    for p in (L - 2, L - 1):
        dec, _ = o.decode(H, KV, d, 0.3, 0, q_rot[p].reshape(1, H, d), ck, cv, [p + 1],
                          want_probs=False)
        _close(dec[0], out[p], 1e-14, f"decode at {p}")


def pin_pair_chunk_equals_two_decode_steps(o):
    """A speculative pair verify: a two-token chunk over a filled cache gives
    the rows of two decode steps, each appending its token and then attending
    (cortiq qwen_attention_batch attends a batch of positions of one sequence;
    its decode path appends, then attends).  Plain, with a sliding window and
    with a soft cap; the two caches agree bit for bit."""
    rng = np.random.default_rng(21)
    H, KV, d, P = 4, 2, 8, 6
    inv = o.rope_inv_freq(d, 10000.0)
    scale = 0.3
    q = rng.standard_normal((P + 2, H, d))
    k = rng.standard_normal((P + 2, KV, d))
    v = rng.standard_normal((P + 2, KV, d))
    for softcap, window in ((0.0, 0), (0.0, 3), (2.5, 0)):
        ck1, cv1 = np.zeros((1, KV, P + 2, d)), np.zeros((1, KV, P + 2, d))
        o.rope_append(H, KV, d, d, 0, 1e-6, inv, 1.0, [0, P], [0], q[:P], k[:P], v[:P], None,
                      None, ck1, cv1)
        ck2, cv2 = ck1.copy(), cv1.copy()
        q_rot = o.rope_append(H, KV, d, d, 0, 1e-6, inv, 1.0, [0, 2], [P], q[P:], k[P:], v[P:],
                              None, None, ck1, cv1)
        pair = o.attend_rows(H, KV, d, scale, 0, [0, 2], [P], q_rot, ck1, cv1, None, [0, 1],
                             softcap=softcap, window=window)
        for t in range(2):
            s = slice(P + t, P + t + 1)
            qt = o.rope_append(H, KV, d, d, 0, 1e-6, inv, 1.0, [0, 1], [P + t], q[s], k[s], v[s],
                               None, None, ck2, cv2)
            dec, _ = o.decode(H, KV, d, scale, 0, qt.reshape(1, H, d), ck2, cv2, [P + t + 1],
                              want_probs=False, softcap=softcap, window=window)
            _close(dec[0], pair[t], 1e-14, f"pair row {t} (cap {softcap}, window {window})")
        _close(ck1, ck2, 0.0, "cache k")
        _close(cv1, cv2, 0.0, "cache v")


def pin_gate_values(o):
    """Gate logits 0 halve the output; logits of +-40 keep or zero it."""
    rng = np.random.default_rng(10)
    d = 8
    q, keys, vals = rng.standard_normal(d), rng.standard_normal((3, d)), rng.standard_normal((3, d))
    plain = _attend_single(o, q, keys, vals, 0.3)
    _close(_attend_single(o, q, keys, vals, 0.3, gate=np.zeros(d)), plain / 2, 1e-15, "gate 0")
    g = np.where(np.arange(d) % 2 == 0, 40.0, -40.0)
    want = np.where(np.arange(d) % 2 == 0, plain, 0.0)
    _close(_attend_single(o, q, keys, vals, 0.3, gate=g), want, 1e-16, "gate +-40")


def pin_norm_before_rope_in_append(o):
    """cortiq fn finish_projection: qk-norm runs before RoPE, V-norm leaves V
    unrotated; the cache slot is the absolute position."""
    rng = np.random.default_rng(11)
    H, KV, d, rd = 2, 1, 8, 6
    inv = o.rope_inv_freq(rd, 100.0)
    q = rng.standard_normal((2, H, d))
    k = rng.standard_normal((2, KV, d))
    v = rng.standard_normal((2, KV, d))
    qw, kw = rng.standard_normal(d) + 1, rng.standard_normal(d) + 1
    ck, cv = np.full((1, KV, 6, d), 99.0), np.full((1, KV, 6, d), 99.0)
    flags = oracle_mod.QK_NORM | oracle_mod.V_NORM
    q_rot = o.rope_append(H, KV, d, rd, flags, 1e-6, inv, 1.2, [0, 2], [3], q, k, v, qw, kw, ck,
                          cv)
    for t in range(2):
        pos = 3 + t
        for h in range(H):
            want = o.rope_rotate(o.rmsnorm_head(q[t, h], qw, 1e-6), rd, pos, inv, 1.2)
            _close(q_rot[t, h], want, 1e-15, "q")
        _close(ck[0, 0, pos], o.rope_rotate(o.rmsnorm_head(k[t, 0], kw, 1e-6), rd, pos, inv, 1.2),
               1e-15, "k slot")
        _close(cv[0, 0, pos], o.vnorm_head(v[t, 0], 1e-6), 1e-15, "v slot")
    untouched = [0, 1, 2, 5]
    assert np.all(ck[0, 0, untouched] == 99.0) and np.all(cv[0, 0, untouched] == 99.0)


def pin_importance_sums_and_brute_force(o):
    """Born-rule importance (cortiq fn qwen_attention_core sums every head's
    probabilities per key): against per-head scipy softmax summed by hand; each
    sequence's importance totals H (every head's probabilities sum to 1), an
    empty sequence gets none, keys past the length stay untouched, and
    accumulation adds to what the buffer holds."""
    rng = np.random.default_rng(13)
    B, H, KV, d, cap = 3, 6, 3, 8, 9
    lens = [9, 0, 4]
    q = rng.standard_normal((B, H, d))
    ck = rng.standard_normal((B, KV, cap, d))
    cv = rng.standard_normal((B, KV, cap, d))
    _, probs = o.decode(H, KV, d, 0.4, 0, q, ck, cv, lens, probs_stride=cap)
    imp = o.decode_importance(H, probs, lens)
    for b in range(B):
        n = lens[b]
        want = np.zeros(cap)
        for h in range(H):
            g = h // (H // KV)
            if n:
                want[:n] += scipy_softmax(0.4 * ck[b, g, :n] @ q[b, h])
        _close(imp[b], want, 1e-13, f"importance {b}")
        assert abs(imp[b].sum() - (H if n else 0)) < 1e-12
    prev = rng.standard_normal((B, cap))
    acc = o.decode_importance(H, probs, lens, imp=prev, accumulate=True)
    for b in range(B):
        n = lens[b]
        _close(acc[b, :n], prev[b, :n] + imp[b, :n], 1e-14, "accumulate")
        _close(acc[b, n:], prev[b, n:], 0.0, "untouched tail")


def pin_importance_page_uniform(o):
    """The pages' uniform example (identical keys: every probability 1/3)
    gives importance H/3 on every key."""
    H, KV, d = 4, 1, 3
    q = np.ones((1, H, d))
    ck = np.ones((1, KV, 3, d))
    cv = np.eye(3).reshape(1, KV, 3, d)
    _, probs = o.decode(H, KV, d, 1.0, 0, q, ck, cv, [3], probs_stride=3)
    _close(o.decode_importance(H, probs, [3])[0], np.full(3, H / 3.0), 1e-14, "uniform")


def pin_softcap(o):
    """Logit soft-capping (QwenAttnCfg.softcap: each scaled score s becomes
    c*tanh(s/c) ahead of the softmax): against library softmax of c*tanh(scale q.k / c); a huge cap
    is plain attention; capped scores never leave (-c, c)."""
    rng = np.random.default_rng(21)
    B, H, KV, d, cap = 2, 4, 2, 8, 10
    lens = [10, 6]
    q = 3.0 * rng.standard_normal((B, H, d))
    ck = rng.standard_normal((B, KV, cap, d))
    cv = rng.standard_normal((B, KV, cap, d))
    c = 2.0
    out, probs = o.decode(H, KV, d, 0.5, 0, q, ck, cv, lens, probs_stride=cap, softcap=c)
    plain_out, plain_p = o.decode(H, KV, d, 0.5, 0, q, ck, cv, lens, probs_stride=cap)
    huge_out, huge_p = o.decode(H, KV, d, 0.5, 0, q, ck, cv, lens, probs_stride=cap, softcap=1e12)
    for b in range(B):
        n = lens[b]
        for h in range(H):
            g = h // (H // KV)
            s = 0.5 * ck[b, g, :n] @ q[b, h]
            p = scipy_softmax(c * np.tanh(s / c))
            _close(probs[b, h, :n], p, 1e-14, "capped probs")
            _close(out[b, h], p @ cv[b, g, :n], 1e-13, "capped out")
            # a cap of 2 bounds the probability ratio by e^(2c)
            assert probs[b, h, :n].max() / probs[b, h, :n].min() < math.exp(2 * c) + 1e-9
    _close(huge_p, plain_p, 1e-12, "huge cap probs")
    _close(huge_out, plain_out, 1e-12, "huge cap out")


def pin_sliding_window(o):
    """Sliding window (QwenAttnCfg.window; fn attend_all_heads attends from
    stored - window): against a brute-force softmax over the last W keys, keys
    before the window get probability 0, W >= n is full attention, W = 1 gives
    exactly the newest value; in prefill, row pos sees keys pos-W+1 .. pos (a
    windowed prefill row equals windowed decode at that position)."""
    rng = np.random.default_rng(22)
    B, H, KV, d, cap = 2, 2, 1, 8, 9
    lens = [9, 4]
    q = rng.standard_normal((B, H, d))
    ck = rng.standard_normal((B, KV, cap, d))
    cv = rng.standard_normal((B, KV, cap, d))
    W = 3
    out, probs = o.decode(H, KV, d, 0.7, 0, q, ck, cv, lens, probs_stride=cap, window=W)
    full_out, full_p = o.decode(H, KV, d, 0.7, 0, q, ck, cv, lens, probs_stride=cap, window=50)
    plain_out, plain_p = o.decode(H, KV, d, 0.7, 0, q, ck, cv, lens, probs_stride=cap)
    one_out, one_p = o.decode(H, KV, d, 0.7, 0, q, ck, cv, lens, probs_stride=cap, window=1)
    for b in range(B):
        n = lens[b]
        lo = max(0, n - W)
        for h in range(H):
            p = scipy_softmax(0.7 * ck[b, 0, lo:n] @ q[b, h])
            _close(probs[b, h, lo:n], p, 1e-14, "window probs")
            _close(probs[b, h, :lo], np.zeros(lo), 0.0, "outside window")
            _close(out[b, h], p @ cv[b, 0, lo:n], 1e-13, "window out")
            _close(one_out[b, h], cv[b, 0, n - 1], 0.0, "window 1 value")
            _close(one_p[b, h, :n], np.eye(n)[n - 1], 0.0, "window 1 probs")
    _close(full_out, plain_out, 0.0, "window >= n")
    _close(full_p, plain_p, 0.0, "window >= n probs")
    # prefill rows against decode at the same positions
    L = 7
    qs = rng.standard_normal((L, H, d))
    kc = rng.standard_normal((1, KV, L, d))
    vc = rng.standard_normal((1, KV, L, d))
    rows = o.attend_rows(H, KV, d, 0.7, 0, [0, L], [0], qs, kc, vc, None, list(range(L)),
                         window=W)
    for t in range(L):
        dec, _ = o.decode(H, KV, d, 0.7, 0, qs[t:t + 1], kc, vc, [t + 1], window=W)
        _close(rows[t], dec[0], 1e-14, f"prefill row {t}")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

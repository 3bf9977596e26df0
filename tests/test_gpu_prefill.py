"""Parity of the chunked causal GQA prefill (append + attend) with the oracle,
from tiny ragged cases to the full-size workloads (sampled rows there)."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import (Guarded, assert_out_close, check_cache, gpu_chunked, gpu_step,
                     oracle_append, oracle_rows, prompt_as_step, sample_rows)

pytestmark = pytest.mark.gpu


def _compare_step(oracle, step, rows=None, what=""):
    g = gpu_step(step)
    assert g.status == 0, f"status {g.status}"
    ost = oracle_append(oracle, step)
    check_cache(g.cache_k, g.cache_v, step, ost)
    T = step.total_tokens
    rows = list(range(T)) if rows is None else rows
    ref = oracle_rows(oracle, step, ost, rows)
    got = g.out[rows].to(torch.float64).numpy()
    return assert_out_close(got, ref, what)


def test_prefill_h4kv2d64_single_chunk_all_rows(oracle):
    """128-token prompt, one chunk, empty cache, 4/2 heads, d 64, base 1e4."""
    prompt = W.make_chunked_prompt(W.C1, seed=0)
    step = prompt_as_step(prompt)
    _compare_step(oracle, step, what="h4kv2d64 t128")


RAGGED = {
    "t1_empty_cache": ([0], [1]),
    "t3_prior77": ([77], [3]),
    "t127": ([0], [127]),
    "t129_prior5": ([5], [129]),
    "t200_prior300": ([300], [200]),
}


@pytest.mark.parametrize("name", list(RAGGED))
def test_prefill_ragged_lengths(oracle, name):
    prior, new = RAGGED[name]
    spec = W.Spec(H=8, KV=2, d=128, rd=128, rope=W.RopeParams(base=5e5), std=0.5)
    step = W.make_step(spec, prior, new, 512, seed=21)
    _compare_step(oracle, step, what=name)


SHAPES = {
    "group5_d128_partial_yarn": W.Spec(H=10, KV=2, d=128, rd=64,
                                        rope=W.RopeParams(base=1e6, yarn=True, factor=4.0,
                                                          orig_max_pos=8192)),
    "group8_d64": W.Spec(H=8, KV=1, d=64, rd=64, rope=W.RopeParams(base=1e4)),
    "mha_d64_qknorm_gate_vnorm": W.Spec(H=3, KV=3, d=64, rd=64, qk_norm=True, v_norm=True,
                                         out_gate=True),
    "group16_qknorm_gate": W.Spec(H=32, KV=2, d=128, rd=128, rope=W.RopeParams(base=1e6),
                                   qk_norm=True, out_gate=True),
    "explicit_scale": W.Spec(H=4, KV=2, d=128, rd=128, sm_scale=0.05),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_prefill_shapes_varlen(oracle, name):
    spec = SHAPES[name]
    step = W.make_step(spec, [0, 250, 31], [70, 1, 140], 512, seed=31)
    _compare_step(oracle, step, what=name)


def test_prefill_short_chunk_long_history_splits_keys(oracle):
    """Few query rows against a long history: the launch splits the keys and
    merges the partials."""
    spec = W.Spec(H=4, KV=1, d=128, rd=128, rope=W.RopeParams(base=5e5))
    step = W.make_step(spec, [3000], [16], 4096, seed=41)
    _compare_step(oracle, step, what="split keys")


@pytest.mark.parametrize("prior,new", [(0, 200), (300, 37), (5000, 96)])
def test_prefill_single_sequence_packed_heads(oracle, prior, new):
    """One sequence whose token count is not a multiple of the 128-row tile:
    the launch packs the group's query heads into each tile (token-major
    rows), takes every tile below the token count as certainly non-empty, and
    (with the long history) splits the keys."""
    spec = W.Spec(H=8, KV=2, d=128, rd=128, rope=W.RopeParams(base=1e4), out_gate=True)
    step = W.make_step(spec, [prior], [new], prior + new + 64, seed=57)
    _compare_step(oracle, step, what=f"packed single {prior}+{new}")


CAPPED_WINDOWED = {
    # unit-scale inputs (the tolerance's regime) with a cap small enough to bend
    # the scores (|s| ~ 1..4 against c = 2)
    "softcap2_group4": (W.Spec(H=8, KV=2, d=128, rd=128, softcap=2.0), [0, 300], [70, 140]),
    "softcap_d64_qknorm_gate": (W.Spec(H=6, KV=3, d=64, rd=64, softcap=5.0, qk_norm=True,
                                       out_gate=True), [17, 0], [40, 9]),
    "window200_varlen": (W.Spec(H=8, KV=2, d=128, rd=128, window=200), [1000, 30, 0], [300, 5, 130]),
    "window1_single": (W.Spec(H=4, KV=1, d=128, rd=128, window=1), [20], [40]),
    "window_and_softcap_mha": (W.Spec(H=3, KV=3, d=64, rd=32, window=77, softcap=8.0), [400], [150]),
}


@pytest.mark.parametrize("name", list(CAPPED_WINDOWED))
def test_prefill_softcap_and_window(oracle, name):
    """Logit soft-capping and sliding-window attention against the oracle."""
    spec, prior, new = CAPPED_WINDOWED[name]
    cap = max(p + n for p, n in zip(prior, new)) + 8
    step = W.make_step(spec, prior, new, cap, seed=71)
    _compare_step(oracle, step, what=name)


def test_prefill_window_long_history_splits(oracle):
    """A short chunk behind a long history with a window: the key range starts at
    the window, and the launch splits it across CTAs."""
    spec = W.Spec(H=4, KV=1, d=128, rd=128, window=1500)
    step = W.make_step(spec, [6000], [24], 6100, seed=73)
    _compare_step(oracle, step, what="window + splits")


SHORT_CHUNKS = {
    # a speculative pair verify: two drafted tokens after a long history
    "pair_verify_h32kv8": (W.Spec(H=32, KV=8, d=128, rd=128, rope=W.RopeParams(base=5e5)),
                           [4093], [2], 4160),
    "varlen_1_to_8_d64_gate": (W.Spec(H=8, KV=2, d=64, rd=64, out_gate=True),
                               [0, 513, 77, 2000], [1, 8, 5, 3], 2048),
    "window_softcap_qknorm": (W.Spec(H=10, KV=2, d=128, rd=64, qk_norm=True, window=300,
                                     softcap=3.0), [1200, 5], [4, 7], 1280),
}


@pytest.mark.parametrize("name", list(SHORT_CHUNKS))
def test_prefill_short_chunks(oracle, name):
    """Chunks of a few new tokens (a speculative pair verify, drafted tokens):
    the tile packs the group's query heads over the few tokens, so each K/V tile
    is streamed once for all of them."""
    spec, prior, new, cap = SHORT_CHUNKS[name]
    step = W.make_step(spec, prior, new, cap, seed=79)
    _compare_step(oracle, step, what=name)


MULTI_WAVE = {
    # one sequence with at least two whole waves of 128-row units on 152 SMs and
    # a tail of leftover units (cut into key ranges when few are left)
    "h40kv8_d64_gate": (W.Spec(H=40, KV=8, d=64, rd=64, out_gate=True), 300, 1024),
    "h40kv8_d128_softcap": (W.Spec(H=40, KV=8, d=128, rd=64, softcap=30.0), 1000, 1024),
    "h40kv8_d128_window_gate": (W.Spec(H=40, KV=8, d=128, rd=128, window=700, out_gate=True),
                                2000, 1024),
    "h48kv8_d128_tail_whole": (W.Spec(H=48, KV=8, d=128, rd=128), 5000, 1152),
}


@pytest.mark.parametrize("name", list(MULTI_WAVE))
def test_prefill_multi_wave_single_sequence(oracle, name):
    """Calls of one sequence with several waves of units and a tail (cut into
    key ranges or whole); sampled rows of every head against the oracle, the
    cache bit for bit."""
    spec, prior, new = MULTI_WAVE[name]
    capacity = (prior + new + 127) // 128 * 128
    step = W.make_step(spec, [prior], [new], capacity, seed=131)
    _compare_step(oracle, step, rows=sample_rows(new, 96, seed=7), what=name)


def _sequences_of(step: W.StepInputs, idx):
    """The sub-step holding only sequences `idx` of a packed step (their tokens,
    bounds and caches), and the packed rows those tokens had."""
    cu = step.cu_seqlens.tolist()
    rows = [t for b in idx for t in range(cu[b], cu[b + 1])]
    new = [cu[b + 1] - cu[b] for b in idx]
    pick = lambda x: None if x is None else x[rows].contiguous()
    sub = W.StepInputs(spec=step.spec,
                       cu_seqlens=torch.tensor(np.concatenate([[0], np.cumsum(new)]),
                                               dtype=torch.int32),
                       cache_lens=step.cache_lens[idx].clone(), q=pick(step.q), k=pick(step.k),
                       v=pick(step.v), gate=pick(step.gate), q_norm_w=step.q_norm_w,
                       k_norm_w=step.k_norm_w, cache_k=step.cache_k[idx].contiguous(),
                       cache_v=step.cache_v[idx].contiguous())
    return sub, rows


def test_full_pair_verify_b64(oracle):
    """The pair-verify workload at full size, as the benchmark runs it: 64
    sequences each appending 2 drafted tokens after 510..8190 cached ones, then
    one attention call over all of them (more than 32 sequences: the slots are
    not ranked by length).  Eight sequences, the longest and the shortest among
    them, are checked against the oracle: every row of every head and their
    caches bit for bit."""
    step = W.make_pair_verify_step()
    g = gpu_step(step)
    assert g.status == 0, f"status {g.status}"
    lens = step.cache_lens.tolist()
    idx = sorted({int(np.argmax(lens)), int(np.argmin(lens))} |
                 set(sample_rows(len(lens), 6, seed=17)))
    sub, rows = _sequences_of(step, idx)
    ost = oracle_append(oracle, sub)
    check_cache(g.cache_k[idx], g.cache_v[idx], sub, ost)
    ref = oracle_rows(oracle, sub, ost, list(range(sub.total_tokens)))
    assert_out_close(g.out[rows].to(torch.float64).numpy(), ref, f"pair verify sequences {idx}")


def test_prefill_ring_cache(oracle):
    """Ring cache (slot = position % capacity) with a window: the chunk is
    appended into the ring, every row attends the last `window` keys, and the
    ring holds exactly the newest `capacity` positions afterwards.  The oracle
    appends into and attends from the same ring."""
    import causal_gqa_attention_rope_gb300 as na
    from harness import (attn_cfg, oracle_append, oracle_rows, ring_from_linear, rope_cfg,
                         assert_within_ulp)
    spec = W.Spec(H=8, KV=2, d=128, rd=128, window=200)
    prior, new = [1000, 37, 0], [150, 5, 60]
    step = W.make_step(spec, prior, new, 1300, seed=83)
    R = 384  # a multiple of 128 and >= window + max new - 1
    dev = "cuda"
    cfg = attn_cfg(spec)
    cfg.ring_cache = True
    ck = ring_from_linear(oracle, step.cache_k, prior, R)
    cv = ring_from_linear(oracle, step.cache_v, prior, R)
    ring_step = W.StepInputs(**{**step.__dict__, "cache_k": ck, "cache_v": cv})
    cache = na.KVCache(ck.clone().to(dev), cv.clone().to(dev))
    q, k, v = step.q.to(dev), step.k.to(dev), step.v.to(dev)
    cu, lens = step.cu_seqlens.to(dev), step.cache_lens.to(dev)
    gq, go = Guarded(q.shape, q.dtype, dev), Guarded(q.shape, q.dtype, dev)
    q_out, out = gq.t, go.t
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    T = step.total_tokens
    max_new, max_tot = max(new), max(p + n for p, n in zip(prior, new))
    na.na_rope_append_kv(cfg, rope_cfg(spec), cu, lens, q, k, v, q_out, cache, status=status)
    ws = na.workspace(na.na_prefill_workspace_size(cfg, 3, T, max_new, max_tot), dev)
    na.na_attn_prefill_chunk(cfg, cu, lens, max_new, max_tot, q_out, cache, out, workspace=ws,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gq.check("ring q_out")
    go.check("ring out")
    ost = oracle_append(oracle, ring_step, ring=True)
    ref = oracle_rows(oracle, ring_step, ost, list(range(T)), ring=True)
    assert_out_close(out.cpu().double().numpy(), ref, "ring prefill")
    gk, gv = cache.k.cpu(), cache.v.cpu()
    for b in range(3):
        end = prior[b] + new[b]
        written = {oracle.ring_slot(pos, R) for pos in range(prior[b], end)}
        for slot in range(R):
            if slot in written:  # appended now: the oracle's ring slot, within 1 ulp
                assert_within_ulp(gk[b, :, slot], ost.cache_k[b, :, slot], f"ring K {b},{slot}")
                assert np.array_equal(gv[b, :, slot].double().numpy(), ost.cache_v[b, :, slot])
            else:  # history (or the sentinel) kept bit for bit
                assert torch.equal(gk[b, :, slot].view(torch.int16), ck[b, :, slot].view(torch.int16))
                assert torch.equal(gv[b, :, slot].view(torch.int16), cv[b, :, slot].view(torch.int16))


def test_prefill_varlen_small_all_rows(oracle):
    """Packed varlen step with qk-norm and gate (the mixed-serving options) at
    a size the oracle checks in full."""
    spec = W.C5.spec
    step = W.make_step(spec, [0, 300, 1024, 77], [130, 1, 65, 200], 1536, seed=51)
    _compare_step(oracle, step, what="varlen small")


def test_chunked_equals_single_chunk_on_gpu():
    """The same prompt in 4 chunks of 64 and in one chunk of 256 gives the same
    outputs (within the output tolerance) and the same cache bits."""
    wl = W.PrefillWorkload(name="t", spec=W.Spec(H=8, KV=2, d=128, rd=128,
                                                 rope=W.RopeParams(base=5e5), std=0.5),
                           batch=2, prompt_len=256, chunk=64, capacity=512)
    p4 = W.make_chunked_prompt(wl, seed=61)
    p1 = W.make_chunked_prompt(W.PrefillWorkload(**{**wl.__dict__, "chunk": 256}), seed=61)
    o4, _, k4, v4, s4 = gpu_chunked(p4)
    o1, _, k1, v1, s1 = gpu_chunked(p1)
    assert s4 == 0 and s1 == 0
    assert torch.equal(k4.view(torch.int16), k1.view(torch.int16))
    assert torch.equal(v4.view(torch.int16), v1.view(torch.int16))
    assert_out_close(o4.double().numpy(), o1.double().numpy(), "chunked vs single")


def test_empty_chunk_is_noop():
    import causal_gqa_attention_rope_gb300 as na
    from harness import attn_cfg
    spec = W.Spec(H=4, KV=2, d=64, rd=64)
    dev = "cuda"
    k = W.sentinel_fill((1, 2, 8, 64)).to(dev)
    cache = na.KVCache(k, k.clone())
    e = torch.empty(0, 4, 64, dtype=torch.bfloat16, device=dev)
    na.na_attn_prefill_chunk(attn_cfg(spec), torch.zeros(2, dtype=torch.int32, device=dev),
                             torch.zeros(1, dtype=torch.int32, device=dev), 0, 0, e, cache, e,
                             total_tokens=0)
    torch.cuda.synchronize()


# ---------------------------------------------------- full-size workloads --

def _chunked_full(oracle, wl, n_rows, seed=0):
    prompt = W.make_chunked_prompt(wl, seed=seed)
    out, q_rot, ck, cv, status = gpu_chunked(prompt)
    assert status == 0
    step = prompt_as_step(prompt)
    ost = oracle_append(oracle, step)
    # cache of the whole prompt: every slot within 1 ulp, the rest untouched
    from harness import assert_within_ulp
    L = prompt.prompt_len
    assert_within_ulp(ck[:, :, :L], ost.cache_k[:, :, :L], "cache K (full prompt)")
    assert np.array_equal(cv[:, :, :L].double().numpy(), ost.cache_v[:, :, :L])
    assert bool((ck[:, :, L:].contiguous().view(torch.int16) == W.SENTINEL_BITS).all())
    # sampled rows: first and last row of every chunk plus seeded random rows
    rows = set()
    for c in range(prompt.num_chunks):
        lo, hi = prompt.chunk_bounds(c)
        rows.update((lo, hi - 1))
    rows.update(sample_rows(L, n_rows, seed=7))
    rows = sorted(rows)
    ref = oracle_rows(oracle, step, ost, rows)
    got = out[0, rows].double().numpy()
    return assert_out_close(got, ref, wl.name)


def test_full_chunked_prefill_h32kv8_t4096_chunk128(oracle):
    _chunked_full(oracle, W.C2, n_rows=24)


def test_full_yarn_prefill_h40kv8_rd64_t32768_chunk2048(oracle):
    _chunked_full(oracle, W.C4, n_rows=6)


def test_full_varlen_step_b16_qknorm_gate(oracle):
    step = W.make_varlen_step(W.C5, seed=0)
    rows = sample_rows(step.total_tokens, 40, seed=9)
    # also the first and last new token of every sequence
    cu = step.cu_seqlens.tolist()
    for b in range(step.batch):
        if cu[b + 1] > cu[b]:
            rows += [cu[b], cu[b + 1] - 1]
    _compare_step(oracle, step, rows=sorted(set(rows)), what="varlen full")


def test_pair_equals_two_sequential_calls():
    """The pages' pair test on the GPU: two drafted tokens per sequence in one
    call against the same tokens in two one-token calls (append, attend, then
    the next): the caches are bit-identical and every output row agrees within
    the output tolerance (the two calls tile and split the keys differently)."""
    import causal_gqa_attention_rope_gb300 as na
    from harness import attn_cfg, rope_cfg
    spec = W.Spec(H=32, KV=8, d=128, rd=128, qk_norm=True, out_gate=True,
                  rope=W.RopeParams(base=5e5))
    prior = [700, 64, 2048, 1]
    B = len(prior)
    step = W.make_step(spec, prior, [2] * B, 2176, seed=221)
    dev = "cuda"
    cfg, rope = attn_cfg(spec), rope_cfg(spec)
    dv = lambda x: None if x is None else x.to(dev).contiguous()
    qw, kw = dv(step.q_norm_w), dv(step.k_norm_w)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def run(cache, cu, lens, q, k, v, gate, n_max):
        T = q.shape[0]
        q_out, out = torch.empty_like(q), torch.empty_like(q)
        na.na_rope_append_kv(cfg, rope, cu, lens, q, k, v, q_out, cache, q_norm_w=qw, k_norm_w=kw,
                             status=st)
        mt = int(lens.max()) + n_max
        ws = na.workspace(na.na_prefill_workspace_size(cfg, B, T, n_max, mt), dev)
        na.na_attn_prefill_chunk(cfg, cu, lens, n_max, mt, q_out, cache, out, gate=gate,
                                 workspace=ws, status=st)
        return out

    # one call: both drafted tokens of every sequence
    pair_cache = na.KVCache(dv(step.cache_k), dv(step.cache_v))
    out_pair = run(pair_cache, dv(step.cu_seqlens), dv(step.cache_lens), dv(step.q), dv(step.k),
                   dv(step.v), dv(step.gate), 2).cpu()
    # two calls of one token per sequence
    seq_cache = na.KVCache(dv(step.cache_k), dv(step.cache_v))
    cu1 = torch.arange(B + 1, dtype=torch.int32, device=dev)
    outs = []
    for i in range(2):
        pick = lambda x: x[i::2].contiguous().to(dev)  # token i of every sequence
        lens = torch.tensor([p + i for p in prior], dtype=torch.int32, device=dev)
        outs.append(run(seq_cache, cu1, lens, pick(step.q), pick(step.k), pick(step.v),
                        pick(step.gate), 1).cpu())
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(pair_cache.k.cpu().view(torch.int16), seq_cache.k.cpu().view(torch.int16))
    assert torch.equal(pair_cache.v.cpu().view(torch.int16), seq_cache.v.cpu().view(torch.int16))
    for i in range(2):
        assert_out_close(out_pair[i::2].double().numpy(), outs[i].double().numpy(),
                         f"drafted token {i}: pair against single calls")


def test_prefill_many_short_sequences(oracle):
    """200 sequences of 0..20 new tokens over 0..2000 cached ones in one call
    (many partly filled GQA-packed tiles; more than 32 sequences, so the slots
    are not ranked): twelve sequences against the oracle, row by row and slot
    by slot."""
    rng = np.random.default_rng(241)
    B = 200
    prior = [int(x) for x in rng.integers(0, 2001, B)]
    new = [int(x) for x in rng.integers(0, 21, B)]
    spec = W.Spec(H=16, KV=4, d=128, rd=128, qk_norm=True, out_gate=True,
                  rope=W.RopeParams(base=1e6))
    step = W.make_step(spec, prior, new, 2048, seed=243)
    g = gpu_step(step)
    assert g.status == 0, f"status {g.status}"
    assert bool(torch.isfinite(g.out.float()).all())
    idx = sorted({int(np.argmax(new)), int(np.argmax(prior))} |
                 {b for b in sample_rows(B, 10, seed=245) if new[b] > 0})
    sub, rows = _sequences_of(step, idx)
    ost = oracle_append(oracle, sub)
    check_cache(g.cache_k[idx], g.cache_v[idx], sub, ost)
    ref = oracle_rows(oracle, sub, ost, list(range(sub.total_tokens)))
    assert_out_close(g.out[rows].to(torch.float64).numpy(), ref, f"sequences {idx}")

"""Conditions only the device can see, reported in the caller's status word:
a sequence longer than the host's max_new_len bound, a chunk reaching past
the host's max_total_len bound, and a decode (or importance) length past
max_kv_len.  The offending sequence is skipped -- its outputs untouched
(prefill), zeroed (decode), its probabilities and importance unwritten --
and every other sequence of the call is still computed exactly as the oracle
says."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import (Guarded, assert_out_close, assert_probs_close, attn_cfg, check_cache,
                     oracle_append, oracle_flags, oracle_rows, rope_cfg, score_scale)

pytestmark = pytest.mark.gpu

FILL = -7.0  # exactly representable in bf16 and fp32: marks outputs never written


def _append_and_attend(step, max_new_len, max_total_len):
    """The step's append (valid), then its attention call with the given host
    bounds; returns (out, cache_k, cache_v, append status, attention status)."""
    import causal_gqa_attention_rope_gb300 as na
    s, dev = step.spec, "cuda"
    dv = lambda x: None if x is None else x.to(dev).contiguous()
    cfg = attn_cfg(s)
    cu, lens = dv(step.cu_seqlens), dv(step.cache_lens)
    cache = na.KVCache(dv(step.cache_k), dv(step.cache_v))
    q = dv(step.q)
    q_out = torch.empty_like(q)
    st_append = torch.zeros(1, dtype=torch.int32, device=dev)
    st_attn = torch.zeros(1, dtype=torch.int32, device=dev)
    na.na_rope_append_kv(cfg, rope_cfg(s), cu, lens, q, dv(step.k), dv(step.v), q_out, cache,
                         q_norm_w=dv(step.q_norm_w), k_norm_w=dv(step.k_norm_w), status=st_append)
    T = step.total_tokens
    go = Guarded(q.shape, q.dtype, dev, fill=FILL)
    ws = na.workspace(na.na_prefill_workspace_size(cfg, step.batch, T, max_new_len,
                                                   max_total_len), dev)
    na.na_attn_prefill_chunk(cfg, cu, lens, max_new_len, max_total_len, q_out, cache, go.t,
                             gate=dv(step.gate), workspace=ws, status=st_attn, total_tokens=T)
    torch.cuda.synchronize()
    go.check("out")
    return (go.t.cpu(), cache.k.cpu(), cache.v.cpu(), int(st_append.item()),
            int(st_attn.item()))


def _check_rows(oracle, step, out, good_seqs, bad_seqs, what):
    cu = step.cu_seqlens.tolist()
    ost = oracle_append(oracle, step)
    rows = [t for b in good_seqs for t in range(cu[b], cu[b + 1])]
    ref = oracle_rows(oracle, step, ost, rows)
    assert_out_close(out[rows].to(torch.float64).numpy(), ref, what)
    for b in bad_seqs:
        assert bool((out[cu[b]:cu[b + 1]] == FILL).all()), f"{what}: skipped sequence {b} written"
    return ost


@pytest.mark.parametrize("gate", [False, True])
def test_prefill_sequence_past_max_new_len(oracle, gate):
    """Sequence 1 brings 40 tokens against a host bound of 16: NA_ERR_INVALID_ARG,
    its rows untouched; sequences 0 and 2 are attended as usual."""
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=8, KV=2, d=128, rd=128, out_gate=gate)
    step = W.make_step(spec, [300, 20, 700], [5, 40, 16], 1024, seed=71)
    out, ck, cv, sa, sb = _append_and_attend(step, max_new_len=16, max_total_len=716)
    assert sa == 0
    assert sb == na.NA_ERR_INVALID_ARG
    ost = _check_rows(oracle, step, out, [0, 2], [1], "past max_new_len")
    check_cache(ck, cv, step, ost)  # the append itself was valid


def test_prefill_chunk_past_max_total_len(oracle):
    """Sequence 1 ends at position 160 but the host bound says 150 (within the
    capacity, so the host accepts it): NA_ERR_CAPACITY, its rows untouched;
    sequence 0 is attended as usual."""
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=4, KV=1, d=64, rd=64)
    step = W.make_step(spec, [100, 130], [50, 30], 256, seed=73)
    out, ck, cv, sa, sb = _append_and_attend(step, max_new_len=50, max_total_len=150)
    assert sa == 0
    assert sb == na.NA_ERR_CAPACITY
    _check_rows(oracle, step, out, [0], [1], "past max_total_len")


def test_decode_length_past_max_kv_len(oracle):
    """kv_lens [300, 900, 0, 64] against max_kv_len 512: NA_ERR_CAPACITY, the
    900-key sequence's output zeroed and its probabilities unwritten; the
    others match the oracle.  The importance pass over the same lengths
    reports the same and leaves that sequence's running score alone."""
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=8, KV=2, d=128, rd=128)
    lens = [300, 900, 0, 64]
    dec = W.make_decode(spec, lens, 1024, seed=75)
    dev, mx = "cuda", 512
    cfg = attn_cfg(spec)
    B = len(lens)
    q = dec.q.to(dev)
    go = Guarded(q.shape, q.dtype, dev, fill=FILL)
    gp = Guarded((B, spec.H, mx), torch.float32, dev, fill=FILL)
    ws = na.workspace(na.na_decode_workspace_size(cfg, B, mx), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kv = dec.kv_lens.to(dev)
    na.na_attn_decode(cfg, q, na.KVCache(dec.cache_k.to(dev), dec.cache_v.to(dev)), kv, mx,
                      go.t, probs=gp.t, workspace=ws, status=status)
    torch.cuda.synchronize()
    go.check("decode out")
    gp.check("decode probs")
    assert int(status.item()) == na.NA_ERR_CAPACITY
    out, probs = go.t.cpu(), gp.t.cpu()
    assert bool((out[1] == 0).all()), "the skipped sequence's output is zero"
    assert bool((probs[1] == FILL).all()), "the skipped sequence's probabilities were written"
    good = [0, 2, 3]
    ref_out, ref_p = oracle.decode(
        spec.H, spec.KV, spec.d, score_scale(spec), oracle_flags(spec, False),
        W.bf16_to_f64(dec.q[good]), np.ascontiguousarray(W.bf16_to_f64(dec.cache_k[good])),
        np.ascontiguousarray(W.bf16_to_f64(dec.cache_v[good])), dec.kv_lens[good].numpy(),
        probs_stride=mx)
    assert_out_close(out[good].double().numpy(), ref_out, "decode, other sequences")
    for i, b in enumerate(good):
        n = lens[b]
        assert_probs_close(probs[b, :, :n].numpy(), ref_p[i, :, :n], f"probs b{b}")
        assert bool((probs[b, :, n:] == FILL).all())

    # importance over those probabilities, same lengths and bound
    init = torch.full((B, mx), 0.5, dtype=torch.float32)
    gi = Guarded((B, mx), torch.float32, dev, fill=init.to(dev))
    st2 = torch.zeros(1, dtype=torch.int32, device=dev)
    na.na_decode_importance(cfg, gp.t, kv, mx, gi.t, accumulate=True, status=st2)
    torch.cuda.synchronize()
    gi.check("importance")
    assert int(st2.item()) == na.NA_ERR_CAPACITY
    imp = gi.t.cpu()
    assert torch.equal(imp[1], init[1]), "the skipped sequence's importance changed"
    ref_imp = oracle.decode_importance(spec.H, ref_p, dec.kv_lens[good].numpy(),
                                       imp=init[good].double().numpy(), accumulate=True)
    for i, b in enumerate(good):
        n = lens[b]
        err = float(np.max(np.abs(imp[b, :n].double().numpy() - ref_imp[i, :n]))) if n else 0.0
        assert err <= spec.H * 1e-4, f"importance b{b}: {err:.3e}"
        assert torch.equal(imp[b, n:], init[b, n:])


def test_prefill_sequence_past_total_tokens(oracle):
    """cu_seqlens says 12 tokens while the call's total_tokens is 10: the
    second sequence (tokens 5..11) would reach past Q and out, so it is
    skipped and NA_ERR_INVALID_ARG written; the first is attended as usual and
    nothing is written outside out's 10 rows (its guard bands intact)."""
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=4, KV=2, d=64, rd=64)
    step = W.make_step(spec, [30, 8], [5, 7], 64, seed=77)
    dev = "cuda"
    cfg, rope = attn_cfg(spec), rope_cfg(spec)
    cu, lens = step.cu_seqlens.to(dev), step.cache_lens.to(dev)
    cache = na.KVCache(step.cache_k.to(dev), step.cache_v.to(dev))
    q = step.q.to(dev)
    q_out = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    na.na_rope_append_kv(cfg, rope, cu, lens, q, step.k.to(dev), step.v.to(dev), q_out, cache,
                         status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    T = 10
    go = Guarded((T, spec.H, spec.d), torch.bfloat16, dev, fill=FILL)
    ws = na.workspace(na.na_prefill_workspace_size(cfg, 2, T, 7, 38), dev)
    na.na_attn_prefill_chunk(cfg, cu, lens, 7, 38, q_out[:T], cache, go.t, workspace=ws,
                             status=st, total_tokens=T)
    torch.cuda.synchronize()
    go.check("out")
    assert int(st.item()) == na.NA_ERR_INVALID_ARG
    out = go.t.cpu()
    ost = oracle_append(oracle, step)
    ref = oracle_rows(oracle, step, ost, list(range(5)))
    assert_out_close(out[:5].to(torch.float64).numpy(), ref, "first sequence")
    assert bool((out[5:] == FILL).all()), "the skipped sequence's rows were written"


def test_loose_host_bounds(oracle):
    """Host bounds far above the real lengths, as a serving loop that passes
    its capacities: max_new_len 1024 for chunks of 100 and 30 tokens and
    max_total_len 131072 over histories of 300 and 50 (the key ranges are cut
    for a 131072-key span, so nearly every piece has no keys), and a decode
    with max_kv_len 131072 over 20..700 keys: every row against the oracle."""
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=8, KV=2, d=128, rd=128, out_gate=True)
    step = W.make_step(spec, [300, 50], [100, 30], 131072, seed=79)
    out, ck, cv, sa, sb = _append_and_attend(step, max_new_len=1024, max_total_len=131072)
    assert sa == 0 and sb == 0
    ost = _check_rows(oracle, step, out, [0, 1], [], "loose bounds")
    check_cache(ck, cv, step, ost)

    dec = W.make_decode(spec, [700, 20, 333], 131072, seed=81)
    dev, mx = "cuda", 131072
    cfg = attn_cfg(spec)
    q = dec.q.to(dev)
    go = Guarded(q.shape, q.dtype, dev)
    gp = Guarded((3, spec.H, mx), torch.float32, dev, fill=FILL)
    ws = na.workspace(na.na_decode_workspace_size(cfg, 3, mx), dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    na.na_attn_decode(cfg, q, na.KVCache(dec.cache_k.to(dev), dec.cache_v.to(dev)),
                      dec.kv_lens.to(dev), mx, go.t, probs=gp.t, gate=dec.gate.to(dev),
                      workspace=ws, status=st)
    torch.cuda.synchronize()
    go.check("decode out")
    gp.check("decode probs")
    assert int(st.item()) == 0
    ref_out, ref_p = oracle.decode(
        spec.H, spec.KV, spec.d, score_scale(spec), oracle_flags(spec, False),
        W.bf16_to_f64(dec.q), np.ascontiguousarray(W.bf16_to_f64(dec.cache_k[:, :, :700])),
        np.ascontiguousarray(W.bf16_to_f64(dec.cache_v[:, :, :700])), dec.kv_lens.numpy(),
        gate=W.bf16_to_f64(dec.gate), probs_stride=mx)
    assert_out_close(go.t.cpu().double().numpy(), ref_out, "decode, loose bound")
    probs = gp.t.cpu()
    for b, n in enumerate([700, 20, 333]):
        assert_probs_close(probs[b, :, :n].numpy(), ref_p[b, :, :n], f"probs b{b}")
        assert bool((probs[b, :, n:] == FILL).all())

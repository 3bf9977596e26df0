"""Seeded random sweeps of the attention calls against the oracle: shapes, head
groupings, lengths, options (window, soft cap, gate, norms, partial rotary)
and strides drawn from a fixed generator, so that combinations the hand-picked
cases do not name are exercised too.  Every case is deterministic.  Inputs are
unit-scale (std 0.5 or 1), the scale the fixed max-abs bound of 2e-2 is meant
for: with std 2 outputs reach |6| and one bf16 ulp there is already 0.031 (the
exact f64 result rounded to bf16 alone is off by 0.015)."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import (PROBS_MAX_ABS, Guarded, assert_out_close, assert_probs_close,
                     assert_within_ulp, attn_cfg, check_cache, gpu_decode, gpu_step, oracle_append,
                     oracle_flags, oracle_rows, ring_from_linear, rope_cfg, score_scale)

pytestmark = pytest.mark.gpu

HEADS = [(4, 1), (8, 2), (6, 2), (12, 4), (16, 2), (5, 5), (10, 2), (32, 8), (24, 3)]


def _random_spec(rng, decode: bool) -> W.Spec:
    H, KV = HEADS[rng.integers(len(HEADS))]
    d = int(rng.choice([64, 128]))
    rd = int(rng.choice([d, d // 2, 16 * int(rng.integers(1, d // 16 + 1))]))
    yarn = bool(rng.random() < 0.3)
    rope = W.RopeParams(base=float(rng.choice([1e4, 5e5, 1e6])), yarn=yarn,
                        factor=4.0 if yarn else 1.0, orig_max_pos=2048 if yarn else 0)
    return W.Spec(H=H, KV=KV, d=d, rd=rd, rope=rope,
                  qk_norm=bool(rng.random() < 0.3) and not decode,
                  v_norm=bool(rng.random() < 0.2) and not decode,
                  out_gate=bool(rng.random() < 0.4),
                  softcap=float(rng.choice([0.0, 0.0, 15.0, 50.0])),
                  window=int(rng.choice([0, 0, 0, int(rng.integers(1, 700))])),
                  std=float(rng.choice([0.5, 1.0])))


@pytest.mark.parametrize("seed", range(24))
def test_random_prefill_steps(oracle, seed):
    """A few sequences with random histories and new-token counts (some empty)
    through append + attend; every row compared with the oracle."""
    rng = np.random.default_rng(1000 + seed)
    spec = _random_spec(rng, decode=False)
    B = int(rng.integers(1, 5))
    prior = [int(x) for x in rng.integers(0, 600, B)]
    new = [int(x) for x in rng.integers(0, 160, B)]
    if sum(new) == 0:
        new[0] = 1
    capacity = (max(p + n for p, n in zip(prior, new)) + 127) // 128 * 128 + 128
    step = W.make_step(spec, prior, new, capacity, seed=2000 + seed)
    g = gpu_step(step)
    assert g.status == 0, f"status {g.status}"
    ost = oracle_append(oracle, step)
    check_cache(g.cache_k, g.cache_v, step, ost)
    rows = list(range(step.total_tokens))
    ref = oracle_rows(oracle, step, ost, rows)
    assert_out_close(g.out[rows].to(torch.float64).numpy(), ref,
                     f"seed {seed}: {spec.H}/{spec.KV} d{spec.d} rd{spec.rd} prior {prior} new {new}")


@pytest.mark.parametrize("seed", range(24))
def test_random_decode_steps(oracle, seed):
    """Random batch, lengths (0 included), options, key splits and probability
    strides (multiples of 4 or not); outputs and every probability compared,
    then the Born-rule importance of those probabilities, accumulated onto a
    random running score."""
    rng = np.random.default_rng(3000 + seed)
    spec = _random_spec(rng, decode=True)
    B = int(rng.integers(1, 9))
    lens = [int(x) for x in rng.integers(0, 2500, B)]
    if rng.random() < 0.3:
        lens[int(rng.integers(B))] = 0
    capacity = max(max(lens), 1) + int(rng.integers(0, 64))
    dec = W.make_decode(spec, lens, capacity, seed=4000 + seed)
    splits = int(rng.choice([0, 0, 1, 3, 7]))
    stride = max(max(lens), 1) + int(rng.integers(0, 6))
    out, probs, status = gpu_decode(dec, num_splits=splits, probs_stride=stride)
    assert status == 0
    s = dec.spec
    ref_out, ref_p = oracle.decode(s.H, s.KV, s.d, score_scale(s), oracle_flags(s),
                                   W.bf16_to_f64(dec.q),
                                   np.ascontiguousarray(W.bf16_to_f64(dec.cache_k)),
                                   np.ascontiguousarray(W.bf16_to_f64(dec.cache_v)),
                                   dec.kv_lens.numpy(), gate=W.bf16_to_f64(dec.gate),
                                   probs_stride=stride, softcap=s.softcap, window=s.window)
    what = f"seed {seed}: {s.H}/{s.KV} d{s.d} lens {lens} splits {splits} stride {stride}"
    assert_out_close(out.double().numpy(), ref_out, what)
    for b, n in enumerate(lens):
        assert_probs_close(probs[b, :, :n].numpy(), ref_p[b, :, :n], f"{what} probs b{b}")
        assert bool((probs[b, :, n:] == -7.0).all()), "probs written past kv_len"

    import causal_gqa_attention_rope_gb300 as na
    init = torch.rand((B, stride), generator=torch.Generator().manual_seed(seed))
    gi = Guarded((B, stride), torch.float32, "cuda", fill=init.to("cuda"))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    na.na_decode_importance(attn_cfg(s), probs.to("cuda"), dec.kv_lens.to("cuda"),
                            max(max(lens), 1), gi.t, accumulate=True, status=st)
    torch.cuda.synchronize()
    gi.check("importance")
    assert int(st.item()) == 0
    ref_imp = oracle.decode_importance(s.H, ref_p, dec.kv_lens.numpy(),
                                       imp=init.double().numpy(), accumulate=True)
    got = gi.t.cpu()
    for b, n in enumerate(lens):
        err = float(np.max(np.abs(got[b, :n].double().numpy() - ref_imp[b, :n]))) if n else 0.0
        assert err <= s.H * PROBS_MAX_ABS, f"{what} importance b{b}: {err:.3e}"
        assert torch.equal(got[b, n:], init[b, n:]), "importance written past kv_len"


@pytest.mark.parametrize("seed", range(8))
def test_random_decode_ring(oracle, seed):
    """A ring cache (capacity a multiple of 64 holding at least the window) with
    random windows and lengths up to three times the ring: windows cross the
    ring's end at random places."""
    import causal_gqa_attention_rope_gb300 as na
    rng = np.random.default_rng(5000 + seed)
    spec = _random_spec(rng, decode=True)
    spec.window = int(rng.integers(1, 600))
    R = (spec.window + int(rng.integers(0, 300)) + 63) // 64 * 64
    B = int(rng.integers(1, 7))
    lens = [int(x) for x in rng.integers(0, 3 * R, B)]
    dec = W.make_decode(spec, lens, max(max(lens), 1), seed=6000 + seed)
    rk = ring_from_linear(oracle, dec.cache_k, lens, R)
    rv = ring_from_linear(oracle, dec.cache_v, lens, R)
    cfg = attn_cfg(spec)
    cfg.ring_cache = True
    dev = "cuda"
    q = dec.q.to(dev)
    mx = max(max(lens), 1)
    go = Guarded(q.shape, q.dtype, dev)
    gp = Guarded((B, spec.H, mx), torch.float32, dev, fill=-7.0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = na.workspace(na.na_decode_workspace_size(cfg, B, mx), dev)
    gate = None if dec.gate is None else dec.gate.to(dev)
    na.na_attn_decode(cfg, q, na.KVCache(rk.to(dev), rv.to(dev)), dec.kv_lens.to(dev), mx, go.t,
                      probs=gp.t, gate=gate, workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.check("ring decode out")
    gp.check("ring decode probs")
    s = dec.spec
    ref_out, ref_p = oracle.decode(s.H, s.KV, s.d, score_scale(s), oracle_flags(s, True),
                                   W.bf16_to_f64(dec.q), np.ascontiguousarray(W.bf16_to_f64(rk)),
                                   np.ascontiguousarray(W.bf16_to_f64(rv)), dec.kv_lens.numpy(),
                                   gate=W.bf16_to_f64(dec.gate), probs_stride=mx,
                                   softcap=s.softcap, window=s.window)
    what = f"seed {seed}: ring {R} window {s.window} {s.H}/{s.KV} d{s.d} lens {lens}"
    assert_out_close(go.t.cpu().double().numpy(), ref_out, what)
    probs = gp.t.cpu()
    for b, n in enumerate(lens):
        assert_probs_close(probs[b, :, :n].numpy(), ref_p[b, :, :n], f"{what} probs b{b}")


@pytest.mark.parametrize("seed", range(16))
def test_random_rope_append(oracle, seed):
    """Any even rotary dim (the register and the staged kernel), both qk-norm
    styles, V-norm, YaRN factors, explicit attention factors and positions up
    to 20000: rotated Q and K within 1 ulp, V and untouched slots bit for bit."""
    rng = np.random.default_rng(7000 + seed)
    H, KV = HEADS[rng.integers(len(HEADS))]
    d = int(rng.choice([64, 128]))
    rd = int(rng.choice([0, d, 2 * int(rng.integers(1, d // 2 + 1))]))
    yarn = bool(rng.random() < 0.5)
    rope = W.RopeParams(base=float(rng.choice([1e4, 5e5, 1e6])), yarn=yarn,
                        factor=float(rng.choice([2.0, 4.0, 8.0])) if yarn else 1.0,
                        orig_max_pos=int(rng.choice([2048, 4096, 8192])) if yarn else 0,
                        attn_factor=float(rng.choice([0.0, 0.0, 1.0, 0.75, 1.25])))
    qk = bool(rng.random() < 0.5)
    zc = qk and bool(rng.random() < 0.5)
    spec = W.Spec(H=H, KV=KV, d=d, rd=rd, rope=rope, qk_norm=qk, qk_norm_zero_centered=zc,
                  v_norm=bool(rng.random() < 0.4), eps=float(rng.choice([1e-6, 1e-5])),
                  norm_w_mean=0.0 if zc else 1.0)
    B = int(rng.integers(1, 5))
    prior = [int(x) for x in rng.integers(0, 20000, B)]
    new = [int(x) for x in rng.integers(0, 48, B)]
    if sum(new) == 0:
        new[0] = 1
    capacity = max(p + n for p, n in zip(prior, new))
    # the history itself is never read by the append: sentinel slots stand in
    step = W.make_step(spec, prior, new, capacity, seed=8000 + seed, history=False)
    import causal_gqa_attention_rope_gb300 as na
    dev = lambda x: None if x is None else x.to("cuda").contiguous()
    cache = na.KVCache(dev(step.cache_k), dev(step.cache_v))
    gq = Guarded(step.q.shape, step.q.dtype, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    na.na_rope_append_kv(attn_cfg(spec), rope_cfg(spec), dev(step.cu_seqlens),
                         dev(step.cache_lens), dev(step.q), dev(step.k), dev(step.v), gq.t, cache,
                         q_norm_w=dev(step.q_norm_w), k_norm_w=dev(step.k_norm_w), status=status,
                         total_tokens=step.total_tokens)
    torch.cuda.synchronize()
    gq.check("q_out")
    assert int(status.item()) == 0
    ost = oracle_append(oracle, step)
    assert_within_ulp(gq.t.cpu(), ost.q_rot, f"seed {seed} rd {rd}: rotated Q")
    check_cache(cache.k.cpu(), cache.v.cpu(), step, ost)


@pytest.mark.parametrize("seed", range(8))
def test_random_prefill_ring(oracle, seed):
    """Append + attend on a ring cache (capacity a multiple of 128 holding at
    least window + chunk - 1 positions) with random windows, histories up to
    three times the ring and chunks of up to 160 tokens, so both the appended
    slots and the windows wrap around the ring's end at random places; every
    row against the oracle attending the same ring, the ring slot by slot."""
    import causal_gqa_attention_rope_gb300 as na
    rng = np.random.default_rng(9000 + seed)
    spec = _random_spec(rng, decode=False)
    spec.window = int(rng.integers(1, 600))
    B = int(rng.integers(1, 4))
    new = [int(x) for x in rng.integers(0, 161, B)]
    if sum(new) == 0:
        new[0] = 1
    R = (spec.window + max(new) - 1 + int(rng.integers(0, 200)) + 127) // 128 * 128
    prior = [int(x) for x in rng.integers(0, 3 * R, B)]
    step = W.make_step(spec, prior, new, max(p + n for p, n in zip(prior, new)), seed=9100 + seed)
    ck = ring_from_linear(oracle, step.cache_k, prior, R)
    cv = ring_from_linear(oracle, step.cache_v, prior, R)
    ring_step = W.StepInputs(**{**step.__dict__, "cache_k": ck, "cache_v": cv})
    cfg = attn_cfg(spec)
    cfg.ring_cache = True
    dev = "cuda"
    dv = lambda x: None if x is None else x.to(dev).contiguous()
    cache = na.KVCache(ck.clone().to(dev), cv.clone().to(dev))
    q = dv(step.q)
    gq, go = Guarded(q.shape, q.dtype, dev), Guarded(q.shape, q.dtype, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    cu, lens = dv(step.cu_seqlens), dv(step.cache_lens)
    T = step.total_tokens
    max_new, max_tot = max(new), max(p + n for p, n in zip(prior, new))
    na.na_rope_append_kv(cfg, rope_cfg(spec), cu, lens, q, dv(step.k), dv(step.v), gq.t, cache,
                         q_norm_w=dv(step.q_norm_w), k_norm_w=dv(step.k_norm_w), status=status)
    ws = na.workspace(na.na_prefill_workspace_size(cfg, B, T, max_new, max_tot), dev)
    na.na_attn_prefill_chunk(cfg, cu, lens, max_new, max_tot, gq.t, cache, go.t, gate=dv(step.gate),
                             workspace=ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gq.check("ring q_out")
    go.check("ring out")
    what = (f"seed {seed}: ring {R} window {spec.window} {spec.H}/{spec.KV} d{spec.d} "
            f"rd{spec.rd} prior {prior} new {new}")
    ost = oracle_append(oracle, ring_step, ring=True)
    assert_within_ulp(gq.t.cpu(), ost.q_rot, f"{what}: rotated Q")
    ref = oracle_rows(oracle, ring_step, ost, list(range(T)), ring=True)
    assert_out_close(go.t.cpu().double().numpy(), ref, what)
    gk, gv = cache.k.cpu(), cache.v.cpu()
    for b in range(B):
        written = sorted({oracle.ring_slot(p, R) for p in range(prior[b], prior[b] + new[b])})
        kept = sorted(set(range(R)) - set(written))
        if written:
            assert_within_ulp(gk[b][:, written], ost.cache_k[b][:, written], f"{what}: ring K b{b}")
            if spec.v_norm:
                assert_within_ulp(gv[b][:, written], ost.cache_v[b][:, written], f"{what}: ring V b{b}")
            else:
                assert np.array_equal(gv[b][:, written].double().numpy(), ost.cache_v[b][:, written])
        assert torch.equal(gk[b][:, kept].view(torch.int16), ck[b][:, kept].view(torch.int16))
        assert torch.equal(gv[b][:, kept].view(torch.int16), cv[b][:, kept].view(torch.int16))

"""Parity of split-KV decode (output and per-key probabilities) with the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import (Guarded, assert_out_close, assert_probs_close, gpu_decode, oracle_flags,
                     sample_rows, score_scale)

pytestmark = pytest.mark.gpu


def _oracle_decode(oracle, dec, rows_bh=None, stride=None, ring=False):
    s = dec.spec
    return oracle.decode(s.H, s.KV, s.d, score_scale(s), oracle_flags(s, ring), W.bf16_to_f64(dec.q),
                         np.ascontiguousarray(W.bf16_to_f64(dec.cache_k)),
                         np.ascontiguousarray(W.bf16_to_f64(dec.cache_v)), dec.kv_lens.numpy(),
                         gate=W.bf16_to_f64(dec.gate), probs_stride=stride, rows_bh=rows_bh,
                         softcap=s.softcap, window=s.window)


def _check(oracle, dec, num_splits=0, with_probs=True):
    s = dec.spec
    out, probs, status = gpu_decode(dec, with_probs=with_probs, num_splits=num_splits)
    assert status == 0
    stride = probs.shape[-1] if probs is not None else None
    ref_out, ref_p = _oracle_decode(oracle, dec, stride=stride)
    assert_out_close(out.double().numpy(), ref_out, "decode out")
    if with_probs:
        lens = dec.kv_lens.tolist()
        for b, n in enumerate(lens):
            assert_probs_close(probs[b, :, :n].numpy(), ref_p[b, :, :n], f"probs b{b}")
            assert bool((probs[b, :, n:] == -7.0).all()), "probs written past kv_len"


def _assert_probs_relative(gpu, ref, what):
    """Each probability within 1e-4 of its own value (plus 1e-9).  Over
    thousands of keys the probabilities are ~1e-4..1e-5 and the fixed max-abs
    bound says little; with unit-scale inputs a score is off by ~1e-6, which
    moves its probability by ~1e-6 of itself (1.5e-6 the worst measured at
    131072 keys), and a missing, doubled or misplaced key moves it by far
    more."""
    g, r = gpu.double().numpy(), ref
    bad = np.abs(g - r) > 1e-4 * r + 1e-9
    assert not bad.any(), (f"{what}: {int(bad.sum())} probabilities beyond 1e-4 relative; "
                           f"worst {float(np.max(np.abs(g - r) / (r + 1e-9))):.3e}")


SHAPES = {
    "h32kv8d128": W.Spec(H=32, KV=8, d=128, rd=128),
    "h4kv1d128_group4": W.Spec(H=4, KV=1, d=128, rd=128),
    "h8kv8d64_mha": W.Spec(H=8, KV=8, d=64, rd=64),
    "h10kv2d128_group5": W.Spec(H=10, KV=2, d=128, rd=128),
    "h16kv2d64_group8_gate": W.Spec(H=16, KV=2, d=64, rd=64, out_gate=True),
    "h4kv2d128_group2_scale": W.Spec(H=4, KV=2, d=128, rd=128, sm_scale=0.2),
    "h16kv2d128_group8": W.Spec(H=16, KV=2, d=128, rd=128),        # 8 heads per MMA
    "h32kv2d128_group16_softcap": W.Spec(H=32, KV=2, d=128, rd=128, softcap=30.0),  # 2 head chunks
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_decode_edge_lengths(oracle, name):
    dec = W.make_decode(SHAPES[name], [0, 1, 63, 64, 65, 700, 1500], 1536, seed=71)
    _check(oracle, dec)


@pytest.mark.parametrize("splits", [1, 3, 17])
def test_decode_forced_splits(oracle, splits):
    dec = W.make_decode(W.Spec(H=8, KV=2, d=128, rd=128), [1200, 5, 999], 1280, seed=81)
    _check(oracle, dec, num_splits=splits)


@pytest.mark.parametrize("splits", [0, 40])
def test_decode_balanced_slices_skip_empty_sequences(oracle, splits):
    """Key slices that start inside runs of empty sequences, a batch wider than
    one warp's scan, and one long sequence cut across many slices."""
    lens = [0] * 37 + [3000] + [1, 0] * 15 + [0, 257, 0]
    dec = W.make_decode(W.Spec(H=8, KV=2, d=128, rd=128), lens, 3072, seed=93)
    _check(oracle, dec, num_splits=splits)


@pytest.mark.parametrize("name,spec", [
    ("plain", W.Spec(H=4, KV=1, d=128, rd=128)),
    ("window4096_gate", W.Spec(H=8, KV=1, d=64, rd=64, window=4096, out_gate=True)),
])
def test_decode_long_context(oracle, name, spec):
    """A 131072-key sequence beside a 50001-key one and a 1-key one: the long
    ones are cut into many equal key slices (pieces of one stream spread over
    most of the grid) and merged; with a window only its last 4096 keys count
    and every probability before them is 0."""
    dec = W.make_decode(spec, [131072, 50001, 1], 131072, seed=107)
    _check(oracle, dec)
    out, probs, status = gpu_decode(dec, with_probs=True)
    assert status == 0
    _, ref_p = _oracle_decode(oracle, dec, stride=probs.shape[-1])
    for b, n in enumerate(dec.kv_lens.tolist()):
        _assert_probs_relative(probs[b, :, :n], ref_p[b, :, :n], f"{name} b{b}")


@pytest.mark.parametrize("name,spec", [
    ("softcap", W.Spec(H=8, KV=2, d=128, rd=128, softcap=20.0, std=2.0)),
    ("window256", W.Spec(H=8, KV=2, d=128, rd=128, window=256)),
    ("window1_d64_gate", W.Spec(H=16, KV=2, d=64, rd=64, window=1, out_gate=True)),
    ("window_softcap_mha", W.Spec(H=4, KV=4, d=128, rd=128, window=700, softcap=6.0)),
])
def test_decode_softcap_and_window(oracle, name, spec):
    """Soft-capped scores and sliding windows in the split/combine decode, with
    probabilities (0 before the window) and their importance."""
    dec = W.make_decode(spec, [0, 1, 5, 256, 257, 1500], 1536, seed=101)
    _check(oracle, dec)
    _check_importance(oracle, dec)


def test_decode_ring_cache(oracle):
    """Ring cache of 448 slots (seven 64-key tiles; not a multiple of the
    prefill's 128-key tile) with a window of 300: windows that cross the end of
    the ring continue at slot 0."""
    import causal_gqa_attention_rope_gb300 as na
    from harness import attn_cfg, ring_from_linear
    spec = W.Spec(H=8, KV=2, d=128, rd=128, window=300)
    lens = [0, 1, 299, 300, 301, 700, 1500]
    dec = W.make_decode(spec, lens, 1536, seed=107)
    R = 448
    dev = "cuda"
    cfg = attn_cfg(spec)
    cfg.ring_cache = True
    rk = ring_from_linear(oracle, dec.cache_k, lens, R)
    rv = ring_from_linear(oracle, dec.cache_v, lens, R)
    cache = na.KVCache(rk.to(dev), rv.to(dev))
    q = dec.q.to(dev)
    B, mx = len(lens), max(lens)
    go = Guarded(q.shape, q.dtype, dev)
    gp = Guarded((B, spec.H, mx), torch.float32, dev, fill=-7.0)
    out, probs = go.t, gp.t
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = na.workspace(na.na_decode_workspace_size(cfg, B, mx), dev)
    na.na_attn_decode(cfg, q, cache, dec.kv_lens.to(dev), mx, out, probs=probs, workspace=ws,
                      status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.check("ring decode out")
    gp.check("ring decode probs")
    # the oracle reads the same ring (key j in its ring slot of j)
    ring_dec = W.DecodeInputs(**{**dec.__dict__, "cache_k": rk, "cache_v": rv})
    ref_out, ref_p = _oracle_decode(oracle, ring_dec, stride=mx, ring=True)
    assert_out_close(out.cpu().double().numpy(), ref_out, "ring decode out")
    for b, n in enumerate(lens):
        assert_probs_close(probs[b, :, :n].cpu().numpy(), ref_p[b, :, :n], f"ring probs {b}")


def test_decode_without_probs(oracle):
    dec = W.make_decode(W.Spec(H=8, KV=2, d=128, rd=128, out_gate=True), [300, 64], 512, seed=91)
    _check(oracle, dec, with_probs=False)


def test_decode_equals_last_prefill_row():
    """Decode of the last token of a prefilled prompt equals that prefill row."""
    from harness import gpu_chunked
    wl = W.PrefillWorkload(name="t", spec=W.Spec(H=8, KV=2, d=128, rd=128), batch=1,
                           prompt_len=300, chunk=300, capacity=512)
    prompt = W.make_chunked_prompt(wl, seed=5)
    out, q_rot, ck, cv, status = gpu_chunked(prompt)
    assert status == 0
    dec = W.DecodeInputs(spec=wl.spec, q=q_rot[:, -1].contiguous(), cache_k=ck, cache_v=cv,
                         kv_lens=torch.tensor([300], dtype=torch.int32), gate=None)
    d_out, _, st = gpu_decode(dec, with_probs=False)
    assert st == 0
    assert_out_close(d_out.double().numpy(), out[:, -1].double().numpy(), "decode vs prefill")


def test_full_decode_b64_h32kv8_kv512to8192(oracle):
    """Full-size decode workload: every output row's probabilities sum to 1,
    and sampled (sequence, head) rows match the oracle in output and in every
    per-key probability."""
    dec = W.make_decode_workload(W.C3, seed=0)
    out, probs, status = gpu_decode(dec)
    assert status == 0
    lens = dec.kv_lens.tolist()
    B, H = dec.q.shape[0], dec.spec.H
    for b in range(B):
        n = lens[b]
        mass = probs[b, :, :n].double().sum(-1)
        assert torch.allclose(mass, torch.ones_like(mass), atol=1e-3), f"mass b{b}"
        assert bool((probs[b, :, n:] == -7.0).all())
    rows = sample_rows(B * H, 48, seed=13)
    ref_out, ref_p = _oracle_decode(oracle, dec, rows_bh=rows, stride=probs.shape[-1])
    for r in rows:
        b, h = divmod(r, H)
        assert_out_close(out[b, h].double().numpy(), ref_out[b, h], f"row {r}")
        assert_probs_close(probs[b, h, :lens[b]].numpy(), ref_p[b, h, :lens[b]], f"probs {r}")
        _assert_probs_relative(probs[b, h, :lens[b]], ref_p[b, h, :lens[b]], f"probs {r}")


# ----------------------------------------------------- Born-rule importance --

def _gpu_importance(dec, probs_cpu, imp_init, accumulate):
    import causal_gqa_attention_rope_gb300 as na
    from harness import attn_cfg
    dev = "cuda"
    gi = Guarded(tuple(imp_init.shape), torch.float32, dev, fill=imp_init.to(dev))
    imp = gi.t
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    max_kv = int(dec.kv_lens.max())
    na.na_decode_importance(attn_cfg(dec.spec), probs_cpu.to(dev), dec.kv_lens.to(dev), max_kv,
                            imp, accumulate=accumulate, status=status)
    torch.cuda.synchronize()
    gi.check("importance")
    return imp.cpu(), int(status.item())


def _check_importance(oracle, dec, probs_stride=None, accumulate=False):
    """GPU importance of the GPU probabilities against the oracle's importance
    of the oracle's probabilities: each probability is within PROBS_MAX_ABS, so
    each sum over H heads is within H * PROBS_MAX_ABS."""
    from harness import PROBS_MAX_ABS
    s = dec.spec
    _, probs, st = gpu_decode(dec, probs_stride=probs_stride)
    assert st == 0
    B, stride = probs.shape[0], probs.shape[-1]
    init = torch.full((B, stride), 0.25, dtype=torch.float32)
    if accumulate:
        init = torch.rand((B, stride), generator=torch.Generator().manual_seed(3))
    got, st = _gpu_importance(dec, probs, init, accumulate)
    assert st == 0
    _, ref_p = _oracle_decode(oracle, dec, stride=stride)
    ref = oracle.decode_importance(s.H, ref_p, dec.kv_lens.numpy(),
                                   imp=init.double().numpy(), accumulate=accumulate)
    lens = dec.kv_lens.tolist()
    for b, n in enumerate(lens):
        err = float(np.max(np.abs(got[b, :n].double().numpy() - ref[b, :n]))) if n else 0.0
        assert err <= s.H * PROBS_MAX_ABS, f"importance b{b}: {err:.3e}"
        assert torch.equal(got[b, n:], init[b, n:]), "importance written past kv_len"


@pytest.mark.parametrize("stride", [None, 1539])
def test_decode_importance(oracle, stride):
    """Sum over heads of the per-key probabilities (vector path; and an odd
    stride, the scalar path), empty and one-key sequences included."""
    dec = W.make_decode(W.Spec(H=8, KV=2, d=128, rd=128), [0, 1, 3, 700, 1500], 1536, seed=97)
    _check_importance(oracle, dec, probs_stride=stride)


@pytest.mark.parametrize("H,stride", [(5, 1028), (3, 1031), (40, 1028), (128, 1028),
                                      (200, 1032), (256, 1028), (300, 1028)])
def test_importance_head_counts(oracle, H, stride):
    """Importance alone, on given probabilities: head counts that do not split
    evenly over the load path's thread groups, ragged lengths around the
    blocks, a stride that is not a multiple of 4 (load path), head counts that
    shrink the tensor-map path's blocks to 128, 64 and 32 keys (40, 128,
    200/256 heads), one past its 256-row box (300 heads: load path), and
    accumulation."""
    gen = torch.Generator().manual_seed(H)
    lens = torch.tensor([0, 1, 255, 256, 257, 1027], dtype=torch.int32)
    B = lens.numel()
    probs = torch.rand((B, H, stride), generator=gen, dtype=torch.float32)
    init = torch.rand((B, stride), generator=gen, dtype=torch.float32)
    dec = W.DecodeInputs(spec=W.Spec(H=H, KV=1, d=64, rd=64), q=None, cache_k=None,
                         cache_v=None, kv_lens=lens, gate=None)
    got, st = _gpu_importance(dec, probs, init, True)
    assert st == 0
    ref = oracle.decode_importance(H, probs.double().numpy(), lens.numpy(),
                                   imp=init.double().numpy(), accumulate=True)
    for b, n in enumerate(lens.tolist()):
        # H fp32 additions of terms in [0, 1) (the start value included): in any
        # order the rounding error is at most H * 2^-24 * (H + 1)
        err = float(np.max(np.abs(got[b, :n].double().numpy() - ref[b, :n]))) if n else 0.0
        assert err <= H * (H + 1) * 2.0 ** -24, f"importance b{b}: {err:.3e}"
        assert torch.equal(got[b, n:], init[b, n:]), "importance written past kv_len"


def test_decode_importance_accumulates(oracle):
    dec = W.make_decode(W.Spec(H=16, KV=2, d=64, rd=64), [5, 64, 333], 512, seed=98)
    _check_importance(oracle, dec, accumulate=True)


def test_full_decode_importance_b64_h32kv8(oracle):
    """Importance of the full decode workload: every sequence totals H (each
    head's probabilities sum to one), and two sampled sequences match the
    oracle key by key."""
    from harness import PROBS_MAX_ABS
    dec = W.make_decode_workload(W.C3, seed=0)
    _, probs, st = gpu_decode(dec)
    assert st == 0
    B, H, stride = probs.shape
    got, st = _gpu_importance(dec, probs, torch.zeros(B, stride), False)
    assert st == 0
    lens = dec.kv_lens.tolist()
    for b, n in enumerate(lens):
        assert abs(float(got[b, :n].double().sum()) - H) < 1e-2, f"total b{b}"
    for b in sample_rows(B, 2, seed=17):
        rows = [b * H + h for h in range(H)]
        _, ref_p = _oracle_decode(oracle, dec, rows_bh=rows, stride=stride)
        ref = oracle.decode_importance(H, ref_p[b:b + 1], dec.kv_lens.numpy()[b:b + 1])
        n = lens[b]
        err = float(np.max(np.abs(got[b, :n].double().numpy() - ref[0, :n])))
        assert err <= H * PROBS_MAX_ABS, f"importance b{b}: {err:.3e}"


def test_calls_follow_the_current_stream(oracle):
    """With no stream argument the binding launches on the current stream, also
    inside a `torch.cuda.stream` block; the result is the same as on the default
    stream."""
    import causal_gqa_attention_rope_gb300 as na
    assert na._stream(None) == torch.cuda.current_stream().cuda_stream
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert na._stream(None) == side.cuda_stream
    dec = W.make_decode(W.Spec(H=8, KV=2, d=128, rd=128), [300, 77], capacity=320, seed=5)
    ref_out, _ = gpu_decode(dec, with_probs=False)[:2]
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        out, _, status = gpu_decode(dec, with_probs=False)
    torch.cuda.synchronize()
    assert status == 0
    assert torch.equal(out, ref_out)


def test_decode_many_sequences(oracle):
    """700 sequences of 0..600 keys (more streams than CTAs: a slice spans
    many short streams and many streams have a single piece); sampled
    sequences against the oracle, every output row finite, every probability
    row summing to 1."""
    rng = np.random.default_rng(231)
    lens = [int(x) for x in rng.integers(0, 601, 700)]
    spec = W.Spec(H=8, KV=2, d=64, rd=64, out_gate=True)
    dec = W.make_decode(spec, lens, 608, seed=233)
    out, probs, status = gpu_decode(dec, with_probs=True)
    assert status == 0
    assert bool(torch.isfinite(out.float()).all())
    for b, n in enumerate(lens):
        if n:
            mass = probs[b, :, :n].double().sum(-1)
            assert torch.allclose(mass, torch.ones_like(mass), atol=1e-4), f"mass b{b}"
        else:
            assert bool((out[b] == 0).all())
    idx = sorted(set(sample_rows(len(lens), 40, seed=235)))
    sub = W.DecodeInputs(spec=spec, q=dec.q[idx], cache_k=dec.cache_k[idx], cache_v=dec.cache_v[idx],
                         kv_lens=dec.kv_lens[idx], gate=dec.gate[idx])
    ref_out, ref_p = _oracle_decode(oracle, sub, stride=probs.shape[-1])
    assert_out_close(out[idx].double().numpy(), ref_out, "many sequences out")
    for i, b in enumerate(idx):
        n = lens[b]
        assert_probs_close(probs[b, :, :n].numpy(), ref_p[i, :, :n], f"many sequences probs b{b}")


@pytest.mark.parametrize("H,stride,lens", [(8, 40, [0, 1, 39, 40]), (32, 4, [4, 3, 1]),
                                           (4, 260, [259, 260, 7])])
def test_importance_short_strides(oracle, H, stride, lens):
    """Probability rows shorter than one 256-key block (40 and 4 keys) and
    just over one (260): the tensor-map path's box reaches past the rows (or
    the call takes the load path); every key against the oracle."""
    gen = torch.Generator().manual_seed(stride)
    kv = torch.tensor(lens, dtype=torch.int32)
    B = kv.numel()
    probs = torch.rand((B, H, stride), generator=gen, dtype=torch.float32)
    init = torch.rand((B, stride), generator=gen, dtype=torch.float32)
    dec = W.DecodeInputs(spec=W.Spec(H=H, KV=1, d=64, rd=64), q=None, cache_k=None,
                         cache_v=None, kv_lens=kv, gate=None)
    got, st = _gpu_importance(dec, probs, init, True)
    assert st == 0
    ref = oracle.decode_importance(H, probs.double().numpy(), kv.numpy(),
                                   imp=init.double().numpy(), accumulate=True)
    for b, n in enumerate(lens):
        err = float(np.max(np.abs(got[b, :n].double().numpy() - ref[b, :n]))) if n else 0.0
        assert err <= H * (H + 1) * 2.0 ** -24, f"importance b{b}: {err:.3e}"
        assert torch.equal(got[b, n:], init[b, n:])

"""The allocation-free decode entry point (na_attn_decode_static_ws).

It serves callers that cannot allocate device memory for a workspace (a
plugin inside a runtime that owns all device memory, a serving loop that may
not allocate once running): the split partials live in a fixed array inside
the library.  This file runs last so that a failure here leaves every other
test already run.  The checks, through the C ABI: two calls in a row give the
same output and probabilities as na_attn_decode with a caller workspace and
match the oracle within the parity tolerances; the largest batch whose
workspace fits the array is accepted and correct, one more sequence is
rejected."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from harness import (Guarded, assert_out_close, assert_probs_close, attn_cfg, oracle_flags,
                     score_scale)

pytestmark = pytest.mark.gpu

STATIC_BYTES = 20 * 2**20  # the array's size, as the header states it


def _run(dec, static: bool, splits: int):
    import causal_gqa_attention_rope_gb300 as na
    dev = "cuda"
    cfg = attn_cfg(dec.spec)
    B = dec.q.shape[0]
    max_kv = int(dec.kv_lens.max())
    q = dec.q.to(dev)
    cache = na.KVCache(dec.cache_k.to(dev), dec.cache_v.to(dev))
    kv = dec.kv_lens.to(dev)
    gate = None if dec.gate is None else dec.gate.to(dev)
    go = Guarded(q.shape, q.dtype, dev)
    gp = Guarded((B, dec.spec.H, max_kv), torch.float32, dev, fill=-7.0)
    out, probs = go.t, gp.t
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if static:
        na.na_attn_decode_static_ws(cfg, q, cache, kv, max_kv, out, probs=probs, gate=gate,
                                    num_splits=splits, status=status)
    else:
        ws = na.workspace(na.na_decode_workspace_size(cfg, B, max_kv, splits), dev)
        na.na_attn_decode(cfg, q, cache, kv, max_kv, out, probs=probs, gate=gate, workspace=ws,
                          num_splits=splits, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.check("static decode out")
    gp.check("static decode probs")
    return out.cpu(), probs.cpu()


def _oracle(oracle, dec, stride):
    s = dec.spec
    return oracle.decode(s.H, s.KV, s.d, score_scale(s), oracle_flags(s), W.bf16_to_f64(dec.q),
                         np.ascontiguousarray(W.bf16_to_f64(dec.cache_k)),
                         np.ascontiguousarray(W.bf16_to_f64(dec.cache_v)), dec.kv_lens.numpy(),
                         gate=W.bf16_to_f64(dec.gate), probs_stride=stride, window=s.window,
                         softcap=s.softcap)


def _check_probs(probs, ref_p, lens, what):
    for b, n in enumerate(lens):
        assert_probs_close(probs[b, :, :n].numpy(), np.asarray(ref_p[b, :, :n]), what)
        assert bool((probs[b, :, n:] == -7.0).all()), "probabilities written past kv_len"


def test_static_scratch_decode_matches_workspace_decode_and_oracle(oracle):
    spec = W.Spec(H=32, KV=8, d=128, rd=128, out_gate=True)
    cases = [W.make_decode(spec, [4096, 700, 1, 2500], 4096, seed=101),
             W.make_decode(W.Spec(H=8, KV=2, d=64, rd=64), [63, 2048, 0], 2048, seed=102)]
    for dec, splits in ((cases[0], 0), (cases[1], 5)):
        lens = dec.kv_lens.tolist()
        ref_out, ref_p = _run(dec, static=False, splits=splits)
        o_out, o_p = _oracle(oracle, dec, stride=max(lens))
        for _ in range(2):  # two calls in a row share the library's array
            out, probs = _run(dec, static=True, splits=splits)
            assert_out_close(out.double().numpy(), ref_out.double().numpy(), "static vs workspace")
            _check_probs(probs, ref_p, lens, "static vs workspace probs")
            assert_out_close(out.double().numpy(), o_out, "static vs oracle")
            _check_probs(probs, o_p, lens, "static vs oracle probs")


def _largest_batch_that_fits(na, cfg, max_kv):
    lo, hi = 1, 1
    while na.na_decode_workspace_size(cfg, hi, max_kv) <= STATIC_BYTES:
        lo, hi = hi, hi * 2
    while hi - lo > 1:  # invariant: lo fits, hi does not
        mid = (lo + hi) // 2
        if na.na_decode_workspace_size(cfg, mid, max_kv) <= STATIC_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


def test_static_scratch_near_the_limit():
    """The largest batch whose workspace (on this device's SM count) fits the
    array runs and matches the workspace decode; one more sequence is rejected
    with NA_ERR_WORKSPACE before anything is enqueued."""
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=32, KV=8, d=128, rd=128)
    cfg = attn_cfg(spec)
    cap = 64
    B = _largest_batch_that_fits(na, cfg, cap)
    assert na.na_decode_workspace_size(cfg, B, cap) <= STATIC_BYTES
    assert na.na_decode_workspace_size(cfg, B + 1, cap) > STATIC_BYTES
    gen = torch.Generator().manual_seed(103)
    lens = torch.randint(1, cap + 1, (B,), generator=gen).tolist()
    dec = W.make_decode(spec, lens, cap, seed=104)
    ref_out, ref_p = _run(dec, static=False, splits=0)
    out, probs = _run(dec, static=True, splits=0)
    assert_out_close(out.double().numpy(), ref_out.double().numpy(), "static at the limit")
    _check_probs(probs, ref_p, lens, "static at the limit probs")

    dev = "cuda"
    q = torch.zeros(B + 1, 32, 128, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(B + 1, 8, cap, 128, dtype=torch.bfloat16, device=dev)
    kv = torch.full((B + 1,), cap, dtype=torch.int32, device=dev)
    cache = na.KVCache(k, k)
    c, kc = cfg.c(), cache.c()
    lib = na.load_library()
    rc = lib.na_attn_decode_static_ws(ctypes.byref(c), B + 1, q.data_ptr(), ctypes.byref(kc),
                                      kv.data_ptr(), cap, None, q.data_ptr(), None, 0, 0, None,
                                      None)
    assert rc == na.NA_ERR_WORKSPACE


def test_static_scratch_rejects_oversized_request():
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=32, KV=8, d=128, rd=128)
    cfg = attn_cfg(spec)
    dev = "cuda"
    # 2048 sequences of up to 8192 keys need ~34 MB of partials: above the 20 MiB array
    B, cap = 2048, 8192
    assert na.na_decode_workspace_size(cfg, B, cap) > STATIC_BYTES
    q = torch.zeros(B, 32, 128, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 8, 16, 128, dtype=torch.bfloat16, device=dev)
    cache = na.KVCache(k, k)
    fake = na.na_kv_cache(cache.k.data_ptr(), cache.v.data_ptr(), B, cap)
    c = cfg.c()
    lib = na.load_library()
    rc = lib.na_attn_decode_static_ws(ctypes.byref(c), B, q.data_ptr(), ctypes.byref(fake),
                                      q.data_ptr(), cap, None, q.data_ptr(), None, 0, 0, None,
                                      None)
    assert rc == na.NA_ERR_WORKSPACE

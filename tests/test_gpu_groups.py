"""Parity at the extremes of the query-head grouping: one kv head serving 64
or 128 query heads (the prefill tile then holds two tokens, or one, of every
head of the group), odd groups that do not divide the 128-row tile (7, and a
single head), and decode groups that take several head chunks of 8, 4 or 1
heads per CTA (24, 12, 7).  Every output row, every appended cache slot and
every per-key probability is compared with the oracle.  Also caches smaller
than one key tile (1 to 130 slots), where a tile reaches into the next
sequence's slab or past the cache."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import (assert_out_close, assert_probs_close, check_cache, gpu_decode, gpu_step,
                     oracle_append, oracle_flags, oracle_rows, score_scale)

pytestmark = pytest.mark.gpu

PREFILL = {
    # group 64: two tokens x 64 heads per tile
    "h64kv1d128_group64": (W.Spec(H=64, KV=1, d=128, rd=128, rope=W.RopeParams(base=5e5)),
                           [300, 0], [5, 130]),
    # group 128: one token x 128 heads per tile, with qk-norm and the gate
    "h128kv1d64_group128_qknorm_gate": (W.Spec(H=128, KV=1, d=64, rd=64, qk_norm=True,
                                               out_gate=True), [40, 200, 0], [3, 1, 9]),
    # group 32, partial rotary, soft cap
    "h64kv2d128_group32_softcap": (W.Spec(H=64, KV=2, d=128, rd=64, softcap=20.0),
                                   [129, 0], [17, 64]),
    # odd groups: no packing
    "h7kv1d128_group7": (W.Spec(H=7, KV=1, d=128, rd=128), [250, 3], [140, 2]),
    "h56kv8d64_group7_window": (W.Spec(H=56, KV=8, d=64, rd=32, window=90), [500], [150]),
    "h1kv1d128_single_head": (W.Spec(H=1, KV=1, d=128, rd=128), [0, 900], [260, 7]),
}


@pytest.mark.parametrize("name", list(PREFILL))
def test_prefill_wide_and_odd_groups(oracle, name):
    spec, prior, new = PREFILL[name]
    capacity = max(p + n for p, n in zip(prior, new))
    capacity = (capacity + 127) // 128 * 128
    step = W.make_step(spec, prior, new, capacity, seed=41)
    g = gpu_step(step)
    assert g.status == 0, f"status {g.status}"
    ost = oracle_append(oracle, step)
    check_cache(g.cache_k, g.cache_v, step, ost)
    rows = list(range(step.total_tokens))
    ref = oracle_rows(oracle, step, ost, rows)
    assert_out_close(g.out[rows].to(torch.float64).numpy(), ref, name)


DECODE = {
    "h128kv1d64_group128": W.Spec(H=128, KV=1, d=64, rd=64),       # 16 head chunks of 8
    "h24kv1d128_group24_gate": W.Spec(H=24, KV=1, d=128, rd=128, out_gate=True),  # 3 of 8
    "h24kv2d128_group12": W.Spec(H=24, KV=2, d=128, rd=128),       # 3 chunks of 4
    "h56kv8d128_group7_softcap": W.Spec(H=56, KV=8, d=128, rd=128, softcap=25.0),  # 7 of 1
    "h1kv1d64_single_head": W.Spec(H=1, KV=1, d=64, rd=64),
}


@pytest.mark.parametrize("name", list(DECODE))
def test_decode_wide_and_odd_groups(oracle, name):
    s = DECODE[name]
    dec = W.make_decode(s, [0, 1, 65, 700, 2100], 2176, seed=43)
    out, probs, status = gpu_decode(dec, with_probs=True)
    assert status == 0
    ref_out, ref_p = oracle.decode(
        s.H, s.KV, s.d, score_scale(s), oracle_flags(s, False), W.bf16_to_f64(dec.q),
        np.ascontiguousarray(W.bf16_to_f64(dec.cache_k)),
        np.ascontiguousarray(W.bf16_to_f64(dec.cache_v)), dec.kv_lens.numpy(),
        gate=W.bf16_to_f64(dec.gate), probs_stride=probs.shape[-1], softcap=s.softcap,
        window=s.window)
    assert_out_close(out.double().numpy(), ref_out, f"{name} out")
    for b, n in enumerate(dec.kv_lens.tolist()):
        assert_probs_close(probs[b, :, :n].numpy(), ref_p[b, :, :n], f"{name} probs b{b}")
        assert bool((probs[b, :, n:] == -7.0).all()), "probs written past kv_len"


@pytest.mark.parametrize("cap,prior,new", [(40, [0, 10], [7, 30]), (1, [0, 0], [1, 1]),
                                           (130, [1, 64], [128, 66])])
def test_prefill_cache_smaller_than_a_key_tile(oracle, cap, prior, new):
    """Capacities of 1, 40 and 130 slots: a 128-key tile reaches past a
    sequence's slab into the next one's (or past the cache), and those rows
    must be masked and zeroed, never attended."""
    spec = W.Spec(H=4, KV=2, d=64, rd=64, out_gate=True)
    step = W.make_step(spec, prior, new, cap, seed=47)
    g = gpu_step(step)
    assert g.status == 0, f"status {g.status}"
    ost = oracle_append(oracle, step)
    check_cache(g.cache_k, g.cache_v, step, ost)
    rows = list(range(step.total_tokens))
    ref = oracle_rows(oracle, step, ost, rows)
    assert_out_close(g.out[rows].to(torch.float64).numpy(), ref, f"capacity {cap}")


@pytest.mark.parametrize("cap,lens", [(40, [40, 1, 0, 17]), (1, [1, 1, 0]), (65, [65, 64, 3])])
def test_decode_cache_smaller_than_a_key_tile(oracle, cap, lens):
    """Decode over caches of 1, 40 and 65 slots (64-key tiles reach into the
    next slab or past the cache)."""
    s = W.Spec(H=8, KV=2, d=128, rd=128)
    dec = W.make_decode(s, lens, cap, seed=49)
    out, probs, status = gpu_decode(dec, with_probs=True)
    assert status == 0
    ref_out, ref_p = oracle.decode(
        s.H, s.KV, s.d, score_scale(s), oracle_flags(s, False), W.bf16_to_f64(dec.q),
        np.ascontiguousarray(W.bf16_to_f64(dec.cache_k)),
        np.ascontiguousarray(W.bf16_to_f64(dec.cache_v)), dec.kv_lens.numpy(),
        probs_stride=probs.shape[-1])
    assert_out_close(out.double().numpy(), ref_out, f"capacity {cap} out")
    for b, n in enumerate(lens):
        assert_probs_close(probs[b, :, :n].numpy(), ref_p[b, :, :n], f"capacity {cap} probs b{b}")

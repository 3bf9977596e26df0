"""Parity of the fused qk-norm + RoPE + cache-append kernel with the oracle.

Rotated Q and K within 1 bf16 ulp, V bit-exact (or within 1 ulp when
V-normed), untouched cache slots bit-identical, positions exact."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import assert_within_ulp, check_cache, gpu_step, oracle_append

pytestmark = pytest.mark.gpu

CASES = {
    "h4kv2d64_full_rotary_128tok": (W.C1.spec, [0], [128], 128),
    "h32kv8d128_base5e5_two_seqs": (W.C2.spec, [0, 1000], [128, 77], 2048),
    "yarn_partial_rotary_high_positions": (W.C4.spec, [5, 32700], [3, 68], 32768),
    "qknorm_gate_varlen_with_empty_seq": (W.C5.spec, [0, 17, 400, 0], [9, 0, 130, 1], 600),
    "d64_qknorm_zero_centred_vnorm_partial": (
        W.Spec(H=6, KV=3, d=64, rd=32, rope=W.RopeParams(base=1e4), qk_norm=True,
               qk_norm_zero_centered=True, v_norm=True, eps=1e-5, norm_w_mean=0.0),
        [3, 0], [5, 31], 64),
    "yarn_attn_factor_one": (
        W.Spec(H=8, KV=2, d=128, rd=64, rope=W.RopeParams(base=1e6, yarn=True, factor=4.0,
                                                          orig_max_pos=8192, attn_factor=1.0)),
        [100], [33], 256),
    "no_rotary": (W.Spec(H=4, KV=4, d=128, rd=0), [2], [7], 16),
    # rotary_dim not a multiple of 16, and more rows than one thread each: the
    # shared-memory staged kernel
    "staged_rd24_d64_qknorm_vnorm": (
        W.Spec(H=4, KV=2, d=64, rd=24, rope=W.RopeParams(base=1e4), qk_norm=True, v_norm=True),
        [40, 3], [6, 9], 64),
    "staged_rd40_d128_yarn": (
        W.Spec(H=8, KV=4, d=128, rd=40, rope=W.RopeParams(base=1e6, yarn=True, factor=4.0,
                                                          orig_max_pos=8192)),
        [9000], [12], 9100),
    "staged_h96kv8_many_rows": (W.Spec(H=96, KV=8, d=128, rd=128), [0, 500], [5, 3], 512),
    "register_h80kv8_widest": (W.Spec(H=80, KV=8, d=128, rd=128, qk_norm=True), [0, 70], [4, 2],
                               128),
}


@pytest.mark.parametrize("name", list(CASES))
def test_rope_append_matches_oracle(oracle, name):
    spec, prior, new, cap = CASES[name]
    step = W.make_step(spec, prior, new, cap, seed=11)
    g = gpu_step(step)
    assert g.status == 0
    ost = oracle_append(oracle, step)
    assert_within_ulp(g.q_out, ost.q_rot, "rotated Q")
    check_cache(g.cache_k, g.cache_v, step, ost)


def test_capacity_overflow_reported_and_skipped(oracle):
    """A token whose position does not fit is skipped and reported; the
    others are written."""
    import causal_gqa_attention_rope_gb300 as na
    from harness import attn_cfg, rope_cfg
    spec = W.Spec(H=4, KV=2, d=64, rd=64)
    step = W.make_step(spec, [6], [4], 8, seed=3)  # positions 6..9, capacity 8
    dev = "cuda"
    cache = na.KVCache(step.cache_k.to(dev), step.cache_v.to(dev))
    q_out = torch.zeros_like(step.q).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    na.na_rope_append_kv(attn_cfg(spec), rope_cfg(spec), step.cu_seqlens.to(dev),
                         step.cache_lens.to(dev), step.q.to(dev), step.k.to(dev), step.v.to(dev),
                         q_out, cache, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == na.NA_ERR_CAPACITY
    ck = cache.k.cpu()
    assert not W.SENTINEL_BITS in ck[0, :, 6:8].contiguous().view(torch.int16).unique().tolist()
    assert torch.equal(ck[0, :, :6].contiguous().view(torch.int16),
                       step.cache_k[0, :, :6].contiguous().view(torch.int16))


def test_zero_tokens_is_noop():
    import causal_gqa_attention_rope_gb300 as na
    from harness import attn_cfg, rope_cfg
    spec = W.Spec(H=4, KV=2, d=64, rd=64)
    dev = "cuda"
    k = W.sentinel_fill((1, 2, 8, 64)).to(dev)
    cache = na.KVCache(k, k.clone())
    e = torch.empty(0, 4, 64, dtype=torch.bfloat16, device=dev)
    ekv = torch.empty(0, 2, 64, dtype=torch.bfloat16, device=dev)
    na.na_rope_append_kv(attn_cfg(spec), rope_cfg(spec), torch.zeros(2, dtype=torch.int32,
                                                                      device=dev),
                         torch.zeros(1, dtype=torch.int32, device=dev), e, ekv, ekv, e, cache,
                         total_tokens=0)
    torch.cuda.synchronize()
    assert torch.equal(cache.k.cpu().view(torch.int16), k.cpu().view(torch.int16))


def test_position_rotation_relative_property_on_gpu():
    """The GPU's rotated q at position m dotted with its rotated k at n depends
    only on m - n: same q/k rows placed at shifted positions."""
    spec = W.Spec(H=1, KV=1, d=128, rd=128, rope=W.RopeParams(base=1e4), std=1.0)
    gen = torch.Generator().manual_seed(5)
    qrow = torch.randn(1, 1, 128, generator=gen).to(torch.bfloat16)
    krow = torch.randn(1, 1, 128, generator=gen).to(torch.bfloat16)
    dots = []
    for shift in (0, 1000, 20000):
        step = W.make_step(spec, [shift], [2], 32768, seed=0, history=False)
        step.q[:] = qrow
        step.k[:] = krow
        g = gpu_step(step)
        qm = g.q_out[1, 0].double()                     # q at shift + 1
        kn = g.cache_k[0, 0, shift].double()            # k at shift
        dots.append(float(qm @ kn))
    assert max(dots) - min(dots) < 0.05 * (1 + abs(dots[0])), dots

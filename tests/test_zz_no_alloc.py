"""The allocation-free decode entry point (na_attn_decode_static_ws).

It serves callers that cannot allocate device memory for a workspace (a
plugin inside a runtime that owns all device memory, a serving loop that may
not allocate once running): the split partials live in a fixed array inside
the library.  This file runs last so that a failure here leaves every other
test already run.  The check: through the C ABI, two calls in a row give the
same output and probabilities as na_attn_decode with a caller workspace,
within the parity tolerances."""
import pytest
import torch

import workloads as W
from harness import assert_out_close, assert_probs_close, attn_cfg

pytestmark = pytest.mark.gpu


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
    out = torch.empty_like(q)
    probs = torch.full((B, dec.spec.H, max_kv), -7.0, dtype=torch.float32, device=dev)
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
    return out.cpu(), probs.cpu()


def test_static_scratch_decode_matches_workspace_decode():
    spec = W.Spec(H=32, KV=8, d=128, rd=128, out_gate=True)
    cases = [W.make_decode(spec, [4096, 700, 1, 2500], 4096, seed=101),
             W.make_decode(W.Spec(H=8, KV=2, d=64, rd=64), [63, 2048, 0], 2048, seed=102)]
    for dec, splits in ((cases[0], 0), (cases[1], 5)):
        ref_out, ref_p = _run(dec, static=False, splits=splits)
        for _ in range(2):  # two calls in a row share the library's array
            out, probs = _run(dec, static=True, splits=splits)
            assert_out_close(out.double().numpy(), ref_out.double().numpy(), "static decode")
            for b, n in enumerate(dec.kv_lens.tolist()):
                assert_probs_close(probs[b, :, :n].numpy(), ref_p[b, :, :n].numpy(), "probs")
                assert bool((probs[b, :, n:] == -7.0).all())


def test_static_scratch_rejects_oversized_request():
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=32, KV=8, d=128, rd=128)
    cfg = attn_cfg(spec)
    dev = "cuda"
    # 2048 sequences of up to 8192 keys need ~34 MB of partials: above the 20 MiB array
    B, cap = 2048, 8192
    assert na.na_decode_workspace_size(cfg, B, cap) > 20 * 2**20
    q = torch.zeros(B, 32, 128, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(1, 8, 16, 128, dtype=torch.bfloat16, device=dev)
    cache = na.KVCache(k, k)
    fake = na.na_kv_cache(cache.k.data_ptr(), cache.v.data_ptr(), B, cap)
    import ctypes
    c = cfg.c()
    lib = na.load_library()
    rc = lib.na_attn_decode_static_ws(ctypes.byref(c), B, q.data_ptr(), ctypes.byref(fake),
                                      q.data_ptr(), cap, None, q.data_ptr(), None, 0, 0, None,
                                      None)
    assert rc == na.NA_ERR_WORKSPACE

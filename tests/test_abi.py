"""The C ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and its host-side validation and planning answer correctly
(no kernel is launched here)."""
import ctypes
import os
import re

import pytest

import causal_gqa_attention_rope_gb300 as na
from causal_gqa_attention_rope_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return na.load_library()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "na.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(na_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_symbols()
    assert set(declared) >= {"na_rope_append_kv", "na_attn_prefill_chunk", "na_attn_decode"}
    for name in declared:
        assert hasattr(lib, name), f"{name} missing from libna.so"
    assert set(declared) == set(na.EXPORTED)


def test_status_strings(lib):
    assert na.status_string(0) == "ok"
    for code in range(-6, 0):
        assert na.status_string(code) not in ("", "unknown status")
    assert na.status_string(-99) == "unknown status"


def _cfg(**kw):
    base = dict(num_heads=32, num_kv_heads=8, head_dim=128, rotary_dim=128)
    base.update(kw)
    return na.AttnConfig(**base).c()


@pytest.mark.parametrize("kw,code", [
    (dict(num_heads=30, num_kv_heads=8), na.NA_ERR_INVALID_ARG),
    (dict(num_kv_heads=0), na.NA_ERR_INVALID_ARG),
    (dict(rotary_dim=63), na.NA_ERR_INVALID_ARG),
    (dict(rotary_dim=130), na.NA_ERR_INVALID_ARG),
    (dict(head_dim=96, rotary_dim=96), na.NA_ERR_UNSUPPORTED),
    (dict(softcap=-1.0), na.NA_ERR_INVALID_ARG),
    (dict(softcap=float("nan")), na.NA_ERR_INVALID_ARG),
    (dict(softcap=float("inf")), na.NA_ERR_INVALID_ARG),
    (dict(window=-3), na.NA_ERR_INVALID_ARG),
    (dict(ring_cache=True), na.NA_ERR_INVALID_ARG),  # a ring needs a window
])
def test_bad_config_rejected_before_launch(lib, kw, code):
    c = _cfg(**kw)
    out = ctypes.c_size_t(0)
    assert lib.na_decode_workspace_size(ctypes.byref(c), 4, 100, 0, ctypes.byref(out)) == code


def test_null_and_misaligned_buffers_rejected(lib):
    c = _cfg()
    cache = na.na_kv_cache(16, 16, 1, 64)  # fake non-null, aligned addresses
    rc = lib.na_attn_decode(ctypes.byref(c), 1, None, ctypes.byref(cache), 16, 10, None, 16,
                            None, 0, 0, 16, 1 << 20, None, None)
    assert rc == na.NA_ERR_INVALID_ARG
    rc = lib.na_attn_decode(ctypes.byref(c), 1, 18, ctypes.byref(cache), 16, 10, None, 16, None,
                            0, 0, 16, 1 << 20, None, None)
    assert rc == na.NA_ERR_INVALID_ARG  # q not 16-byte aligned
    bad_cache = na.na_kv_cache(16, 24, 1, 64)
    rc = lib.na_attn_decode(ctypes.byref(c), 1, 16, ctypes.byref(bad_cache), 16, 10, None, 16,
                            None, 0, 0, 16, 1 << 20, None, None)
    assert rc == na.NA_ERR_INVALID_ARG


def test_capacity_and_workspace_checks(lib):
    c = _cfg()
    cache = na.na_kv_cache(16, 16, 2, 64)
    # max_kv_len past capacity
    rc = lib.na_attn_decode(ctypes.byref(c), 2, 16, ctypes.byref(cache), 16, 65, None, 16, None,
                            0, 0, 16, 1 << 20, None, None)
    assert rc == na.NA_ERR_CAPACITY
    # probability stride shorter than the longest sequence
    rc = lib.na_attn_decode(ctypes.byref(c), 2, 16, ctypes.byref(cache), 16, 40, None, 16, 16, 32,
                            0, 16, 1 << 20, None, None)
    assert rc == na.NA_ERR_CAPACITY
    # workspace too small
    rc = lib.na_attn_decode(ctypes.byref(c), 2, 16, ctypes.byref(cache), 16, 40, None, 16, None, 0,
                            0, 16, 8, None, None)
    assert rc == na.NA_ERR_WORKSPACE
    # prefill: total length past capacity
    rc = lib.na_attn_prefill_chunk(ctypes.byref(c), 1, 16, 16, 10, 10, 65, 16,
                                   ctypes.byref(cache), None, 16, None, 0, None, None)
    assert rc == na.NA_ERR_CAPACITY
    # batch larger than the cache's
    rc = lib.na_attn_prefill_chunk(ctypes.byref(c), 3, 16, 16, 10, 10, 20, 16,
                                   ctypes.byref(cache), None, 16, None, 0, None, None)
    assert rc == na.NA_ERR_INVALID_ARG
    # gate required when the gate flag is set
    cg = _cfg()
    cg.flags = na.NA_OUT_GATE
    rc = lib.na_attn_prefill_chunk(ctypes.byref(cg), 1, 16, 16, 10, 10, 20, 16,
                                   ctypes.byref(cache), None, 16, None, 1 << 30, None, None)
    assert rc == na.NA_ERR_INVALID_ARG


def test_wait_selftest_needs_a_status_word(lib):
    assert lib.na_selftest_wait_timeout(None, None) == na.NA_ERR_INVALID_ARG


def test_rope_params_validated(lib):
    c = _cfg()
    cache = na.na_kv_cache(16, 16, 1, 64)
    bad = na.na_rope_params(1.0, 0, 1.0, 0, 32.0, 1.0, 0.0)  # base must exceed 1
    rc = lib.na_rope_append_kv(ctypes.byref(c), ctypes.byref(bad), 1, 16, 16, 4, 16, 16, 16, None,
                               None, 16, ctypes.byref(cache), None, None)
    assert rc == na.NA_ERR_INVALID_ARG
    bad_yarn = na.na_rope_params(1e6, 1, 4.0, 0, 32.0, 1.0, 0.0)  # yarn needs orig_max_pos
    rc = lib.na_rope_append_kv(ctypes.byref(c), ctypes.byref(bad_yarn), 1, 16, 16, 4, 16, 16, 16,
                               None, None, 16, ctypes.byref(cache), None, None)
    assert rc == na.NA_ERR_INVALID_ARG
    qk = _cfg()
    qk.flags = na.NA_QK_NORM
    good = na.na_rope_params(1e4, 0, 1.0, 0, 32.0, 1.0, 0.0)
    rc = lib.na_rope_append_kv(ctypes.byref(qk), ctypes.byref(good), 1, 16, 16, 4, 16, 16, 16,
                               None, None, 16, ctypes.byref(cache), None, None)
    assert rc == na.NA_ERR_INVALID_ARG  # norm weights required


def test_zero_tokens_return_ok_without_launch(lib):
    c = _cfg()
    cache = na.na_kv_cache(16, 16, 1, 64)
    good = na.na_rope_params(1e4, 0, 1.0, 0, 32.0, 1.0, 0.0)
    assert lib.na_rope_append_kv(ctypes.byref(c), ctypes.byref(good), 1, None, None, 0, None, None,
                                 None, None, None, None, ctypes.byref(cache), None, None) == 0
    assert lib.na_attn_prefill_chunk(ctypes.byref(c), 1, None, None, 0, 0, 0, None,
                                     ctypes.byref(cache), None, None, None, 0, None, None) == 0


def test_workspace_sizes_follow_the_plan(lib):
    # Whole units run one per CTA; only those left over after the last whole
    # wave (152 SMs here and on the GB300) are cut, into up to 152 / leftover
    # key ranges of at least four key tiles: 128 rows of (d + 2) floats each.
    # 1024 tokens x 19 heads = 152 units: no leftover, no workspace.
    assert na.na_prefill_workspace_size(na.AttnConfig(19, 19, 128), 1, 1024, 1024, 4096) == 0
    # 2048 tokens x 40 heads = 640 units: 32 left over, cut in 4 (8192 keys each)
    ws = na.na_prefill_workspace_size(na.AttnConfig(40, 8, 128, 64), 1, 2048, 2048, 32768)
    assert ws == 32 * 4 * 128 * 130 * 4
    # a short chunk with long history: all 32 units cut, in 4
    ws = na.na_prefill_workspace_size(na.AttnConfig(32, 8, 128), 1, 128, 128, 4096)
    assert ws == 32 * 4 * 128 * 130 * 4
    # a short history cannot be cut into pieces of four key tiles: no workspace
    assert na.na_prefill_workspace_size(na.AttnConfig(32, 8, 128), 1, 128, 128, 512) == 0
    # decode: one (d + 2)-float partial per head of each slice piece; pieces are
    # at most streams + grid, so the size follows the batch, not the lengths
    cfg = na.AttnConfig(32, 8, 128)
    ws = na.na_decode_workspace_size(cfg, 64, 8192)
    assert ws == na.na_decode_workspace_size(cfg, 64, 512)
    assert ws == na.na_decode_workspace_size(cfg, 64, 8192, 4)
    assert ws % 16 == 0
    assert 64 * 32 * 130 * 4 <= ws <= 64 * 32 * 130 * 4 + 2 * 256 * 4 * 130 * 4 + 64 * 8 * 8
    assert na.na_decode_workspace_size(cfg, 128, 64) > ws


def test_ring_cache_capacity_rules(lib):
    """A ring cache needs whole 128-key tiles and room for a window plus a chunk
    in prefill, and at least a window in whole 64-key tiles in decode (checked
    before any launch)."""
    c = _cfg(window=200, ring_cache=True)
    odd = na.na_kv_cache(16, 16, 1, 200)       # not a multiple of 128
    rc = lib.na_attn_prefill_chunk(ctypes.byref(c), 1, 16, 16, 10, 10, 5000, 16,
                                   ctypes.byref(odd), None, 16, None, 1 << 30, None, None)
    assert rc == na.NA_ERR_UNSUPPORTED
    small = na.na_kv_cache(16, 16, 1, 128)     # window + 10 new - 1 > 128
    rc = lib.na_attn_prefill_chunk(ctypes.byref(c), 1, 16, 16, 10, 10, 5000, 16,
                                   ctypes.byref(small), None, 16, None, 1 << 30, None, None)
    assert rc == na.NA_ERR_CAPACITY
    rc = lib.na_attn_decode(ctypes.byref(c), 1, 16, ctypes.byref(small), 16, 5000, None, 16,
                            None, 0, 0, 16, 1 << 30, None, None)
    assert rc == na.NA_ERR_CAPACITY            # window 200 > 128 slots
    ring200 = na.na_kv_cache(16, 16, 1, 200)   # holds the window, not a multiple of 64
    rc = lib.na_attn_decode(ctypes.byref(c), 1, 16, ctypes.byref(ring200), 16, 5000, None, 16,
                            None, 0, 0, 16, 1 << 30, None, None)
    assert rc == na.NA_ERR_UNSUPPORTED         # decode reads the ring in whole 64-key tiles


def test_cache_row_count_limit(lib):
    """Cache rows (sequences x kv heads x slots) are addressed with 32-bit tensor
    coordinates: a cache with more rows is refused before any launch."""
    c = _cfg()
    huge = na.na_kv_cache(16, 16, 1 << 20, 1 << 12)   # 2^20 x 8 kv heads x 2^12 = 2^35 rows
    rc = lib.na_attn_prefill_chunk(ctypes.byref(c), 1, 16, 16, 10, 10, 5000, 16,
                                   ctypes.byref(huge), None, 16, None, 1 << 30, None, None)
    assert rc == na.NA_ERR_UNSUPPORTED
    rc = lib.na_attn_decode(ctypes.byref(c), 1, 16, ctypes.byref(huge), 16, 5000, None, 16,
                            None, 0, 0, 16, 1 << 30, None, None)
    assert rc == na.NA_ERR_UNSUPPORTED


def test_no_fallback_without_the_library(tmp_path, monkeypatch):
    """A missing libna.so raises instead of falling back to any other path."""
    monkeypatch.setattr(na, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        na.load_library(str(tmp_path / "libna.so"))


def test_no_fallback_for_cpu_tensors(lib):
    """Compute calls take CUDA tensors only: CPU tensors raise before any launch."""
    import torch
    cfg = na.AttnConfig(4, 2, 64)
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    cache = na.KVCache(torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16),
                       torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16))
    kv = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        na.na_attn_decode(cfg, q, cache, kv, 1, torch.empty_like(q))


def test_binding_checks_dtypes_and_shapes(lib):
    """The binding checks each tensor's dtype and shape against the config
    before its pointer crosses the C ABI (the library sees pointers only):
    a wrong dtype, a wrong head count or head dim, too few rows or a cache of
    the wrong layout raise ValueError, before any CUDA work."""
    import torch
    bf = dict(dtype=torch.bfloat16)
    cfg = na.AttnConfig(4, 2, 64)
    cache = na.KVCache(torch.zeros(2, 2, 8, 64, **bf), torch.zeros(2, 2, 8, 64, **bf))
    q = torch.zeros(2, 4, 64, **bf)
    kv = torch.ones(2, dtype=torch.int32)
    cases = [
        (lambda: na.na_attn_decode(cfg, q.float(), cache, kv, 1, q), "q_rot: expected bfloat16"),
        (lambda: na.na_attn_decode(cfg, torch.zeros(2, 3, 64, **bf), cache, kv, 1, q),
         "q_rot: expected shape"),
        (lambda: na.na_attn_decode(cfg, q, cache, kv.long(), 1, q), "kv_lens: expected int32"),
        (lambda: na.na_attn_decode(cfg, q, cache, kv[:1], 1, q), "kv_lens: 1 rows"),
        (lambda: na.na_attn_decode(cfg, q, cache, kv, 1, q, probs=torch.zeros(2, 4, 8)[:, :3]),
         "probs: expected shape"),
        (lambda: na.na_attn_decode(cfg, q, na.KVCache(cache.k, cache.v[:, :, :4]), kv, 1, q),
         "cache.v: expected shape"),
        (lambda: na.na_attn_decode(cfg, q, na.KVCache(torch.zeros(2, 2, 8, 32, **bf),
                                                      torch.zeros(2, 2, 8, 32, **bf)), kv, 1, q),
         "cache.k: expected shape"),
        (lambda: na.na_rope_append_kv(cfg, na.RopeConfig(), torch.tensor([0, 3], dtype=torch.int32),
                                      torch.zeros(1, dtype=torch.int32), q, torch.zeros(3, 2, 64, **bf),
                                      torch.zeros(3, 2, 64, **bf), q, cache, total_tokens=3),
         "q: 2 rows, at least 3 needed"),
        (lambda: na.na_attn_prefill_chunk(cfg, torch.tensor([0, 2], dtype=torch.int32),
                                          torch.zeros(1, dtype=torch.int32), 2, 2, q, cache, q,
                                          gate=torch.zeros(2, 4, 64)), "gate: expected bfloat16"),
        (lambda: na.na_decode_importance(cfg, torch.zeros(2, 4, 8), kv, 8,
                                         torch.zeros(2, 8, dtype=torch.float64)),
         "imp: expected float32"),
    ]
    for call, msg in cases:
        with pytest.raises(ValueError, match=msg):
            call()
    # right dtypes and shapes: refused only for being CPU tensors
    with pytest.raises(ValueError, match="CUDA tensors only"):
        na.na_attn_decode(cfg, q, cache, kv, 1, torch.empty_like(q),
                          probs=torch.zeros(2, 4, 8))

"""Python binding of the GB300 attention library ``libna.so`` (C ABI in ``include/na.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libna.so``.  PyTorch supplies device memory and streams.  There is
no CPU fallback: importing works without a GPU (so the symbols can be checked),
but every compute call needs the built library and CUDA tensors, and raises
otherwise.

Entry points (same names as the C ABI):
  na_rope_append_kv      fused qk-norm + RoPE + KV-cache append
  na_attn_prefill_chunk  causal GQA attention of a chunk against the cache
  na_attn_decode         single-token decode with per-key probabilities
  na_decode_importance   the step's Born-rule importance (sum over heads of the probabilities)
  na_attn_decode_static_ws  na_attn_decode with library-owned scratch
  na_prefill_workspace_size / na_decode_workspace_size / na_status_string
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libna.so")

NA_OK = 0
NA_ERR_INVALID_ARG = -1
NA_ERR_UNSUPPORTED = -2
NA_ERR_CAPACITY = -3
NA_ERR_WORKSPACE = -4
NA_ERR_CUDA = -5
NA_ERR_DEVICE_TIMEOUT = -6

NA_QK_NORM = 1
NA_QK_NORM_ZERO_CENTERED = 2
NA_V_NORM = 4
NA_OUT_GATE = 8
NA_RING_CACHE = 16

# Every symbol include/na.h declares.
EXPORTED = ("na_rope_append_kv", "na_attn_prefill_chunk", "na_attn_decode",
            "na_attn_decode_static_ws", "na_decode_importance",
            "na_prefill_workspace_size", "na_decode_workspace_size", "na_status_string",
            "na_selftest_wait_timeout")


class na_attn_cfg(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("rotary_dim", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("flags", ctypes.c_uint32), ("softcap", ctypes.c_float),
                ("window", ctypes.c_int32)]


class na_rope_params(ctypes.Structure):
    _fields_ = [("base", ctypes.c_double), ("yarn", ctypes.c_int32), ("factor", ctypes.c_double),
                ("orig_max_pos", ctypes.c_int32), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double), ("attn_factor", ctypes.c_double)]


class na_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("capacity", ctypes.c_int32)]


class NAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {status_string(code)} ({code})")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libna.so (raises when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libna.so is not built ({path}); run __graft_entry__.build() or "
                           f"python -m causal_gqa_attention_rope_gb300._build")
    lib = ctypes.CDLL(path)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    cfgp = ctypes.POINTER(na_attn_cfg)
    ropep = ctypes.POINTER(na_rope_params)
    cachep = ctypes.POINTER(na_kv_cache)
    lib.na_rope_append_kv.argtypes = [cfgp, ropep, I32, P, P, I32, P, P, P, P, P, P, cachep, P, P]
    lib.na_attn_prefill_chunk.argtypes = [cfgp, I32, P, P, I32, I32, I32, P, cachep, P, P, P, SZ,
                                          P, P]
    lib.na_attn_decode.argtypes = [cfgp, I32, P, cachep, P, I32, P, P, P, I32, I32, P, SZ, P, P]
    lib.na_attn_decode_static_ws.argtypes = [cfgp, I32, P, cachep, P, I32, P, P, P, I32, I32, P,
                                             P]
    lib.na_decode_importance.argtypes = [cfgp, I32, P, I32, P, I32, P, I32, I32, P, P]
    lib.na_prefill_workspace_size.argtypes = [cfgp, I32, I32, I32, I32, ctypes.POINTER(SZ)]
    lib.na_decode_workspace_size.argtypes = [cfgp, I32, I32, I32, ctypes.POINTER(SZ)]
    lib.na_selftest_wait_timeout.argtypes = [P, P]
    lib.na_status_string.argtypes = [ctypes.c_int]
    lib.na_status_string.restype = ctypes.c_char_p
    for name in ("na_rope_append_kv", "na_attn_prefill_chunk", "na_attn_decode",
                 "na_attn_decode_static_ws", "na_decode_importance",
                 "na_prefill_workspace_size", "na_decode_workspace_size",
                 "na_selftest_wait_timeout"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().na_status_string(int(code)).decode()


# ------------------------------------------------------------ configuration --

@dataclass
class AttnConfig:
    num_heads: int
    num_kv_heads: int
    head_dim: int
    rotary_dim: Optional[int] = None
    sm_scale: float = 0.0
    rms_eps: float = 1e-6
    qk_norm: bool = False
    qk_norm_zero_centered: bool = False
    v_norm: bool = False
    out_gate: bool = False
    softcap: float = 0.0
    window: int = 0
    ring_cache: bool = False

    @property
    def flags(self) -> int:
        return ((NA_QK_NORM if self.qk_norm else 0)
                | (NA_QK_NORM_ZERO_CENTERED if self.qk_norm_zero_centered else 0)
                | (NA_V_NORM if self.v_norm else 0) | (NA_OUT_GATE if self.out_gate else 0)
                | (NA_RING_CACHE if self.ring_cache else 0))

    def c(self) -> na_attn_cfg:
        rd = self.head_dim if self.rotary_dim is None else self.rotary_dim
        return na_attn_cfg(self.num_heads, self.num_kv_heads, self.head_dim, rd, self.sm_scale,
                           self.rms_eps, self.flags, self.softcap, self.window)


@dataclass
class RopeConfig:
    base: float = 10000.0
    yarn: bool = False
    factor: float = 1.0
    orig_max_pos: int = 0
    beta_fast: float = 32.0
    beta_slow: float = 1.0
    attn_factor: float = 0.0

    def c(self) -> na_rope_params:
        return na_rope_params(self.base, int(self.yarn), self.factor, self.orig_max_pos,
                              self.beta_fast, self.beta_slow, self.attn_factor)


@dataclass
class KVCache:
    """Caller-owned bf16 cache tensors [batch, num_kv_heads, capacity, head_dim]."""
    k: "object"
    v: "object"

    def c(self) -> na_kv_cache:
        return na_kv_cache(_ptr(self.k), _ptr(self.v), int(self.k.shape[0]), int(self.k.shape[2]))


# ---------------------------------------------------------------- helpers --

def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libna operates on CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libna needs contiguous tensors")
    return t.data_ptr()


_current_stream = None


def _stream(stream) -> Optional[int]:
    """Raw handle of `stream`, or of the current device's current stream."""
    global _current_stream
    if stream is not None:
        return stream.cuda_stream
    if _current_stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:  # the handle alone, without building a Stream object
            _current_stream = lambda: raw(torch.cuda.current_device())
        else:
            _current_stream = lambda: torch.cuda.current_stream().cuda_stream
    return _current_stream()


def _want(t, name: str, dtype: str, shape=None, min_rows: int = 0):
    """A tensor's dtype and shape, checked before its pointer crosses the C ABI
    (the library sees only pointers: a wrong dtype would be read as another
    type, a short tensor past its end).  `shape` entries of None match any
    size; the first dimension must also hold at least `min_rows`."""
    if t is None:
        return
    import torch
    if t.dtype != getattr(torch, dtype):
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if shape is not None:
        ok = t.dim() == len(shape) and all(w is None or int(t.shape[i]) == w
                                           for i, w in enumerate(shape))
        if not ok:
            want = "[" + ", ".join("*" if w is None else str(w) for w in shape) + "]"
            raise ValueError(f"{name}: expected shape {want}, got {list(t.shape)}")
        if int(t.shape[0]) < min_rows:
            raise ValueError(f"{name}: {int(t.shape[0])} rows, at least {min_rows} needed")


def _want_cache(cache: "KVCache", cfg: "AttnConfig", batch: int):
    _want(cache.k, "cache.k", "bfloat16", (None, cfg.num_kv_heads, None, cfg.head_dim), batch)
    _want(cache.v, "cache.v", "bfloat16", tuple(cache.k.shape))


def _check(fn: str, rc: int):
    if rc != NA_OK:
        raise NAError(fn, rc)


# ------------------------------------------------------------ entry points --

def na_rope_append_kv(cfg: AttnConfig, rope: RopeConfig, cu_seqlens, cache_lens, q, k, v,
                      q_out, cache: KVCache, q_norm_w=None, k_norm_w=None, status=None,
                      total_tokens: Optional[int] = None, stream=None):
    lib = load_library()
    T = int(q.shape[0]) if total_tokens is None else int(total_tokens)
    batch = int(cu_seqlens.numel()) - 1
    H, KV, d = cfg.num_heads, cfg.num_kv_heads, cfg.head_dim
    _want(cu_seqlens, "cu_seqlens", "int32", (None,))
    _want(cache_lens, "cache_lens", "int32", (None,), batch)
    _want(q, "q", "bfloat16", (None, H, d), T)
    _want(q_out, "q_out", "bfloat16", (None, H, d), T)
    _want(k, "k", "bfloat16", (None, KV, d), T)
    _want(v, "v", "bfloat16", (None, KV, d), T)
    _want(q_norm_w, "q_norm_w", "bfloat16", (d,))
    _want(k_norm_w, "k_norm_w", "bfloat16", (d,))
    _want(status, "status", "int32", (None,), 1)
    _want_cache(cache, cfg, batch)
    c, r, kc = cfg.c(), rope.c(), cache.c()
    rc = lib.na_rope_append_kv(ctypes.byref(c), ctypes.byref(r), batch, _ptr(cu_seqlens),
                               _ptr(cache_lens), T, _ptr(q), _ptr(k), _ptr(v), _ptr(q_norm_w),
                               _ptr(k_norm_w), _ptr(q_out), ctypes.byref(kc), _ptr(status),
                               _stream(stream))
    _check("na_rope_append_kv", rc)


def na_prefill_workspace_size(cfg: AttnConfig, batch: int, total_tokens: int, max_new_len: int,
                              max_total_len: int) -> int:
    lib = load_library()
    out = ctypes.c_size_t(0)
    c = cfg.c()
    _check("na_prefill_workspace_size",
           lib.na_prefill_workspace_size(ctypes.byref(c), batch, total_tokens, max_new_len,
                                         max_total_len, ctypes.byref(out)))
    return int(out.value)


def na_decode_workspace_size(cfg: AttnConfig, batch: int, max_kv_len: int,
                             num_splits: int = 0) -> int:
    lib = load_library()
    out = ctypes.c_size_t(0)
    c = cfg.c()
    _check("na_decode_workspace_size",
           lib.na_decode_workspace_size(ctypes.byref(c), batch, max_kv_len, num_splits,
                                        ctypes.byref(out)))
    return int(out.value)


def na_attn_prefill_chunk(cfg: AttnConfig, cu_seqlens, cache_lens, max_new_len: int,
                          max_total_len: int, q_rot, cache: KVCache, out, gate=None,
                          workspace=None, status=None, total_tokens: Optional[int] = None,
                          stream=None):
    lib = load_library()
    T = int(q_rot.shape[0]) if total_tokens is None else int(total_tokens)
    batch = int(cu_seqlens.numel()) - 1
    H, d = cfg.num_heads, cfg.head_dim
    _want(cu_seqlens, "cu_seqlens", "int32", (None,))
    _want(cache_lens, "cache_lens", "int32", (None,), batch)
    _want(q_rot, "q_rot", "bfloat16", (None, H, d), T)
    _want(out, "out", "bfloat16", (None, H, d), T)
    _want(gate, "gate", "bfloat16", (None, H, d), T)
    _want(status, "status", "int32", (None,), 1)
    _want_cache(cache, cfg, batch)
    c, kc = cfg.c(), cache.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.na_attn_prefill_chunk(ctypes.byref(c), batch, _ptr(cu_seqlens), _ptr(cache_lens), T,
                                   int(max_new_len), int(max_total_len), _ptr(q_rot),
                                   ctypes.byref(kc), _ptr(gate), _ptr(out), _ptr(workspace),
                                   ws_bytes, _ptr(status), _stream(stream))
    _check("na_attn_prefill_chunk", rc)


def _want_decode(cfg, q_rot, cache, kv_lens, out, probs, gate, status):
    H, d = cfg.num_heads, cfg.head_dim
    _want(q_rot, "q_rot", "bfloat16", (None, H, d))
    B = int(q_rot.shape[0])
    _want(out, "out", "bfloat16", (B, H, d))
    _want(gate, "gate", "bfloat16", (B, H, d))
    _want(kv_lens, "kv_lens", "int32", (None,), B)
    _want(probs, "probs", "float32", (B, H, None))
    _want(status, "status", "int32", (None,), 1)
    _want_cache(cache, cfg, B)


def na_attn_decode(cfg: AttnConfig, q_rot, cache: KVCache, kv_lens, max_kv_len: int, out,
                   probs=None, gate=None, workspace=None, num_splits: int = 0, status=None,
                   stream=None):
    lib = load_library()
    batch = int(q_rot.shape[0])
    _want_decode(cfg, q_rot, cache, kv_lens, out, probs, gate, status)
    c, kc = cfg.c(), cache.c()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    stride = int(probs.shape[-1]) if probs is not None else 0
    rc = lib.na_attn_decode(ctypes.byref(c), batch, _ptr(q_rot), ctypes.byref(kc), _ptr(kv_lens),
                            int(max_kv_len), _ptr(gate), _ptr(out), _ptr(probs), stride,
                            int(num_splits), _ptr(workspace), ws_bytes, _ptr(status),
                            _stream(stream))
    _check("na_attn_decode", rc)


def na_attn_decode_static_ws(cfg: AttnConfig, q_rot, cache: KVCache, kv_lens, max_kv_len: int,
                             out, probs=None, gate=None, num_splits: int = 0, status=None,
                             stream=None):
    """na_attn_decode without a workspace argument: the split partials live in
    a fixed 20 MiB device array inside the library, for callers that cannot
    allocate device memory.  Calls that overlap on the GPU race on that array."""
    lib = load_library()
    batch = int(q_rot.shape[0])
    _want_decode(cfg, q_rot, cache, kv_lens, out, probs, gate, status)
    c, kc = cfg.c(), cache.c()
    stride = int(probs.shape[-1]) if probs is not None else 0
    rc = lib.na_attn_decode_static_ws(ctypes.byref(c), batch, _ptr(q_rot), ctypes.byref(kc),
                                      _ptr(kv_lens), int(max_kv_len), _ptr(gate), _ptr(out),
                                      _ptr(probs), stride, int(num_splits), _ptr(status),
                                      _stream(stream))
    _check("na_attn_decode_static_ws", rc)


def na_decode_importance(cfg: AttnConfig, probs, kv_lens, max_kv_len: int, imp,
                         accumulate: bool = False, status=None, stream=None):
    """Born-rule importance of a decode step: imp[b][j] (+)= sum over heads of
    probs[b][h][j] for j < kv_lens[b].  probs [B,H,stride] fp32, imp [B,stride2]."""
    lib = load_library()
    _want(probs, "probs", "float32", (None, cfg.num_heads, None))
    B = int(probs.shape[0])
    _want(imp, "imp", "float32", (B, None))
    _want(kv_lens, "kv_lens", "int32", (None,), B)
    _want(status, "status", "int32", (None,), 1)
    c = cfg.c()
    rc = lib.na_decode_importance(ctypes.byref(c), int(probs.shape[0]), _ptr(probs),
                                  int(probs.shape[-1]), _ptr(kv_lens), int(max_kv_len), _ptr(imp),
                                  int(imp.shape[-1]), 1 if accumulate else 0, _ptr(status),
                                  _stream(stream))
    _check("na_decode_importance", rc)


def na_selftest_wait_timeout(status, stream=None):
    """Run the library's bounded device wait on a barrier nothing completes:
    after about a second `status` holds NA_ERR_DEVICE_TIMEOUT."""
    _check("na_selftest_wait_timeout",
           load_library().na_selftest_wait_timeout(_ptr(status), _stream(stream)))


def workspace(nbytes: int, device="cuda"):
    """A byte tensor usable as workspace (None when nbytes is 0)."""
    import torch
    if nbytes == 0:
        return None
    return torch.empty((nbytes + 15) // 16 * 16, dtype=torch.uint8, device=device)

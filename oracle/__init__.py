"""Reference oracle: plain f64 CPU statement of RoPE + causal GQA attention.

TEST INFRASTRUCTURE ONLY.  The oracle is the slow, obviously correct C
implementation in ``na_oracle.c``; this module compiles it with gcc and wraps
it with numpy-friendly calls.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it.  It shares no code with the
CUDA library and the library never calls it.

Pages it follows (docs.rs source pages): cortiq-engine 0.5.39
``src/attention.rs`` (fns ``rope_inv_freq``, ``yarn_inv_freq``,
``rope_rotate_scaled``, ``rmsnorm_head``, ``vnorm_head``, ``attention_head``,
``apply_gate``, ``qwen_attention_batch``) and needle-core 0.3.1
``src/v2/batch.rs`` (module doc "What has to stay sequential",
fn ``batch_attention`` and its ring of ``kv_window`` positions).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "na_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")

QK_NORM = 1
QK_NORM_ZERO_CENTERED = 2
V_NORM = 4
OUT_GATE = 8
RING_CACHE = 16


def compile_oracle(source: str = SOURCE, out_path: str = LIB_PATH) -> str:
    """Compile the oracle C source into a shared library (plain -O2, no fast-math)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
           "-shared", "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)


def _dp(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_D)


def _ip(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(_I)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_rope_inv_freq.argtypes = [ctypes.c_int, ctypes.c_double, _D]
        lib.oracle_rope_inv_freq.restype = None
        lib.oracle_yarn_inv_freq.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                             ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                             _D, _I, _I]
        lib.oracle_yarn_inv_freq.restype = None
        lib.oracle_rope_attn_factor.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double]
        lib.oracle_rope_attn_factor.restype = ctypes.c_double
        lib.oracle_rope_rotate.argtypes = [_D, ctypes.c_int, ctypes.c_int64, _D, ctypes.c_double]
        lib.oracle_rope_rotate.restype = None
        lib.oracle_rmsnorm_head.argtypes = [_D, _D, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        lib.oracle_rmsnorm_head.restype = None
        lib.oracle_vnorm_head.argtypes = [_D, ctypes.c_int, ctypes.c_double]
        lib.oracle_vnorm_head.restype = None
        lib.oracle_rope_append.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, _D, ctypes.c_double, ctypes.c_int, _I, _I, _D, _D, _D, _D, _D,
            _D, _D, _D, ctypes.c_int]
        lib.oracle_rope_append.restype = ctypes.c_int
        lib.oracle_attend_rows.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
            ctypes.c_int, _I, _I, _D, _D, _D, ctypes.c_int, _D, ctypes.c_int, _I, _D,
            ctypes.c_double, ctypes.c_int]
        lib.oracle_attend_rows.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
            ctypes.c_int, _D, _D, _D, ctypes.c_int, _I, _D, _D, _D, ctypes.c_int,
            ctypes.c_int, _I, ctypes.c_double, ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_decode_importance.argtypes = [ctypes.c_int, ctypes.c_int, _D, ctypes.c_int, _I,
                                                 _D, ctypes.c_int, ctypes.c_int]
        lib.oracle_decode_importance.restype = None
        lib.oracle_ring_slot.argtypes = [ctypes.c_int64, ctypes.c_int]
        lib.oracle_ring_slot.restype = ctypes.c_int
        self.lib = lib

    # --- cache layout ---
    def ring_slot(self, pos: int, capacity: int) -> int:
        """Slot of position ``pos`` in a ring cache of ``capacity`` slots."""
        return int(self.lib.oracle_ring_slot(int(pos), int(capacity)))

    # --- RoPE frequencies (cortiq fns rope_inv_freq / yarn_inv_freq) ---
    def rope_inv_freq(self, rd: int, base: float) -> np.ndarray:
        out = np.zeros(rd // 2, dtype=np.float64)
        self.lib.oracle_rope_inv_freq(rd, base, _dp(out))
        return out

    def yarn_inv_freq(self, rd: int, base: float, factor: float, orig_max_pos: int,
                      beta_fast: float, beta_slow: float, with_bounds: bool = False):
        out = np.zeros(rd // 2, dtype=np.float64)
        low = ctypes.c_int(0)
        high = ctypes.c_int(0)
        self.lib.oracle_yarn_inv_freq(rd, base, factor, orig_max_pos, beta_fast, beta_slow,
                                      _dp(out), ctypes.byref(low), ctypes.byref(high))
        if with_bounds:
            return out, low.value, high.value
        return out

    def rope_attn_factor(self, yarn: bool, factor: float, attn_factor: float) -> float:
        return float(self.lib.oracle_rope_attn_factor(int(bool(yarn)), factor, attn_factor))

    def inv_freq_for(self, rope: dict, rd: int) -> np.ndarray:
        """Frequencies for a rope parameter dict (keys of ``workloads.RopeParams``)."""
        if rope.get("yarn"):
            return self.yarn_inv_freq(rd, rope["base"], rope["factor"], rope["orig_max_pos"],
                                      rope["beta_fast"], rope["beta_slow"])
        return self.rope_inv_freq(rd, rope["base"])

    # --- per-vector math ---
    def rope_rotate(self, x: np.ndarray, rd: int, pos: int, inv_freq: np.ndarray,
                    scale: float = 1.0) -> np.ndarray:
        y = np.array(x, dtype=np.float64, copy=True)
        self.lib.oracle_rope_rotate(_dp(y), rd, int(pos), _dp(np.ascontiguousarray(inv_freq)),
                                    scale)
        return y

    def rmsnorm_head(self, x: np.ndarray, w: np.ndarray, eps: float,
                     zero_centered: bool = False) -> np.ndarray:
        y = np.array(x, dtype=np.float64, copy=True)
        self.lib.oracle_rmsnorm_head(_dp(y), _dp(np.ascontiguousarray(w, dtype=np.float64)),
                                     y.size, eps, int(zero_centered))
        return y

    def vnorm_head(self, x: np.ndarray, eps: float) -> np.ndarray:
        y = np.array(x, dtype=np.float64, copy=True)
        self.lib.oracle_vnorm_head(_dp(y), y.size, eps)
        return y

    # --- the path ---
    def rope_append(self, H, KV, d, rd, flags, eps, inv_freq, rope_scale, cu_seqlens,
                    cache_lens, q, k, v, q_norm_w, k_norm_w, cache_k, cache_v):
        """RoPE + cache append for every new token.  Returns q_rot [T,H,d];
        cache_k / cache_v ([B,KV,cap,d] float64) are written in place."""
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        cl = np.ascontiguousarray(cache_lens, dtype=np.int32)
        T = int(cu[-1])
        q_out = np.zeros((T, H, d), dtype=np.float64)
        f = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float64)
        rc = self.lib.oracle_rope_append(
            H, KV, d, rd, flags, eps, _dp(f(inv_freq)), rope_scale, len(cu) - 1, _ip(cu),
            _ip(cl), _dp(f(q)), _dp(f(k)), _dp(f(v)), _dp(f(q_norm_w)), _dp(f(k_norm_w)),
            _dp(q_out), _dp(cache_k), _dp(cache_v), cache_k.shape[2])
        if rc != 0:
            raise ValueError("oracle_rope_append: position beyond capacity")
        return q_out

    def attend_rows(self, H, KV, d, scale, flags, cu_seqlens, cache_lens, q_rot, cache_k,
                    cache_v, gate, rows: Sequence[int], softcap: float = 0.0, window: int = 0):
        """Causal attention output for the listed new-token rows: [len(rows), H, d]
        (softcap > 0 caps the scores; window > 0 keeps only the last keys)."""
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        cl = np.ascontiguousarray(cache_lens, dtype=np.int32)
        r = np.ascontiguousarray(rows, dtype=np.int32)
        out = np.zeros((len(r), H, d), dtype=np.float64)
        g = None if gate is None else np.ascontiguousarray(gate, dtype=np.float64)
        rc = self.lib.oracle_attend_rows(H, KV, d, scale, flags, len(cu) - 1, _ip(cu), _ip(cl),
                                         _dp(np.ascontiguousarray(q_rot)), _dp(cache_k),
                                         _dp(cache_v), cache_k.shape[2], _dp(g), len(r), _ip(r),
                                         _dp(out), float(softcap), int(window))
        if rc != 0:
            raise ValueError("oracle_attend_rows: bad row or position")
        return out

    def decode(self, H, KV, d, scale, flags, q, cache_k, cache_v, kv_lens, gate=None,
               want_probs=True, probs_stride=None, rows_bh: Optional[Sequence[int]] = None,
               softcap: float = 0.0, window: int = 0):
        """Single-token decode.  Returns (out [B,H,d], probs [B,H,stride] or None).
        With rows_bh only those (b*H+h) rows are computed (others stay zero)."""
        B = q.shape[0]
        kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
        if probs_stride is None:
            probs_stride = max(1, int(kl.max()) if kl.size else 1)
        out = np.zeros((B, H, d), dtype=np.float64)
        probs = np.zeros((B, H, probs_stride), dtype=np.float64) if want_probs else None
        g = None if gate is None else np.ascontiguousarray(gate, dtype=np.float64)
        rb = None if rows_bh is None else np.ascontiguousarray(rows_bh, dtype=np.int32)
        rc = self.lib.oracle_decode(H, KV, d, scale, flags, B,
                                    _dp(np.ascontiguousarray(q, dtype=np.float64)), _dp(cache_k),
                                    _dp(cache_v), cache_k.shape[2], _ip(kl), _dp(g), _dp(out),
                                    _dp(probs), probs_stride, 0 if rb is None else len(rb),
                                    _ip(rb), float(softcap), int(window))
        if rc != 0:
            raise ValueError("oracle_decode: length beyond capacity or stride")
        return out, probs


    def decode_importance(self, H, probs, kv_lens, imp=None, accumulate=False):
        """Born-rule importance of a decode step: imp[b][j] (+)= sum over heads of
        probs[b][h][j] for j < kv_lens[b] (cortiq fn qwen_attention_core).
        probs [B,H,stride]; returns imp [B,stride] (a new zero array unless given)."""
        probs = np.ascontiguousarray(probs, dtype=np.float64)
        B, _, stride = probs.shape
        kl = np.ascontiguousarray(kv_lens, dtype=np.int32)
        if imp is None:
            imp = np.zeros((B, stride), dtype=np.float64)
        out = np.ascontiguousarray(imp, dtype=np.float64).copy()
        self.lib.oracle_decode_importance(H, B, _dp(probs), stride, _ip(kl), _dp(out),
                                          out.shape[1], 1 if accumulate else 0)
        return out


_default: Optional[Oracle] = None


def load(rebuild: bool = False) -> Oracle:
    """The oracle built from ``na_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None or rebuild:
        if rebuild or not os.path.exists(LIB_PATH) or (
                os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE)):
            compile_oracle()
        _default = Oracle(LIB_PATH)
    return _default


def build_variant(source_text: str, tag: str) -> Oracle:
    """Compile a modified copy of the oracle source (used by the tests that
    plant a mistake in the oracle to check the pins catch it)."""
    d = tempfile.mkdtemp(prefix=f"oracle_{tag}_")
    src = os.path.join(d, "variant.c")
    with open(src, "w") as fh:
        fh.write(source_text)
    return Oracle(compile_oracle(src, os.path.join(d, "libvariant.so")))

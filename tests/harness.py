"""Run the CUDA path (through the C ABI binding) and the oracle on the same
seeded inputs, and compare them at the stated tolerances.

Tolerances (written here, used by every parity test):
  - cache slots and positions: bit-exact (untouched slots keep the sentinel);
  - rotated K (and rotated Q, normed V) in bf16: within 1 bf16 ulp of the oracle;
  - attention output: max-abs error <= 2e-2 and relative L2 error <= 5e-3;
  - per-key probabilities: max-abs error <= 1e-4.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np
import torch

import workloads as W

OUT_MAX_ABS = 2e-2
OUT_REL_L2 = 5e-3
PROBS_MAX_ABS = 1e-4


# ------------------------------------------------------------ comparisons --

def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significand bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def ulp_tolerance(ref: np.ndarray) -> np.ndarray:
    """One bf16 ulp of the reference value's own binade.  The one exception:
    where the reference lies within half a step below a power of two, its
    correctly rounded bf16 value is that power of two (round to nearest, ties
    to the even significand, which the power of two has), and the tolerance is
    one ulp of that value -- one step of the binade above."""
    ax = np.abs(ref)
    u = bf16_ulp(ref)
    boundary = np.exp2(np.floor(np.log2(np.maximum(ax, np.finfo(np.float32).tiny))) + 1)
    rounds_up = (boundary - ax) <= 0.5 * u
    return np.where(rounds_up, 2.0 * u, u)


def assert_within_ulp(gpu_bf16: torch.Tensor, ref: np.ndarray, what: str, ulps: float = 1.0):
    g = gpu_bf16.to(torch.float64).numpy()
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    err = np.abs(g - ref)
    tol = ulps * ulp_tolerance(ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} values beyond {ulps} ulp; "
                           f"worst {float((err / tol).max()):.3f} ulp-units")


def assert_out_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    assert gpu.shape == ref.shape, f"{what}: shape {gpu.shape} vs {ref.shape}"
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU values"
    diff = gpu - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff)) / denom if denom > 0 else float(np.linalg.norm(diff))
    assert max_abs <= OUT_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {OUT_MAX_ABS}"
    assert rel <= OUT_REL_L2, f"{what}: rel-L2 {rel:.3e} > {OUT_REL_L2}"
    return max_abs, rel


def assert_probs_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite probabilities"
    err = float(np.max(np.abs(gpu - ref))) if gpu.size else 0.0
    assert err <= PROBS_MAX_ABS, f"{what}: probs max-abs {err:.3e} > {PROBS_MAX_ABS}"
    return err


# ----------------------------------------------------------- guard bands ---
# Every output buffer of a GPU parity case sits between two bands of a NaN
# bit pattern (bf16 0x7FC1, fp32 0x7FC0DEAD); after the call the bands must be
# bit for bit as they were: no kernel writes before or past its buffer.
GUARD_ELEMS = 512  # per side: 1 KiB of bf16, 2 KiB of fp32 (keeps 16-byte alignment)
_GUARD_BITS = {torch.bfloat16: (torch.int16, W.SENTINEL_BITS),
               torch.float32: (torch.int32, 0x7FC0DEAD)}


class Guarded:
    """A device tensor of `shape` with guard bands on both sides; `t` is the
    interior view handed to the library."""

    def __init__(self, shape, dtype, device="cuda", fill=None):
        self.n = int(np.prod(shape)) if len(shape) else 1
        ity, bits = _GUARD_BITS[dtype]
        self.buf = torch.empty(self.n + 2 * GUARD_ELEMS, dtype=dtype, device=device)
        self.buf.view(ity).fill_(bits)
        self.ity, self.bits = ity, bits
        self.t = self.buf[GUARD_ELEMS:GUARD_ELEMS + self.n].view(shape)
        if fill is not None:
            self.t.copy_(fill) if torch.is_tensor(fill) else self.t.fill_(fill)

    def check(self, what: str):
        g = self.buf.view(self.ity)
        lo, hi = g[:GUARD_ELEMS], g[GUARD_ELEMS + self.n:]
        assert bool((lo == self.bits).all()), f"{what}: written before the buffer"
        assert bool((hi == self.bits).all()), f"{what}: written past the end of the buffer"


def sentinel_mask(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int16) == W.SENTINEL_BITS


# --------------------------------------------------------------- configs ---

def attn_cfg(spec: W.Spec):
    import causal_gqa_attention_rope_gb300 as na
    return na.AttnConfig(num_heads=spec.H, num_kv_heads=spec.KV, head_dim=spec.d,
                         rotary_dim=spec.rd, sm_scale=spec.sm_scale, rms_eps=spec.eps,
                         qk_norm=spec.qk_norm, qk_norm_zero_centered=spec.qk_norm_zero_centered,
                         v_norm=spec.v_norm, out_gate=spec.out_gate, softcap=spec.softcap,
                         window=spec.window)


def rope_cfg(spec: W.Spec):
    import causal_gqa_attention_rope_gb300 as na
    r = spec.rope
    return na.RopeConfig(base=r.base, yarn=r.yarn, factor=r.factor, orig_max_pos=r.orig_max_pos,
                         beta_fast=r.beta_fast, beta_slow=r.beta_slow, attn_factor=r.attn_factor)


def score_scale(spec: W.Spec) -> float:
    return spec.sm_scale if spec.sm_scale > 0 else 1.0 / math.sqrt(spec.d)


def oracle_flags(spec: W.Spec, ring: bool = False) -> int:
    import oracle as O
    return ((O.QK_NORM if spec.qk_norm else 0)
            | (O.QK_NORM_ZERO_CENTERED if spec.qk_norm_zero_centered else 0)
            | (O.V_NORM if spec.v_norm else 0) | (O.OUT_GATE if spec.out_gate else 0)
            | (O.RING_CACHE if ring else 0))


# ------------------------------------------------------------- GPU runs ---

@dataclass
class GpuStep:
    q_out: torch.Tensor     # bf16 [T,H,d] (cpu)
    out: torch.Tensor       # bf16 [T,H,d] (cpu)
    cache_k: torch.Tensor   # bf16 [B,KV,cap,d] (cpu)
    cache_v: torch.Tensor
    status: int


def gpu_step(step: W.StepInputs, device="cuda", max_total_len: Optional[int] = None) -> GpuStep:
    """One append + attend step through the C ABI."""
    import causal_gqa_attention_rope_gb300 as na
    s = step.spec
    cfg, rope = attn_cfg(s), rope_cfg(s)
    dev = lambda x: None if x is None else x.to(device).contiguous()
    cu, lens = dev(step.cu_seqlens), dev(step.cache_lens)
    q, k, v, gate = dev(step.q), dev(step.k), dev(step.v), dev(step.gate)
    qw, kw = dev(step.q_norm_w), dev(step.k_norm_w)
    cache = na.KVCache(dev(step.cache_k), dev(step.cache_v))
    T = step.total_tokens
    gq, go = Guarded(q.shape, q.dtype, device), Guarded(q.shape, q.dtype, device)
    q_out, out = gq.t, go.t
    status = torch.zeros(1, dtype=torch.int32, device=device)
    new = (step.cu_seqlens[1:] - step.cu_seqlens[:-1])
    max_new = int(new.max()) if new.numel() else 0
    if max_total_len is None:
        max_total_len = int((step.cache_lens + new).max())
    na.na_rope_append_kv(cfg, rope, cu, lens, q, k, v, q_out, cache, q_norm_w=qw, k_norm_w=kw,
                         status=status, total_tokens=T)
    ws = na.workspace(na.na_prefill_workspace_size(cfg, step.batch, T, max_new, max_total_len),
                      device)
    na.na_attn_prefill_chunk(cfg, cu, lens, max_new, max_total_len, q_out, cache, out, gate=gate,
                             workspace=ws, status=status, total_tokens=T)
    torch.cuda.synchronize()
    gq.check("q_out")
    go.check("out")
    return GpuStep(q_out.cpu(), out.cpu(), cache.k.cpu(), cache.v.cpu(), int(status.item()))


def gpu_chunked(prompt: W.ChunkedPrompt, device="cuda"):
    """Feed a chunked prompt; returns (outputs [B,L,H,d] bf16 cpu, q_rot, cache_k, cache_v, status)."""
    import causal_gqa_attention_rope_gb300 as na
    s = prompt.spec
    cfg, rope = attn_cfg(s), rope_cfg(s)
    B, L = prompt.batch, prompt.prompt_len
    cache = na.KVCache(W.sentinel_fill((B, s.KV, prompt.capacity, s.d)).to(device),
                       W.sentinel_fill((B, s.KV, prompt.capacity, s.d)).to(device))
    status = torch.zeros(1, dtype=torch.int32, device=device)
    qw = None if prompt.q_norm_w is None else prompt.q_norm_w.to(device)
    kw = None if prompt.k_norm_w is None else prompt.k_norm_w.to(device)
    outs, qrots = [], []
    ws_bytes = 0
    for c in range(prompt.num_chunks):
        cu, lens, q, k, v, gate = prompt.chunk_tensors(c)
        lo, hi = prompt.chunk_bounds(c)
        n = hi - lo
        ws_bytes = max(ws_bytes, na.na_prefill_workspace_size(cfg, B, B * n, n, hi))
    ws = na.workspace(ws_bytes, device)
    for c in range(prompt.num_chunks):
        cu, lens, q, k, v, gate = prompt.chunk_tensors(c)
        lo, hi = prompt.chunk_bounds(c)
        n = hi - lo
        cu, lens, q, k, v = (x.to(device) for x in (cu, lens, q, k, v))
        gate = None if gate is None else gate.to(device)
        gq, go = Guarded(q.shape, q.dtype, device), Guarded(q.shape, q.dtype, device)
        q_out, out = gq.t, go.t
        na.na_rope_append_kv(cfg, rope, cu, lens, q, k, v, q_out, cache, q_norm_w=qw, k_norm_w=kw,
                             status=status)
        na.na_attn_prefill_chunk(cfg, cu, lens, n, hi, q_out, cache, out, gate=gate, workspace=ws,
                                 status=status)
        gq.check(f"q_out of chunk {c}")
        go.check(f"out of chunk {c}")
        outs.append(out.view(B, n, s.H, s.d).cpu())
        qrots.append(q_out.view(B, n, s.H, s.d).cpu())
    torch.cuda.synchronize()
    return (torch.cat(outs, 1), torch.cat(qrots, 1), cache.k.cpu(), cache.v.cpu(),
            int(status.item()))


def gpu_decode(dec: W.DecodeInputs, device="cuda", with_probs=True, num_splits=0,
               probs_stride: Optional[int] = None):
    import causal_gqa_attention_rope_gb300 as na
    s = dec.spec
    cfg = attn_cfg(s)
    B = dec.q.shape[0]
    max_kv = int(dec.kv_lens.max()) if B else 0
    q = dec.q.to(device)
    cache = na.KVCache(dec.cache_k.to(device), dec.cache_v.to(device))
    kv = dec.kv_lens.to(device)
    gate = None if dec.gate is None else dec.gate.to(device)
    go = Guarded(q.shape, q.dtype, device)
    out = go.t
    stride = probs_stride or max(max_kv, 1)
    probs, gp = None, None
    if with_probs:
        gp = Guarded((B, s.H, stride), torch.float32, device, fill=-7.0)
        probs = gp.t
    ws = na.workspace(na.na_decode_workspace_size(cfg, B, max_kv, num_splits), device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    na.na_attn_decode(cfg, q, cache, kv, max_kv, out, probs=probs, gate=gate, workspace=ws,
                      num_splits=num_splits, status=status)
    torch.cuda.synchronize()
    go.check("decode out")
    if gp is not None:
        gp.check("decode probs")
    return out.cpu(), (None if probs is None else probs.cpu()), int(status.item())


# ---------------------------------------------------------- oracle runs ---

@dataclass
class OracleStep:
    q_rot: np.ndarray
    cache_k: np.ndarray
    cache_v: np.ndarray
    rope_scale: float
    inv_freq: np.ndarray


def oracle_append(o, step: W.StepInputs, ring: bool = False) -> OracleStep:
    """The oracle's append of the step's new tokens into (a copy of) its cache;
    with ring=True the step's cache is a ring (slot = position mod capacity)."""
    s = step.spec
    inv = o.inv_freq_for(s.rope.as_dict(), s.rd)
    scale = o.rope_attn_factor(s.rope.yarn, s.rope.factor, s.rope.attn_factor)
    ck = np.ascontiguousarray(W.bf16_to_f64(step.cache_k))
    cv = np.ascontiguousarray(W.bf16_to_f64(step.cache_v))
    q_rot = o.rope_append(s.H, s.KV, s.d, s.rd, oracle_flags(s, ring), s.eps, inv, scale,
                          step.cu_seqlens.numpy(), step.cache_lens.numpy(),
                          W.bf16_to_f64(step.q), W.bf16_to_f64(step.k), W.bf16_to_f64(step.v),
                          W.bf16_to_f64(step.q_norm_w), W.bf16_to_f64(step.k_norm_w), ck, cv)
    return OracleStep(q_rot, ck, cv, scale, inv)


def oracle_rows(o, step: W.StepInputs, ost: OracleStep, rows: Sequence[int],
                ring: bool = False) -> np.ndarray:
    s = step.spec
    return o.attend_rows(s.H, s.KV, s.d, score_scale(s), oracle_flags(s, ring),
                         step.cu_seqlens.numpy(), step.cache_lens.numpy(), ost.q_rot,
                         ost.cache_k, ost.cache_v, W.bf16_to_f64(step.gate), list(rows),
                         softcap=s.softcap, window=s.window)


def prompt_as_step(prompt: W.ChunkedPrompt) -> W.StepInputs:
    """The whole chunked prompt as one chunk (the oracle's view)."""
    s, B, L = prompt.spec, prompt.batch, prompt.prompt_len
    pack = lambda x: None if x is None else x.reshape(-1, *x.shape[2:]).contiguous()
    cu = torch.arange(0, B + 1, dtype=torch.int32) * L
    return W.StepInputs(spec=s, cu_seqlens=cu, cache_lens=torch.zeros(B, dtype=torch.int32),
                        q=pack(prompt.q), k=pack(prompt.k), v=pack(prompt.v),
                        gate=pack(prompt.gate), q_norm_w=prompt.q_norm_w,
                        k_norm_w=prompt.k_norm_w,
                        cache_k=W.sentinel_fill((B, s.KV, prompt.capacity, s.d)),
                        cache_v=W.sentinel_fill((B, s.KV, prompt.capacity, s.d)))


def check_cache(gpu_k: torch.Tensor, gpu_v: torch.Tensor, step: W.StepInputs, ost: OracleStep,
                written: Optional[List[tuple]] = None):
    """Written slots within 1 ulp (V bit-exact when not normed), others untouched."""
    s = step.spec
    B = step.batch
    was_sentinel = sentinel_mask(step.cache_k)
    new_mask = torch.zeros_like(was_sentinel)
    cu, lens = step.cu_seqlens.tolist(), step.cache_lens.tolist()
    for b in range(B):
        n = cu[b + 1] - cu[b]
        new_mask[b, :, lens[b]:lens[b] + n] = True
    # untouched slots: bit-identical to what was there
    keep = ~new_mask
    assert torch.equal(gpu_k.view(torch.int16)[keep], step.cache_k.view(torch.int16)[keep]), \
        "cache K changed outside the appended slots"
    assert torch.equal(gpu_v.view(torch.int16)[keep], step.cache_v.view(torch.int16)[keep]), \
        "cache V changed outside the appended slots"
    nm = new_mask.numpy()
    assert_within_ulp(gpu_k[new_mask], ost.cache_k[nm], "cache K")
    if s.v_norm:
        assert_within_ulp(gpu_v[new_mask], ost.cache_v[nm], "cache V")
    else:
        assert np.array_equal(gpu_v[new_mask].to(torch.float64).numpy(), ost.cache_v[nm]), \
            "cache V must be the input bits"


def sample_rows(n: int, k: int, seed: int) -> List[int]:
    """First, last and k seeded random row indices."""
    if n <= k + 2:
        return list(range(n))
    g = torch.Generator().manual_seed(seed)
    mid = torch.randperm(n - 2, generator=g)[:k] + 1
    return sorted(set([0, n - 1] + mid.tolist()))


def ring_from_linear(o, cache: torch.Tensor, lens: Sequence[int], ring: int) -> torch.Tensor:
    """A linear cache [B, KV, cap, d] laid out as a ring of `ring` slots per
    (sequence, kv head): position p of the first lens[b] goes to the oracle's
    ring slot of p, so only the last `ring` positions survive; untouched slots
    hold the sentinel."""
    B, KV, _, d = cache.shape
    out = W.sentinel_fill((B, KV, ring, d))
    for b, n in enumerate(lens):
        for pos in range(max(0, n - ring), n):
            out[b, :, o.ring_slot(pos, ring)] = cache[b, :, pos]
    return out

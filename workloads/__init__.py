"""Seeded synthetic inputs for the attention path.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA library's tests/benchmark and the oracle
read the tensors it produces, so the two sides see identical bf16 bits.

Recipe (all draws on the CPU with ``torch.Generator().manual_seed(seed)``):
  1. lengths first (prior cache lengths, then new-token counts), each an
     integer uniform on the stated closed range, drawn with ``torch.randint``;
  2. then, in this order, Q [T,H,d], K [T,KV,d], V [T,KV,d], the gate logits
     [T,H,d] (if gated), the q-norm and k-norm weights [d] (if normed), and
     finally the cache history K and V for each sequence's prior positions;
  3. every tensor is drawn in fp32 as ``mean + std * N(0,1)`` and rounded to
     bf16 with round-to-nearest-even (``Tensor.to(torch.bfloat16)``).
Cache slots past a sequence's length hold the sentinel bit pattern 0x7FC1 (a
bf16 quiet NaN) so a test can check that nothing wrote them.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import List, Optional

import torch

SENTINEL_BITS = 0x7FC1  # bf16 quiet NaN with a payload, never produced by the kernels


@dataclass
class RopeParams:
    base: float = 10000.0
    yarn: bool = False
    factor: float = 1.0
    orig_max_pos: int = 0
    beta_fast: float = 32.0
    beta_slow: float = 1.0
    attn_factor: float = 0.0  # <= 0: default (1, or 0.1 ln(factor) + 1 with YaRN)

    def as_dict(self):
        return dataclasses.asdict(self)


@dataclass
class Spec:
    """One attention layer's shapes, options and length mix."""
    H: int
    KV: int
    d: int
    rd: int
    rope: RopeParams = field(default_factory=RopeParams)
    qk_norm: bool = False
    qk_norm_zero_centered: bool = False
    v_norm: bool = False
    out_gate: bool = False
    eps: float = 1e-6
    std: float = 1.0            # Q/K/V standard deviation
    norm_w_mean: float = 1.0    # norm weights ~ N(norm_w_mean, norm_w_std)
    norm_w_std: float = 0.1
    sm_scale: float = 0.0       # <= 0: 1/sqrt(d)
    softcap: float = 0.0        # > 0: logit soft-capping
    window: int = 0             # > 0: sliding-window attention


@dataclass
class PrefillWorkload:
    """A prompt fed as a run of equal chunks (batch of one or more sequences
    with identical lengths) or a single varlen packed step."""
    name: str
    spec: Spec
    batch: int
    prompt_len: int = 0          # per sequence, chunked workloads
    chunk: int = 0
    capacity: int = 0
    prior_range: Optional[tuple] = None  # varlen: (lo, hi) inclusive
    new_range: Optional[tuple] = None
    description: str = ""


@dataclass
class DecodeWorkload:
    name: str
    spec: Spec
    batch: int
    kv_range: tuple
    capacity: int
    with_probs: bool = True
    description: str = ""


# The five workloads, named by what they are.
C1 = PrefillWorkload(
    name="prefill_h4kv2d64_t128_single_chunk",
    spec=Spec(H=4, KV=2, d=64, rd=64, rope=RopeParams(base=10000.0), std=1.0),
    batch=1, prompt_len=128, chunk=128, capacity=128,
    description="1 sequence, 4/2 heads, d 64, 128-token prompt in one chunk, empty cache, "
                "RoPE base 1e4 full rotary, Q/K/V ~ N(0,1), seed 0")
C2 = PrefillWorkload(
    name="chunked_prefill_h32kv8d128_t4096_chunk128",
    spec=Spec(H=32, KV=8, d=128, rd=128, rope=RopeParams(base=500000.0), std=0.5),
    batch=1, prompt_len=4096, chunk=128, capacity=8192,
    description="1 sequence, 32/8 heads, d 128, 4096-token prompt as 32 chunks of 128, "
                "RoPE base 5e5, Q/K/V ~ 0.5 N(0,1), cache of 8192 slots")
C3 = DecodeWorkload(
    name="decode_b64_h32kv8d128_kv512to8192",
    spec=Spec(H=32, KV=8, d=128, rd=128, std=1.0),
    batch=64, kv_range=(512, 8192), capacity=8192, with_probs=True,
    description="64 sequences, one new token each, cached length ~ U{512..8192}, 32/8 heads, "
                "d 128, cache and q ~ N(0,1), fp32 per-key probabilities")
C4 = PrefillWorkload(
    name="yarn_prefill_h40kv8d128_rd64_t32768_chunk2048",
    spec=Spec(H=40, KV=8, d=128, rd=64,
              rope=RopeParams(base=1e6, yarn=True, factor=4.0, orig_max_pos=8192,
                              beta_fast=32.0, beta_slow=1.0), std=1.0),
    batch=1, prompt_len=32768, chunk=2048, capacity=32768,
    description="1 sequence, 40/8 heads, d 128, partial rotary 64, YaRN (1e6, x4, 8192, "
                "32, 1), 32768 tokens in chunks of 2048, Q/K/V ~ N(0,1)")
C5 = PrefillWorkload(
    name="varlen_step_b16_h32kv4d128_qknorm_gate",
    spec=Spec(H=32, KV=4, d=128, rd=128, rope=RopeParams(base=1e6), qk_norm=True,
              out_gate=True, eps=1e-6, std=1.0, norm_w_mean=1.0, norm_w_std=0.1),
    batch=16, capacity=16896, prior_range=(0, 16384), new_range=(1, 512),
    description="16 sequences packed, prior cache ~ U{0..16384}, new tokens ~ U{1..512}, "
                "32/4 heads, d 128, qk RMSNorm (eps 1e-6, w ~ N(1, 0.1)), sigmoid gate "
                "(logits ~ N(0,1)), RoPE base 1e6")

WORKLOADS = {w.name: w for w in (C1, C2, C3, C4, C5)}


def _normal(gen: torch.Generator, shape, std=1.0, mean=0.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x.to(torch.bfloat16)


def sentinel_fill(shape) -> torch.Tensor:
    return torch.full(shape, SENTINEL_BITS, dtype=torch.int16).view(torch.bfloat16)


@dataclass
class StepInputs:
    """One append + attend step over a packed batch (host tensors)."""
    spec: Spec
    cu_seqlens: torch.Tensor     # int32 [B+1]
    cache_lens: torch.Tensor     # int32 [B], prior lengths
    q: torch.Tensor              # bf16 [T,H,d]
    k: torch.Tensor              # bf16 [T,KV,d]
    v: torch.Tensor              # bf16 [T,KV,d]
    gate: Optional[torch.Tensor]       # bf16 [T,H,d]
    q_norm_w: Optional[torch.Tensor]   # bf16 [d]
    k_norm_w: Optional[torch.Tensor]
    cache_k: torch.Tensor        # bf16 [B,KV,cap,d], history filled, rest sentinel
    cache_v: torch.Tensor

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def batch(self) -> int:
        return int(self.cu_seqlens.numel() - 1)


def make_step(spec: Spec, prior_lens: List[int], new_lens: List[int], capacity: int,
              seed: int, gen: Optional[torch.Generator] = None,
              history: bool = True) -> StepInputs:
    """Draw one packed step: sequences b with prior_lens[b] cached tokens and
    new_lens[b] new ones."""
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    B = len(prior_lens)
    assert len(new_lens) == B
    cu = [0]
    for n in new_lens:
        cu.append(cu[-1] + int(n))
    T = cu[-1]
    H, KV, d = spec.H, spec.KV, spec.d
    q = _normal(gen, (T, H, d), spec.std)
    k = _normal(gen, (T, KV, d), spec.std)
    v = _normal(gen, (T, KV, d), spec.std)
    gate = _normal(gen, (T, H, d)) if spec.out_gate else None
    qw = kw = None
    if spec.qk_norm:
        qw = _normal(gen, (d,), spec.norm_w_std, spec.norm_w_mean)
        kw = _normal(gen, (d,), spec.norm_w_std, spec.norm_w_mean)
    cache_k = sentinel_fill((B, KV, capacity, d))
    cache_v = sentinel_fill((B, KV, capacity, d))
    if history:
        for b in range(B):
            n = int(prior_lens[b])
            if n:
                cache_k[b, :, :n] = _normal(gen, (KV, n, d), spec.std)
                cache_v[b, :, :n] = _normal(gen, (KV, n, d), spec.std)
    return StepInputs(spec=spec, cu_seqlens=torch.tensor(cu, dtype=torch.int32),
                      cache_lens=torch.tensor(prior_lens, dtype=torch.int32), q=q, k=k, v=v,
                      gate=gate, q_norm_w=qw, k_norm_w=kw, cache_k=cache_k, cache_v=cache_v)


def draw_lengths(gen: torch.Generator, n: int, lo: int, hi: int) -> List[int]:
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def make_varlen_step(w: PrefillWorkload, seed: int = 0, history: bool = True) -> StepInputs:
    gen = torch.Generator().manual_seed(seed)
    prior = draw_lengths(gen, w.batch, *w.prior_range)
    new = draw_lengths(gen, w.batch, *w.new_range)
    return make_step(w.spec, prior, new, w.capacity, seed, gen=gen, history=history)


@dataclass
class ChunkedPrompt:
    """A prompt for `batch` sequences fed as equal chunks: the whole prompt's
    Q/K/V are drawn once; chunk c covers tokens [c*chunk, (c+1)*chunk)."""
    spec: Spec
    batch: int
    prompt_len: int
    chunk: int
    capacity: int
    q: torch.Tensor  # [B, L, H, d]
    k: torch.Tensor  # [B, L, KV, d]
    v: torch.Tensor
    gate: Optional[torch.Tensor]
    q_norm_w: Optional[torch.Tensor]
    k_norm_w: Optional[torch.Tensor]

    @property
    def num_chunks(self) -> int:
        return (self.prompt_len + self.chunk - 1) // self.chunk

    def chunk_bounds(self, c: int):
        lo = c * self.chunk
        return lo, min(self.prompt_len, lo + self.chunk)

    def chunk_tensors(self, c: int):
        """Packed [T,.,d] tensors of chunk c, sequences back to back."""
        lo, hi = self.chunk_bounds(c)
        pack = lambda x: None if x is None else x[:, lo:hi].reshape(-1, *x.shape[2:]).contiguous()
        n = hi - lo
        cu = torch.arange(0, self.batch + 1, dtype=torch.int32) * n
        lens = torch.full((self.batch,), lo, dtype=torch.int32)
        return cu, lens, pack(self.q), pack(self.k), pack(self.v), pack(self.gate)


def make_chunked_prompt(w: PrefillWorkload, seed: int = 0) -> ChunkedPrompt:
    gen = torch.Generator().manual_seed(seed)
    s, B, L = w.spec, w.batch, w.prompt_len
    q = _normal(gen, (B, L, s.H, s.d), s.std)
    k = _normal(gen, (B, L, s.KV, s.d), s.std)
    v = _normal(gen, (B, L, s.KV, s.d), s.std)
    gate = _normal(gen, (B, L, s.H, s.d)) if s.out_gate else None
    qw = kw = None
    if s.qk_norm:
        qw = _normal(gen, (s.d,), s.norm_w_std, s.norm_w_mean)
        kw = _normal(gen, (s.d,), s.norm_w_std, s.norm_w_mean)
    return ChunkedPrompt(spec=s, batch=B, prompt_len=L, chunk=w.chunk, capacity=w.capacity,
                         q=q, k=k, v=v, gate=gate, q_norm_w=qw, k_norm_w=kw)


@dataclass
class DecodeInputs:
    spec: Spec
    q: torch.Tensor          # bf16 [B,H,d] (already rotated)
    cache_k: torch.Tensor    # bf16 [B,KV,cap,d] (already rotated keys)
    cache_v: torch.Tensor
    kv_lens: torch.Tensor    # int32 [B], includes the current token
    gate: Optional[torch.Tensor]


def make_decode(spec: Spec, kv_lens: List[int], capacity: int, seed: int,
                gen: Optional[torch.Generator] = None) -> DecodeInputs:
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    B = len(kv_lens)
    q = _normal(gen, (B, spec.H, spec.d), spec.std)
    gate = _normal(gen, (B, spec.H, spec.d)) if spec.out_gate else None
    cache_k = sentinel_fill((B, spec.KV, capacity, spec.d))
    cache_v = sentinel_fill((B, spec.KV, capacity, spec.d))
    for b, n in enumerate(kv_lens):
        if n:
            cache_k[b, :, :n] = _normal(gen, (spec.KV, n, spec.d), spec.std)
            cache_v[b, :, :n] = _normal(gen, (spec.KV, n, spec.d), spec.std)
    return DecodeInputs(spec=spec, q=q, cache_k=cache_k, cache_v=cache_v,
                        kv_lens=torch.tensor(kv_lens, dtype=torch.int32), gate=gate)


def make_decode_workload(w: DecodeWorkload, seed: int = 0) -> DecodeInputs:
    gen = torch.Generator().manual_seed(seed)
    lens = draw_lengths(gen, w.batch, *w.kv_range)
    return make_decode(w.spec, lens, w.capacity, seed, gen=gen)


def make_pair_verify_step(seed: int = 5) -> StepInputs:
    """Speculative pair verify over the decode workload: each of its 64
    sequences (lengths drawn as for the decode, kv_len ~ U{512..8192}) holds
    kv_len - 2 cached tokens and brings 2 drafted ones."""
    gen = torch.Generator().manual_seed(3)
    lens = draw_lengths(gen, C3.batch, *C3.kv_range)
    return make_step(C3.spec, [n - 2 for n in lens], [2] * C3.batch, C3.capacity, seed=seed)


def bf16_to_f64(t: Optional[torch.Tensor]):
    """Exact widening of bf16 data for the oracle (no arithmetic)."""
    if t is None:
        return None
    return t.to(torch.float64).numpy()

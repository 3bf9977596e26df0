"""Benchmark of the attention hot path on one GB300 (one JSON line on stdout).

Headline workload: chunked prefill of a 4096-token prompt in 32 chunks of 128
(32 query heads, 8 KV heads, head_dim 128, RoPE base 5e5).  One step is the
whole path over that prompt: for every chunk, the fused norm + RoPE + cache
append call, then the causal GQA attention call.  `value` is the algorithmic
attention TFLOP/s of the step (4 * d * H * sum over rows of visible keys).

Also measured and reported in the same line (`workloads`): single-token
decode over 64 cached sequences (KV GB/s), long-context YaRN prefill and the
mixed varlen serving step (TFLOP/s), each with the roofline of its dominant
kernel.

Timing: CUDA events on the launching stream, W untimed warm-up steps, then K
timed steps with the L2 flushed (a 256 MiB buffer written) before each; the
step runs as a captured CUDA graph (`value`) and eagerly (`eager`); the
end-to-end number (`e2e`) goes through the public API with host buffers,
host<->device copies included.  `--impl reference` times the f64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------- helpers --

def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--only", choices=["chunked", "decode", "varlen", "yarn", "pair"], default=None,
                    help="time one workload and print its record (profiling runs)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as fh:
                d = json.load(fh)
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(key)
                if isinstance(v, dict):
                    v = v.get("value")
                out[key] = float(v) if v is not None else FALLBACK_PEAKS[key]
            out["source"] = "measured"
            return out
        except Exception:
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed loops run."""
    QUERY = ("index,uuid,clocks.sm,clocks.max.sm,utilization.gpu,power.draw,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"na_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        try:
            uuid = str(torch.cuda.get_device_properties(0).uuid)
        except Exception:
            uuid = ""
        rows = []
        with open(self.path) as fh:
            for line in fh:
                f = [x.strip() for x in line.split(",")]
                if len(f) < 10:
                    continue
                rows.append(f)
        if not rows:
            return None
        if uuid:
            mine = [r for r in rows if uuid in r[1]]
            rows = mine or rows
        if not uuid or not any(uuid in r[1] for r in rows):
            first = rows[0][0]
            rows = [r for r in rows if r[0] == first]
        try:
            loaded = [r for r in rows if float(r[4]) > 0] or rows
            sm = [float(r[2]) for r in loaded]
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            reasons = sorted({names[i] for r in loaded for i in range(4)
                              if r[6 + i].lower().startswith("active")})
            return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(loaded[0][3]),
                    "samples": len(loaded), "reasons": reasons}
        except Exception:
            return None


class Flusher:
    def __init__(self):
        self.buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def __call__(self):
        self.buf.fill_(1)


def kernel_fingerprint(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "causal_gqa_attention_rope_gb300", "csrc", n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def traffic_from_profiles(kernel_file: str, key: str):
    """Per-launch DRAM bytes recorded from an ncu capture (profiles/traffic.json),
    or None when the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as fh:
            d = json.load(fh)
        ent = d.get(key)
        if not ent or ent.get("source_sha") != kernel_fingerprint(kernel_file):
            return None
        return ent.get("bytes_per_launch")
    except Exception:
        return None


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


def causal_flops(H, d, prior, n):
    """4 d H sum over the chunk's rows of visible keys (pos + 1)."""
    return 4.0 * d * H * (n * prior + n * (n + 1) / 2.0)


# ------------------------------------------------------- chunked prefill --

def bench_chunked(wl: W.PrefillWorkload, steps: int, warmup: int, peaks, flush: Flusher,
                  with_e2e=True):
    import causal_gqa_attention_rope_gb300 as na
    s = wl.spec
    prompt = W.make_chunked_prompt(wl, seed=0)
    B, L, H, KV, d = wl.batch, wl.prompt_len, s.H, s.KV, s.d
    assert B == 1
    cfg, rope = attn_cfg(s), rope_cfg(s)
    dev = "cuda"
    q = prompt.q[0].to(dev)
    k = prompt.k[0].to(dev)
    v = prompt.v[0].to(dev)
    gate = None if prompt.gate is None else prompt.gate[0].to(dev)
    qw = None if prompt.q_norm_w is None else prompt.q_norm_w.to(dev)
    kw = None if prompt.k_norm_w is None else prompt.k_norm_w.to(dev)
    cache = na.KVCache(torch.zeros(1, KV, wl.capacity, d, dtype=torch.bfloat16, device=dev),
                       torch.zeros(1, KV, wl.capacity, d, dtype=torch.bfloat16, device=dev))
    q_out = torch.empty_like(q)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    chunks = []
    ws_bytes = 0
    flops_total = 0.0
    launches = 0
    for c in range(prompt.num_chunks):
        lo, hi = prompt.chunk_bounds(c)
        n = hi - lo
        cu = torch.tensor([0, n], dtype=torch.int32, device=dev)
        lens = torch.tensor([lo], dtype=torch.int32, device=dev)
        wsb = na.na_prefill_workspace_size(cfg, 1, n, n, hi)
        ws_bytes = max(ws_bytes, wsb)
        f = causal_flops(H, d, lo, n)
        flops_total += f
        launches += 1 + 1 + (1 if wsb > 0 else 0)
        # the chunk's views of the prompt buffers, made once as a serving loop would
        views = (q[lo:hi], k[lo:hi], v[lo:hi], q_out[lo:hi], out[lo:hi],
                 None if gate is None else gate[lo:hi])
        chunks.append((lo, hi, n, cu, lens, f, views))
    ws = na.workspace(ws_bytes, dev)

    def run(events=None):
        for i, (lo, hi, n, cu, lens, f, (qc, kc, vc, qoc, oc, gc)) in enumerate(chunks):
            na.na_rope_append_kv(cfg, rope, cu, lens, qc, kc, vc, qoc, cache, q_norm_w=qw,
                                 k_norm_w=kw, status=status)
            if events is not None:
                events[i][0].record()
            na.na_attn_prefill_chunk(cfg, cu, lens, n, hi, qoc, cache, oc, gate=gc, workspace=ws,
                                     status=status)
            if events is not None:
                events[i][1].record()

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    # graph-captured step
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        run()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    g_times = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        g_times.append(a.elapsed_time(b))

    # eager step with per-launch events on the attention calls (the GPU is kept
    # behind the host by a short spin so the events time the kernels, not the
    # host's launch rate)
    e_times, k_durs = [], []
    for _ in range(steps):
        flush()
        torch.cuda._sleep(20_000_000)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in chunks]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run(evs)
        b.record()
        torch.cuda.synchronize()
        e_times.append(a.elapsed_time(b))
        k_durs.append(sum(x.elapsed_time(y) for x, y in evs))
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    res = {
        "flops_per_step": flops_total,
        "graph_ms": statistics.mean(g_times),
        "eager_ms": statistics.mean(e_times),
        "attn_kernel_ms_per_step": statistics.mean(k_durs),
        "launches_per_step": launches,
        "attn_launches_per_step": len(chunks),
    }
    achieved = flops_total / (res["attn_kernel_ms_per_step"] * 1e-3) / 1e12
    res["roofline"] = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                       "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                       "traffic": traffic_from_profiles("prefill.cu", wl.name),
                       "kernel": "na_attn_prefill_chunk (prefill split pass + combine)",
                       "peak_source": peaks["source"] + " bf16 burst"}

    if with_e2e:
        hq, hk, hv = (x.pin_memory() for x in (prompt.q[0], prompt.k[0], prompt.v[0]))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        e2e = []
        for _ in range(max(1, steps // 2)):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            run()
            hout.copy_(out, non_blocking=True)
            b.record()
            torch.cuda.synchronize()
            e2e.append(a.elapsed_time(b))
        res["e2e_ms"] = statistics.mean(e2e)
        res["h2d_bytes"] = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
        res["d2h_bytes"] = hout.numel() * hout.element_size()
    return res


# ------------------------------------------------------------ varlen step --

def bench_varlen(wl: W.PrefillWorkload, steps, warmup, peaks, flush):
    import causal_gqa_attention_rope_gb300 as na
    s = wl.spec
    step = W.make_varlen_step(wl, seed=0)
    dev = "cuda"
    cfg, rope = attn_cfg(s), rope_cfg(s)
    cu, lens = step.cu_seqlens.to(dev), step.cache_lens.to(dev)
    q, k, v = step.q.to(dev), step.k.to(dev), step.v.to(dev)
    gate = None if step.gate is None else step.gate.to(dev)
    qw = None if step.q_norm_w is None else step.q_norm_w.to(dev)
    kw = None if step.k_norm_w is None else step.k_norm_w.to(dev)
    ck0, cv0 = step.cache_k.to(dev), step.cache_v.to(dev)
    cache = na.KVCache(ck0.clone(), cv0.clone())
    T = step.total_tokens
    new = (step.cu_seqlens[1:] - step.cu_seqlens[:-1])
    max_new = int(new.max())
    max_total = int((step.cache_lens + new).max())
    ws = na.workspace(na.na_prefill_workspace_size(cfg, step.batch, T, max_new, max_total), dev)
    q_out, out = torch.empty_like(q), torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flops = sum(causal_flops(s.H, s.d, int(p), int(n))
                for p, n in zip(step.cache_lens.tolist(), new.tolist()))

    def run(ev=None):
        na.na_rope_append_kv(cfg, rope, cu, lens, q, k, v, q_out, cache, q_norm_w=qw, k_norm_w=kw,
                             status=status)
        if ev:
            ev[0].record()
        na.na_attn_prefill_chunk(cfg, cu, lens, max_new, max_total, q_out, cache, out, gate=gate,
                                 workspace=ws, status=status)
        if ev:
            ev[1].record()

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    times, kd = [], []
    for _ in range(steps):
        flush()
        torch.cuda._sleep(5_000_000)
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run(ev)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
        kd.append(ev[0].elapsed_time(ev[1]))
    assert int(status.item()) == 0
    ms, kms = statistics.mean(times), statistics.mean(kd)
    ach = flops / (kms * 1e-3) / 1e12
    return {"workload": wl.name, "metric": "prefill attn TFLOP/s", "unit": "TFLOP/s",
            "value": flops / (ms * 1e-3) / 1e12, "ms_per_step": ms, "tokens": T,
            "flops_per_step": flops,
            "roofline": {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                         "traffic": traffic_from_profiles("prefill.cu", wl.name),
                         "kernel": "na_attn_prefill_chunk",
                         "peak_source": peaks["source"] + " bf16 burst"}}


# ---------------------------------------------------------------- decode --

def bench_decode(wl: W.DecodeWorkload, steps, warmup, peaks, flush):
    import causal_gqa_attention_rope_gb300 as na
    s = wl.spec
    dec = W.make_decode_workload(wl, seed=0)
    dev = "cuda"
    B, H, KV, d = wl.batch, s.H, s.KV, s.d
    cfg, rope = attn_cfg(s), rope_cfg(s)
    cache = na.KVCache(dec.cache_k.to(dev), dec.cache_v.to(dev))
    kv_lens = dec.kv_lens.to(dev)
    max_kv = int(dec.kv_lens.max())
    # the current token: append its K/V at position kv_len - 1, then attend
    gen = torch.Generator().manual_seed(1)
    q_new = dec.q.to(dev)
    k_new = torch.randn(B, KV, d, generator=gen).to(torch.bfloat16).to(dev)
    v_new = torch.randn(B, KV, d, generator=gen).to(torch.bfloat16).to(dev)
    cu = torch.arange(0, B + 1, dtype=torch.int32, device=dev)
    prior = (kv_lens - 1).to(torch.int32)
    q_rot = torch.empty_like(q_new)
    out = torch.empty_like(q_new)
    stride = (max_kv + 3) // 4 * 4  # 16-byte rows: the probability passes use 16-byte accesses
    probs = torch.empty(B, H, stride, dtype=torch.float32, device=dev)
    ws = na.workspace(na.na_decode_workspace_size(cfg, B, max_kv), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lens = dec.kv_lens.tolist()
    kv_bytes = sum(lens) * KV * d * 2 * 2
    probs_bytes = sum(lens) * H * 4
    io_bytes = 2 * B * H * d * 2
    alg_bytes = kv_bytes + probs_bytes + io_bytes

    def run(ev=None):
        na.na_rope_append_kv(cfg, rope, cu, prior, q_new, k_new, v_new, q_rot, cache,
                             status=status)
        if ev:
            ev[0].record()
        na.na_attn_decode(cfg, q_rot, cache, kv_lens, max_kv, out, probs=probs, workspace=ws,
                          status=status)
        if ev:
            ev[1].record()

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    times, kd = [], []
    for _ in range(steps):
        flush()
        torch.cuda._sleep(5_000_000)
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run(ev)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
        kd.append(ev[0].elapsed_time(ev[1]))
    assert int(status.item()) == 0
    ms, kms = statistics.mean(times), statistics.mean(kd)
    ach = alg_bytes / (kms * 1e-3) / 1e9

    # Born-rule importance of the step, accumulated into a running per-key
    # buffer (reads every head's probabilities, reads and writes the buffer).
    imp = torch.zeros(B, stride, dtype=torch.float32, device=dev)
    imp_bytes = sum(lens) * (H * 4 + 2 * 4)
    for _ in range(warmup):
        na.na_decode_importance(cfg, probs, kv_lens, max_kv, imp, accumulate=True, status=status)
    torch.cuda.synchronize()
    it = []
    for _ in range(steps):
        flush()
        torch.cuda._sleep(5_000_000)  # host lead: the launch is queued before the start event runs
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        na.na_decode_importance(cfg, probs, kv_lens, max_kv, imp, accumulate=True, status=status)
        b.record()
        torch.cuda.synchronize()
        it.append(a.elapsed_time(b))
    assert int(status.item()) == 0
    ims = statistics.mean(it)
    iach = imp_bytes / (ims * 1e-3) / 1e9
    # The same decode with the importance summed in its merge pass (one call):
    # the K/V, the probabilities once (written) and the running importance
    # (read and written) per step.
    def run_fused(ev=None):
        na.na_rope_append_kv(cfg, rope, cu, prior, q_new, k_new, v_new, q_rot, cache,
                             status=status)
        if ev:
            ev[0].record()
        na.na_attn_decode_imp(cfg, q_rot, cache, kv_lens, max_kv, out, probs, imp,
                              accumulate=True, workspace=ws, status=status)
        if ev:
            ev[1].record()

    for _ in range(warmup):
        run_fused()
    torch.cuda.synchronize()
    ft, fk = [], []
    for _ in range(steps):
        flush()
        torch.cuda._sleep(5_000_000)
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run_fused(ev)
        b.record()
        torch.cuda.synchronize()
        ft.append(a.elapsed_time(b))
        fk.append(ev[0].elapsed_time(ev[1]))
    assert int(status.item()) == 0
    fms, fkms = statistics.mean(ft), statistics.mean(fk)
    fused_bytes = alg_bytes + sum(lens) * 2 * 4
    fach = fused_bytes / (fkms * 1e-3) / 1e9
    fused = {"workload": "decode_imp_" + wl.name, "metric": "decode+importance KV GB/s",
             "unit": "GB/s", "value": (fused_bytes + B * 3 * KV * d * 2) / (fms * 1e-3) / 1e9,
             "ms_per_step": fms, "bytes_per_step": fused_bytes,
             "roofline": {"bound": "hbm", "achieved": fach, "peak": peaks["hbm_gbs"],
                          "unit": "GB/s", "frac": fach / peaks["hbm_gbs"],
                          "traffic": traffic_from_profiles("decode.cu", "decode_imp_" + wl.name),
                          "kernel": "na_attn_decode_imp (split pass + merge pass with importance)",
                          "peak_source": peaks["source"] + " HBM copy"}}

    importance = {"workload": "importance_" + wl.name, "metric": "importance GB/s", "unit": "GB/s",
                  "value": iach, "ms_per_step": ims, "bytes_per_step": imp_bytes,
                  "roofline": {"bound": "hbm", "achieved": iach, "peak": peaks["hbm_gbs"],
                               "unit": "GB/s", "frac": iach / peaks["hbm_gbs"],
                               "traffic": traffic_from_profiles("importance.cu",
                                                                "importance_" + wl.name),
                               "kernel": "na_decode_importance",
                               "peak_source": peaks["source"] + " HBM copy"}}
    return {"workload": wl.name, "metric": "decode KV GB/s", "unit": "GB/s",
            "value": (alg_bytes + B * 3 * KV * d * 2) / (ms * 1e-3) / 1e9, "ms_per_step": ms,
            "bytes_per_step": alg_bytes,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"],
                         "traffic": traffic_from_profiles("decode.cu", wl.name),
                         "kernel": "na_attn_decode (split pass + combine)",
                         "peak_source": peaks["source"] + " HBM copy"},
            "importance": importance, "fused": fused}


def bench_pair_verify(steps, warmup, peaks, flush):
    """Speculative pair verify: every sequence of the decode workload checks two
    drafted tokens (a 2-token chunk after kv_len - 2 cached ones).  HBM-bound:
    the K/V of each (sequence, kv head) is streamed once for both tokens and
    all query heads of the group (GQA-packed tiles)."""
    import causal_gqa_attention_rope_gb300 as na
    wl = W.C3
    s = wl.spec
    gen = torch.Generator().manual_seed(3)
    lens = W.draw_lengths(gen, wl.batch, *wl.kv_range)
    step = W.make_step(s, [n - 2 for n in lens], [2] * wl.batch, wl.capacity, seed=5)
    dev = "cuda"
    cfg = attn_cfg(s)
    cu, cl = step.cu_seqlens.to(dev), step.cache_lens.to(dev)
    q = step.q.to(dev)
    out = torch.empty_like(q)
    cache = na.KVCache(step.cache_k.to(dev), step.cache_v.to(dev))
    T, mt = int(step.cu_seqlens[-1]), max(lens)
    ws = na.workspace(na.na_prefill_workspace_size(cfg, wl.batch, T, 2, mt), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def run():
        na.na_attn_prefill_chunk(cfg, cu, cl, 2, mt, q, cache, out, workspace=ws, status=status)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    assert int(status.item()) == 0
    ms = statistics.mean(ts)
    kv_bytes = sum(lens) * s.KV * s.d * 2 * 2
    ach = kv_bytes / (ms * 1e-3) / 1e9
    name = "pair_verify_b64_h32kv8d128_kv512to8192"
    return {"workload": name, "metric": "pair verify KV GB/s", "unit": "GB/s", "value": ach,
            "ms_per_step": ms, "bytes_per_step": kv_bytes,
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"], "traffic": traffic_from_profiles("prefill.cu", name),
                         "kernel": "na_attn_prefill_chunk (2-token chunks, GQA-packed tiles)",
                         "peak_source": peaks["source"] + " HBM copy"}}


# ---------------------------------------------------- oracle (CPU) timing --

def cpu_baseline_chunked(wl: W.PrefillWorkload, budget_s: float):
    """Time the f64 oracle on a bounded sample: the RoPE + append of the whole
    prompt, then as many attention rows (evenly spread over the prompt) as fit
    the budget.  Returns TFLOP/s over the sampled rows' algorithmic flops."""
    import numpy as np
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from harness import oracle_append, oracle_rows, prompt_as_step
    o = oracle.load()
    prompt = W.make_chunked_prompt(wl, seed=0)
    step = prompt_as_step(prompt)
    s = wl.spec
    t0 = time.perf_counter()
    ost = oracle_append(o, step)
    t_append = time.perf_counter() - t0
    L = wl.prompt_len
    rows, spent, flops = [], 0.0, 0.0
    order = np.linspace(0, L - 1, 64).astype(int).tolist()
    i = 0
    while spent < budget_s and i < len(order) * 64:
        r = order[i % len(order)] if i < len(order) else int(np.random.default_rng(i).integers(L))
        t0 = time.perf_counter()
        oracle_rows(o, step, ost, [r])
        spent += time.perf_counter() - t0
        flops += 4.0 * s.d * s.H * (r + 1)
        rows.append(r)
        i += 1
    return {"value": flops / spent / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"RoPE+append of all {L} tokens ({t_append:.2f} s, not in the rate) and "
                      f"causal attention of {len(rows)} rows x {s.H} heads spread over the "
                      f"prompt ({spent:.1f} s, {flops / 1e9:.2f} GFLOP), single thread f64",
            "host_cores_available": len(os.sched_getaffinity(0))}


# ------------------------------------------------------------------ main --

def main():
    args = parse_args()
    rank, world, local = dist_setup(args)
    wl = W.C2
    base = {"metric": "prefill attn TFLOP/s", "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "description": wl.description,
                       "heads": wl.spec.H, "kv_heads": wl.spec.KV, "head_dim": wl.spec.d,
                       "prompt_len": wl.prompt_len, "chunk": wl.chunk,
                       "parallelism": f"replicas{args.gpus}",
                       "l2": "flushed (256 MiB write) before every timed step",
                       "launch": "CUDA graph of the 32 chunk call pairs"}}

    if args.impl == "reference":
        if rank != 0:
            return
        budget = max(2.0, min(20.0, args.cpu_budget / max(1, args.steps)))
        vals, samples = [], None
        for i in range(args.warmup + args.steps):
            cb = cpu_baseline_chunked(wl, budget)
            if i >= args.warmup:
                vals.append(cb["value"])
                samples = cb
        v = statistics.mean(vals)
        flops = causal_flops(wl.spec.H, wl.spec.d, 0, wl.prompt_len)
        line = dict(base, impl="reference", value=v, ms_per_step=flops / (v * 1e12) * 1e3,
                    cpu_baseline=dict(samples, value=v),
                    e2e={"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                         "d2h_bytes_per_step": 0})
        line["config"] = dict(base["config"], launch="CPU oracle, single thread")
        print(json.dumps(line))
        return

    torch.cuda.set_device(local)
    import causal_gqa_attention_rope_gb300 as na
    na.load_library()
    peaks = load_peaks()
    flush = Flusher()
    if args.only:
        fn = {"chunked": lambda: bench_chunked(W.C2, args.steps, args.warmup, peaks, flush, False),
              "decode": lambda: bench_decode(W.C3, args.steps, args.warmup, peaks, flush),
              "pair": lambda: bench_pair_verify(args.steps, args.warmup, peaks, flush),
              "varlen": lambda: bench_varlen(W.C5, args.steps, args.warmup, peaks, flush),
              "yarn": lambda: bench_chunked(W.C4, args.steps, args.warmup, peaks, flush, False)}
        rec = fn[args.only]()
        if rank == 0:
            print(json.dumps(dict(rec, only=args.only)))
        return
    sampler = ClockSampler()
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    r = bench_chunked(wl, args.steps, args.warmup, peaks, flush)
    extra = []
    if not args.no_extra:
        dec_rec = bench_decode(W.C3, args.steps, args.warmup, peaks, flush)
        extra.append({k: v for k, v in dec_rec.items() if k not in ("importance", "fused")})
        extra.append(dec_rec["importance"])
        extra.append(dec_rec["fused"])
        extra.append(bench_pair_verify(args.steps, args.warmup, peaks, flush))
        extra.append(bench_varlen(W.C5, args.steps, args.warmup, peaks, flush))
        r4 = bench_chunked(W.C4, max(2, args.steps // 4), min(args.warmup, 3), peaks, flush,
                           with_e2e=False)
        extra.append({"workload": W.C4.name, "metric": "prefill attn TFLOP/s", "unit": "TFLOP/s",
                      "value": r4["flops_per_step"] / (r4["graph_ms"] * 1e-3) / 1e12,
                      "ms_per_step": r4["graph_ms"], "eager_ms": r4["eager_ms"],
                      "roofline": r4["roofline"]})
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()

    ms = max_over_ranks(r["graph_ms"], world)
    value = r["flops_per_step"] * world / (ms * 1e-3) / 1e12
    e2e_ms = max_over_ranks(r["e2e_ms"], world)
    line = dict(base, value=value, ms_per_step=ms)
    line["e2e"] = {"value": r["flops_per_step"] * world / (e2e_ms * 1e-3) / 1e12,
                   "unit": "TFLOP/s", "h2d_bytes_per_step": r["h2d_bytes"],
                   "d2h_bytes_per_step": r["d2h_bytes"], "ms_per_step": e2e_ms,
                   "api": "na_rope_append_kv + na_attn_prefill_chunk per chunk, eager, pinned "
                          "host inputs copied in and output copied out each step"}
    line["eager"] = {"value": r["flops_per_step"] / (r["eager_ms"] * 1e-3) / 1e12,
                     "ms_per_step": r["eager_ms"]}
    line["gpu_launches"] = r["launches_per_step"] * args.steps
    line["roofline"] = r["roofline"]
    line["clocks"] = clocks
    line["workloads"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_chunked(wl, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()

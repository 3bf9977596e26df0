"""Benchmark of the attention hot path on one GB300 (one JSON line on stdout).

Headline workload: long-context YaRN prefill, the largest single-GPU
configuration -- one sequence of 32768 tokens fed in 16 chunks of 2048 (40
query heads, 8 KV heads, head_dim 128, partial rotary 64, YaRN base 1e6 x4).
One step is the whole path over that prompt: for every chunk, the fused
norm + RoPE + cache append call, then the causal GQA attention call.  `value`
is the algorithmic attention TFLOP/s of the step (4 * d * H * sum over rows of
visible keys) replayed as a CUDA graph.

Also measured in the same line (`workloads`), each with its own roofline and
its own CPU oracle baseline: the single-chunk 128-token parity workload (us
and TFLOP/s), chunked prefill of 4096 tokens in 32 chunks of 128, single-token
decode over 64 cached sequences (KV GB/s, with the importance pass),
speculative pair verify, and the mixed varlen serving step.

Timing: CUDA events on the launching stream around graph replays, W untimed
warm-up replays, then K timed replays with the L2 flushed (a 256 MiB buffer
written, then another read, outside the timed region) before each; every figure is the median of
the K timed replays, with min and max beside it.  A roofline's `achieved` is
the dominant call's algorithmic work over the median replay time of a graph
that holds only that call (for a chunked prompt: the step's attention calls,
over the cache the step fills), so it is measured in the same launch
configuration as the step and never exceeds it.  The end-to-end figure (`e2e`)
runs the headline step through the public API with host buffers: the prompt
is copied in from pinned host memory and the output copied back inside the
timed region.  Chunked prompts are also timed eager (`eager`: the same calls
launched from Python every step, device buffers, same flushes).
`--impl reference` times the f64 CPU oracle on a bounded sample of the
headline workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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
NOMINAL_HBM_GBS = 8000.0  # "about 8 TB/s", the decode target's reference bandwidth


# --------------------------------------------------------------- helpers --

def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--cpu-budget", type=float, default=16.0,
                    help="seconds of oracle work over all workloads")
    ap.add_argument("--only", choices=["c1", "chunked", "decode", "varlen", "yarn", "pair"],
                    default=None, help="time one workload and print its record (profiling runs)")
    return ap.parse_args(argv)


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
    """Evicts every line of the workload from the L2 before a timed step: a
    256 MiB buffer is written, then a second 256 MiB buffer is read, so the L2
    is left holding clean lines of that second buffer -- no line the step
    reads, and no dirty line of the flush itself whose write-back would be
    charged to the step."""

    def __init__(self):
        self.buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
        self.rd = torch.ones(64 * 1024 * 1024, dtype=torch.int32, device="cuda")
        self.acc = torch.empty((), dtype=torch.int64, device="cuda")

    def __call__(self):
        self.buf.fill_(1)
        torch.sum(self.rd, dim=0, out=self.acc)
        # ~50 us of GPU spin, so the timed launches that follow are queued
        # before the GPU reaches them (no host latency inside the timed region)
        torch.cuda._sleep(100000)


def spread(xs):
    """Median with min and max (ms)."""
    return {"median": statistics.median(xs), "min": min(xs), "max": max(xs), "n": len(xs)}


def capture(run):
    """`run` captured as a CUDA graph (after one warm run on a side stream)."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        run()
    torch.cuda.synchronize()
    return g


def time_graph(g, steps, warmup, flush):
    """Milliseconds of `steps` replays, each after an L2 flush (not timed)."""
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return ts


def time_eager(run, steps, warmup, flush):
    """Milliseconds of `steps` eager runs (the calls launched from Python each
    time), each after an L2 flush (not timed)."""
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
    return ts


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


def tensor_roofline(flops, ms, peaks, kernel, traffic):
    ach = flops / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": ach / peaks["bf16_tflops"], "traffic": traffic, "kernel": kernel,
            "peak_source": peaks["source"] + " bf16 burst",
            "frac_of_sustained": ach / peaks["bf16_tflops_sustained"]}


def hbm_roofline(nbytes, ms, peaks, kernel, traffic):
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": ach / peaks["hbm_gbs"], "traffic": traffic, "kernel": kernel,
            "peak_source": peaks["source"] + " HBM copy",
            "frac_of_nominal_8tbs": ach / NOMINAL_HBM_GBS}


# ------------------------------------------------------- chunked prefill --

def bench_chunked(wl: W.PrefillWorkload, steps: int, warmup: int, peaks, flush,
                  with_e2e=False):
    """A prompt fed chunk by chunk: append + attend per chunk, as one graph."""
    import causal_gqa_attention_rope_gb300 as na
    s = wl.spec
    prompt = W.make_chunked_prompt(wl, seed=0)
    H, KV, d = s.H, s.KV, s.d
    assert wl.batch == 1
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
    attn_launches = 0
    for c in range(prompt.num_chunks):
        lo, hi = prompt.chunk_bounds(c)
        n = hi - lo
        cu = torch.tensor([0, n], dtype=torch.int32, device=dev)
        lens = torch.tensor([lo], dtype=torch.int32, device=dev)
        wsb = na.na_prefill_workspace_size(cfg, 1, n, n, hi)
        ws_bytes = max(ws_bytes, wsb)
        flops_total += causal_flops(H, d, lo, n)
        attn_launches += 1 + (1 if wsb > 0 else 0)
        # the chunk's views of the prompt buffers, made once as a serving loop would
        views = (q[lo:hi], k[lo:hi], v[lo:hi], q_out[lo:hi], out[lo:hi],
                 None if gate is None else gate[lo:hi])
        chunks.append((lo, hi, n, cu, lens, views))
    ws = na.workspace(ws_bytes, dev)

    def append(i):
        lo, hi, n, cu, lens, (qc, kc, vc, qoc, oc, gc) = chunks[i]
        na.na_rope_append_kv(cfg, rope, cu, lens, qc, kc, vc, qoc, cache, q_norm_w=qw,
                             k_norm_w=kw, status=status)

    def attend(i):
        lo, hi, n, cu, lens, (qc, kc, vc, qoc, oc, gc) = chunks[i]
        na.na_attn_prefill_chunk(cfg, cu, lens, n, hi, qoc, cache, oc, gate=gc, workspace=ws,
                                 status=status)

    def run_step():
        for i in range(len(chunks)):
            append(i)
            attend(i)

    def run_attn():
        for i in range(len(chunks)):
            attend(i)

    for _ in range(warmup):
        run_step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    g_step, g_attn = capture(run_step), capture(run_attn)
    step_ms = time_graph(g_step, steps, warmup, flush)
    attn_ms = time_graph(g_attn, steps, warmup, flush)
    eager_ms = time_eager(run_step, steps, warmup, flush)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    launches = len(chunks) + attn_launches
    st, at, et = spread(step_ms), spread(attn_ms), spread(eager_ms)
    res = {"workload": wl.name, "metric": "prefill attn TFLOP/s", "unit": "TFLOP/s",
           "value": flops_total / (st["median"] * 1e-3) / 1e12, "ms_per_step": st["median"],
           "ms_spread": st, "flops_per_step": flops_total, "launches_per_step": launches,
           "attn_calls_ms": at,
           "eager": {"value": flops_total / (et["median"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                     "ms_per_step": et["median"], "ms_spread": et,
                     "launch": "the same calls launched from Python every step (no graph), "
                               "device buffers"},
           "roofline": tensor_roofline(flops_total, at["median"], peaks,
                                       "na_attn_prefill_chunk (its calls of the step, graph-"
                                       "replayed)", traffic_from_profiles("prefill.cu", wl.name))}

    if with_e2e:
        # The step through the public API with host buffers, pipelined as a
        # serving loop would: chunk c's Q/K/V are copied in on one stream and
        # its output copied back on another, so the copies of other chunks
        # overlap the kernels of chunk c.  Every byte crosses inside the timed
        # region: it opens before the first copy-in and closes after the last
        # copy-out.
        hq, hk, hv = (x.pin_memory() for x in (prompt.q[0], prompt.k[0], prompt.v[0]))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        comp = torch.cuda.current_stream()
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        e2e = []
        for i in range(max(1, steps // 2) + 1):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(comp)
            h2d.wait_event(a)
            ins = []
            with torch.cuda.stream(h2d):
                for (lo, hi, n, cu, lens, views) in chunks:
                    q[lo:hi].copy_(hq[lo:hi], non_blocking=True)
                    k[lo:hi].copy_(hk[lo:hi], non_blocking=True)
                    v[lo:hi].copy_(hv[lo:hi], non_blocking=True)
                    e = ev()
                    e.record(h2d)
                    ins.append(e)
            for c, (lo, hi, n, cu, lens, views) in enumerate(chunks):
                comp.wait_event(ins[c])
                append(c)
                attend(c)
                e = ev()
                e.record(comp)
                d2h.wait_event(e)
                with torch.cuda.stream(d2h):
                    hout[lo:hi].copy_(out[lo:hi], non_blocking=True)
            comp.wait_stream(d2h)
            b.record(comp)
            torch.cuda.synchronize()
            if i > 0:  # the first is a warm-up of the host path
                e2e.append(a.elapsed_time(b))
        es = spread(e2e)
        res["e2e"] = {"value": flops_total / (es["median"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                      "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in (hq, hk, hv)),
                      "d2h_bytes_per_step": hout.numel() * hout.element_size(),
                      "ms_per_step": es["median"], "ms_spread": es,
                      "api": "na_rope_append_kv + na_attn_prefill_chunk per chunk, eager; each "
                             "chunk's Q/K/V copied in from pinned host memory on a copy stream "
                             "and its output copied back on another, overlapping the kernels of "
                             "the other chunks; all copies inside the timed region"}
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
    cache = na.KVCache(step.cache_k.to(dev), step.cache_v.to(dev))
    T = step.total_tokens
    new = (step.cu_seqlens[1:] - step.cu_seqlens[:-1])
    max_new = int(new.max())
    max_total = int((step.cache_lens + new).max())
    wsb = na.na_prefill_workspace_size(cfg, step.batch, T, max_new, max_total)
    ws = na.workspace(wsb, dev)
    q_out, out = torch.empty_like(q), torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flops = sum(causal_flops(s.H, s.d, int(p), int(n))
                for p, n in zip(step.cache_lens.tolist(), new.tolist()))

    def attend():
        na.na_attn_prefill_chunk(cfg, cu, lens, max_new, max_total, q_out, cache, out, gate=gate,
                                 workspace=ws, status=status)

    def run():
        na.na_rope_append_kv(cfg, rope, cu, lens, q, k, v, q_out, cache, q_norm_w=qw, k_norm_w=kw,
                             status=status)
        attend()

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    st = spread(time_graph(capture(run), steps, warmup, flush))
    kt = spread(time_graph(capture(attend), steps, warmup, flush))
    assert int(status.item()) == 0
    return {"workload": wl.name, "metric": "prefill attn TFLOP/s", "unit": "TFLOP/s",
            "value": flops / (st["median"] * 1e-3) / 1e12, "ms_per_step": st["median"],
            "ms_spread": st, "attn_call_ms": kt, "tokens": T, "flops_per_step": flops,
            "launches_per_step": 2 + (1 if wsb > 0 else 0),
            "roofline": tensor_roofline(flops, kt["median"], peaks, "na_attn_prefill_chunk",
                                        traffic_from_profiles("prefill.cu", wl.name))}


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
    imp = torch.zeros(B, stride, dtype=torch.float32, device=dev)
    ws = na.workspace(na.na_decode_workspace_size(cfg, B, max_kv), dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lens = dec.kv_lens.tolist()
    kv_bytes = sum(lens) * KV * d * 2 * 2
    probs_bytes = sum(lens) * H * 4
    io_bytes = 2 * B * H * d * 2
    alg_bytes = kv_bytes + probs_bytes + io_bytes
    append_bytes = B * 3 * KV * d * 2  # new K/V read and written, roughly (context for `value`)

    def append():
        na.na_rope_append_kv(cfg, rope, cu, prior, q_new, k_new, v_new, q_rot, cache,
                             status=status)

    def decode():
        na.na_attn_decode(cfg, q_rot, cache, kv_lens, max_kv, out, probs=probs, workspace=ws,
                          status=status)

    def importance():  # accumulated into a running per-key buffer
        na.na_decode_importance(cfg, probs, kv_lens, max_kv, imp, accumulate=True, status=status)

    def step():
        append()
        decode()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    st = spread(time_graph(capture(step), steps, warmup, flush))
    kt = spread(time_graph(capture(decode), steps, warmup, flush))
    it = spread(time_graph(capture(importance), steps, warmup, flush))
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    imp_bytes = sum(lens) * (H * 4 + 2 * 4)
    importance_rec = {
        "workload": "importance_" + wl.name, "metric": "importance GB/s", "unit": "GB/s",
        "value": imp_bytes / (it["median"] * 1e-3) / 1e9, "ms_per_step": it["median"],
        "ms_spread": it, "bytes_per_step": imp_bytes,
        "roofline": hbm_roofline(imp_bytes, it["median"], peaks, "na_decode_importance",
                                 traffic_from_profiles("importance.cu", "importance_" + wl.name))}
    return {"workload": wl.name, "metric": "decode KV GB/s", "unit": "GB/s",
            "value": (alg_bytes + append_bytes) / (st["median"] * 1e-3) / 1e9,
            "ms_per_step": st["median"], "ms_spread": st, "decode_call_ms": kt,
            "bytes_per_step": alg_bytes, "launches_per_step": 3,
            "roofline": hbm_roofline(alg_bytes, kt["median"], peaks,
                                     "na_attn_decode (split pass + combine)",
                                     traffic_from_profiles("decode.cu", wl.name)),
            "importance": importance_rec}


def bench_pair_verify(steps, warmup, peaks, flush):
    """Speculative pair verify: every sequence of the decode workload checks two
    drafted tokens (a 2-token chunk after kv_len - 2 cached ones).  A step is
    the append of the drafted tokens, then the attention call, which is
    HBM-bound: the K/V of each (sequence, kv head) is streamed once for both
    tokens and all query heads of the group (GQA-packed tiles)."""
    import causal_gqa_attention_rope_gb300 as na
    wl = W.C3
    s = wl.spec
    step = W.make_pair_verify_step()
    lens = [int(x) + 2 for x in step.cache_lens.tolist()]
    dev = "cuda"
    cfg, rope = attn_cfg(s), rope_cfg(s)
    cu, cl = step.cu_seqlens.to(dev), step.cache_lens.to(dev)
    q, k, v = step.q.to(dev), step.k.to(dev), step.v.to(dev)
    q_out, out = torch.empty_like(q), torch.empty_like(q)
    cache = na.KVCache(step.cache_k.to(dev), step.cache_v.to(dev))
    T, mt = int(step.cu_seqlens[-1]), max(lens)
    wsb = na.na_prefill_workspace_size(cfg, wl.batch, T, 2, mt)
    ws = na.workspace(wsb, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def attend():
        na.na_attn_prefill_chunk(cfg, cu, cl, 2, mt, q_out, cache, out, workspace=ws,
                                 status=status)

    def run():
        na.na_rope_append_kv(cfg, rope, cu, cl, q, k, v, q_out, cache, status=status)
        attend()

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    st = spread(time_graph(capture(run), steps, warmup, flush))
    kt = spread(time_graph(capture(attend), steps, warmup, flush))
    assert int(status.item()) == 0
    kv_bytes = sum(lens) * s.KV * s.d * 2 * 2
    name = "pair_verify_b64_h32kv8d128_kv512to8192"
    return {"workload": name, "metric": "pair verify KV GB/s", "unit": "GB/s",
            "value": kv_bytes / (st["median"] * 1e-3) / 1e9, "ms_per_step": st["median"],
            "ms_spread": st, "attn_call_ms": kt, "bytes_per_step": kv_bytes,
            "launches_per_step": 2 + (1 if wsb > 0 else 0),
            "roofline": hbm_roofline(kv_bytes, kt["median"], peaks,
                                     "na_attn_prefill_chunk (2-token chunks, GQA-packed tiles)",
                                     traffic_from_profiles("prefill.cu", name))}


# ---------------------------------------------------- oracle (CPU) timing --
# The oracle as it stands (plain C, f64, one thread) on the host cores of the
# box.  Work that runs in seconds is timed in full; the large workloads are
# timed on a seeded sample and labelled with the sample and an extrapolation
# of the full workload's time at the measured rate.

def _oracle_tools():
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import harness
    return oracle.load(), harness


def _host_cores():
    return len(os.sched_getaffinity(0))


def cpu_baseline_rows(step: W.StepInputs, rows, budget_s: float, full_flops: float, what: str):
    """RoPE + append of every new token of `step`, then the listed attention
    rows (all heads) in order until the budget is spent; TFLOP/s of the timed
    rows' algorithmic flops."""
    o, h = _oracle_tools()
    s = step.spec
    t0 = time.perf_counter()
    ost = h.oracle_append(o, step)
    t_append = time.perf_counter() - t0
    cu, prior = step.cu_seqlens.tolist(), step.cache_lens.tolist()

    def pos_of(t):
        b = max(i for i in range(step.batch) if cu[i] <= t)
        return prior[b] + t - cu[b]

    spent, flops, done = 0.0, 0.0, 0
    for r in rows:
        if spent >= budget_s:
            break
        t0 = time.perf_counter()
        h.oracle_rows(o, step, ost, [r])
        spent += time.perf_counter() - t0
        flops += 4.0 * s.d * s.H * (pos_of(r) + 1)
        done += 1
    rate = flops / spent / 1e12
    full = done == len(rows)
    return {"value": rate, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": (f"{what}: RoPE+append of all {step.total_tokens} tokens ({t_append:.2f} s, "
                       f"not in the rate), then causal attention of {done} of {len(rows)} listed "
                       f"rows x {s.H} heads ({spent:.2f} s, {flops / 1e9:.3f} GFLOP), f64, one "
                       f"thread" + ("" if full else "; measured on sample")),
            "measured_on_sample": not full,
            "extrapolated_full_s": full_flops / (rate * 1e12) + t_append,
            "host_cores_available": _host_cores()}


def _spread_rows(n, k, seed):
    """k rows spread evenly over [0, n) followed by seeded random ones."""
    import numpy as np
    even = np.linspace(0, n - 1, k).astype(int).tolist()
    rnd = np.random.default_rng(seed).integers(0, n, size=4 * k).tolist()
    seen, out = set(), []
    for r in even + rnd:
        if r not in seen:
            seen.add(r)
            out.append(int(r))
    return out


def cpu_baseline_chunked(wl: W.PrefillWorkload, budget_s: float):
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from harness import prompt_as_step
    prompt = W.make_chunked_prompt(wl, seed=0)
    step = prompt_as_step(prompt)
    full = causal_flops(wl.spec.H, wl.spec.d, 0, wl.prompt_len)
    L = wl.prompt_len
    rows = list(range(L)) if L <= 256 else _spread_rows(L, 64, seed=1)
    return cpu_baseline_rows(step, rows, budget_s, full, wl.name)


def cpu_baseline_varlen(wl: W.PrefillWorkload, budget_s: float):
    step = W.make_varlen_step(wl, seed=0)
    new = (step.cu_seqlens[1:] - step.cu_seqlens[:-1]).tolist()
    full = sum(causal_flops(wl.spec.H, wl.spec.d, int(p), int(n))
               for p, n in zip(step.cache_lens.tolist(), new))
    rows = _spread_rows(step.total_tokens, 64, seed=2)
    return cpu_baseline_rows(step, rows, budget_s, full, wl.name)


def cpu_baseline_decode(wl: W.DecodeWorkload, budget_s: float):
    """The oracle's decode (output and per-key probabilities of every head) on
    seeded sequences of the decode workload, one at a time until the budget is
    spent; GB/s of those sequences' algorithmic bytes."""
    import numpy as np
    o, h = _oracle_tools()
    s = wl.spec
    dec = W.make_decode_workload(wl, seed=0)
    lens = dec.kv_lens.tolist()
    order = np.random.default_rng(3).permutation(len(lens)).tolist()
    spent, nbytes, done = 0.0, 0.0, 0
    for b in order:
        if spent >= budget_s:
            break
        n = lens[b]
        ck = np.ascontiguousarray(W.bf16_to_f64(dec.cache_k[b:b + 1, :, :n]))
        cv = np.ascontiguousarray(W.bf16_to_f64(dec.cache_v[b:b + 1, :, :n]))
        q = W.bf16_to_f64(dec.q[b:b + 1])
        t0 = time.perf_counter()
        o.decode(s.H, s.KV, s.d, h.score_scale(s), h.oracle_flags(s), q, ck, cv, [n],
                 probs_stride=n)
        spent += time.perf_counter() - t0
        nbytes += n * s.KV * s.d * 2 * 2 + n * s.H * 4 + 2 * s.H * s.d * 2
        done += 1
    rate = nbytes / spent / 1e9
    full_bytes = sum(lens) * (s.KV * s.d * 4 + s.H * 4) + wl.batch * 2 * s.H * s.d * 2
    return {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": (f"{wl.name}: decode with probabilities of {done} of {wl.batch} seeded "
                       f"sequences ({spent:.2f} s, {nbytes / 1e6:.1f} MB of algorithmic bytes), "
                       f"f64, one thread" + ("" if done == wl.batch else "; measured on sample")),
            "measured_on_sample": done < wl.batch,
            "extrapolated_full_s": full_bytes / (rate * 1e9),
            "host_cores_available": _host_cores()}


# ------------------------------------------------------------------ main --

def base_line(args, wl):
    return {"metric": "prefill attn TFLOP/s", "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 inputs of the workload's shapes)",
            "config": {"workload": wl.name, "description": wl.description,
                       "heads": wl.spec.H, "kv_heads": wl.spec.KV, "head_dim": wl.spec.d,
                       "rotary_dim": wl.spec.rd, "prompt_len": wl.prompt_len,
                       "chunk": wl.chunk, "parallelism": f"replicas{args.gpus}",
                       "l2": "flushed before every timed step: 256 MiB written, then 256 MiB read",
                       "launch": f"CUDA graph of the {wl.prompt_len // wl.chunk} chunk call "
                                 "pairs (append, attend)",
                       "statistic": "median of the timed steps (min and max in ms_spread)"}}


def reference_arm(args, wl):
    """The f64 CPU oracle on a bounded sample of the headline workload, one
    sample per step; ms_per_step is extrapolated to the full workload."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from harness import oracle_append, oracle_rows, prompt_as_step
    import oracle
    o = oracle.load()
    prompt = W.make_chunked_prompt(wl, seed=0)
    step = prompt_as_step(prompt)
    ost = oracle_append(o, step)
    s = wl.spec
    rows = _spread_rows(wl.prompt_len, 256, seed=4)
    budget = max(1.0, min(10.0, args.cpu_budget / max(1, args.steps + args.warmup)))
    vals, walls, nrows, ri = [], [], 0, 0
    for i in range(args.warmup + args.steps):
        spent, flops, w0 = 0.0, 0.0, time.perf_counter()
        while spent < budget:
            r = rows[ri % len(rows)]
            ri += 1
            t0 = time.perf_counter()
            oracle_rows(o, step, ost, [r])
            spent += time.perf_counter() - t0
            flops += 4.0 * s.d * s.H * (r + 1)
            if i >= args.warmup:
                nrows += 1
        if i >= args.warmup:
            vals.append(flops / spent / 1e12)
            walls.append((time.perf_counter() - w0) * 1e3)
    v = statistics.median(vals)
    full = causal_flops(s.H, s.d, 0, wl.prompt_len)
    line = dict(base_line(args, wl), impl="reference", value=v,
                ms_per_step=full / (v * 1e12) * 1e3,
                ms_per_step_basis=("extrapolated: the full workload's algorithmic flops over the "
                                   "measured oracle rate (each step times a bounded sample)"),
                sample_wall_ms_per_step=spread(walls))
    cb = {"value": v, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
          "sample": (f"per step {budget:.1f} s of causal attention rows (all {s.H} heads) of "
                     f"the {wl.prompt_len}-token prompt, rows spread over the prompt, after the "
                     f"RoPE+append of the whole prompt; {nrows} rows timed in total; f64, one "
                     f"thread; measured on sample"),
          "measured_on_sample": True, "host_cores_available": _host_cores()}
    line["cpu_baseline"] = cb
    line["e2e"] = {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    line["config"] = dict(line["config"], launch="CPU oracle, single thread")
    line["dtype"] = "f64"  # the oracle's arithmetic (bf16 inputs widened exactly)
    return line


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_setup(args)
    wl = W.C4  # headline: the largest single-GPU configuration

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(reference_arm(args, wl)))
        return

    torch.cuda.set_device(local)
    import causal_gqa_attention_rope_gb300 as na
    na.load_library()
    peaks = load_peaks()
    flush = Flusher()
    S, Wm = args.steps, args.warmup
    if args.only:
        fn = {"c1": lambda: bench_chunked(W.C1, S, Wm, peaks, flush),
              "chunked": lambda: bench_chunked(W.C2, S, Wm, peaks, flush),
              "decode": lambda: bench_decode(W.C3, S, Wm, peaks, flush),
              "pair": lambda: bench_pair_verify(S, Wm, peaks, flush),
              "varlen": lambda: bench_varlen(W.C5, S, Wm, peaks, flush),
              "yarn": lambda: bench_chunked(W.C4, S, Wm, peaks, flush)}
        rec = fn[args.only]()
        if rank == 0:
            print(json.dumps(dict(rec, only=args.only)))
        return
    sampler = ClockSampler()
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    r = bench_chunked(wl, S, Wm, peaks, flush, with_e2e=True)
    extra = []
    if not args.no_extra:
        extra.append(bench_chunked(W.C1, S, Wm, peaks, flush))
        extra.append(bench_chunked(W.C2, S, Wm, peaks, flush))
        dec_rec = bench_decode(W.C3, S, Wm, peaks, flush)
        extra.append({k: v for k, v in dec_rec.items() if k != "importance"})
        extra.append(dec_rec["importance"])
        extra.append(bench_pair_verify(S, Wm, peaks, flush))
        extra.append(bench_varlen(W.C5, S, Wm, peaks, flush))
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()

    ms = max_over_ranks(r["ms_per_step"], world)
    value = r["flops_per_step"] * world / (ms * 1e-3) / 1e12
    e2e_ms = max_over_ranks(r["e2e"]["ms_per_step"], world)
    line = dict(base_line(args, wl), value=value, ms_per_step=ms, ms_spread=r["ms_spread"])
    line["e2e"] = dict(r["e2e"], value=r["flops_per_step"] * world / (e2e_ms * 1e-3) / 1e12,
                       ms_per_step=e2e_ms)
    eager_ms = max_over_ranks(r["eager"]["ms_per_step"], world)
    line["eager"] = dict(r["eager"], value=r["flops_per_step"] * world / (eager_ms * 1e-3) / 1e12,
                         ms_per_step=eager_ms)
    line["gpu_launches"] = r["launches_per_step"] * args.steps
    line["roofline"] = r["roofline"]
    line["attn_calls_ms"] = r["attn_calls_ms"]
    line["clocks"] = clocks
    line["workloads"] = extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b = args.cpu_budget
        line["cpu_baseline"] = cpu_baseline_chunked(wl, 0.3 * b)
        per = {W.C1.name: lambda: cpu_baseline_chunked(W.C1, 0.1 * b),
               W.C2.name: lambda: cpu_baseline_chunked(W.C2, 0.2 * b),
               W.C3.name: lambda: cpu_baseline_decode(W.C3, 0.2 * b),
               W.C5.name: lambda: cpu_baseline_varlen(W.C5, 0.2 * b)}
        for rec in extra:
            if rec["workload"] in per:
                rec["cpu_baseline"] = per[rec["workload"]]()
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()

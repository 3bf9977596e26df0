"""The calls as a serving loop uses them: under CUDA graph capture -- captured
once, then replayed with new values in the same buffers (new queries, new
lengths, new positions within the bounds given at capture), where nothing but
pointers, host bounds and the plan derived from them may be baked into the
graph -- and on several streams at once.  Every run must equal the eager,
one-at-a-time calls on the same inputs bit for bit (every kernel here is
deterministic: fixed summation orders, no atomics)."""
import pytest
import torch

import workloads as W
from harness import attn_cfg, rope_cfg

pytestmark = pytest.mark.gpu


def _capture(fn):
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _bits(t):
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def test_decode_and_importance_replayed_with_new_lengths():
    """Decode (with probabilities) + accumulated importance captured with
    max_kv_len 3000; replayed after the lengths grow, shrink and hit zero and
    the queries change: each replay equals the eager calls."""
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=16, KV=4, d=128, rd=128, out_gate=True)
    B, cap, mx = 5, 3072, 3000
    dec = W.make_decode(spec, [3000] * B, cap, seed=201)
    dev = "cuda"
    cfg = attn_cfg(spec)
    cache = na.KVCache(dec.cache_k.to(dev), dec.cache_v.to(dev))
    q = torch.empty_like(dec.q, device=dev)
    gate = dec.gate.to(dev)
    kv = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    probs = torch.full((B, spec.H, mx), -7.0, device=dev)
    imp = torch.zeros(B, mx, device=dev)
    ws = na.workspace(na.na_decode_workspace_size(cfg, B, mx), dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        na.na_attn_decode(cfg, q, cache, kv, mx, out, probs=probs, gate=gate, workspace=ws,
                          status=st)
        na.na_decode_importance(cfg, probs, kv, mx, imp, accumulate=True, status=st)

    gen = torch.Generator().manual_seed(7)
    q.copy_(dec.q)
    kv.copy_(torch.tensor([3000, 1, 64, 700, 0], dtype=torch.int32))
    g = _capture(step)
    for lens in ([3000, 1, 64, 700, 0], [2999, 2, 65, 701, 1], [5, 0, 1500, 3000, 63]):
        newq = torch.randn(dec.q.shape, generator=gen).to(torch.bfloat16)
        results = []
        for run in ("graph", "eager"):
            q.copy_(newq)
            kv.copy_(torch.tensor(lens, dtype=torch.int32))
            probs.fill_(-7.0)
            imp.fill_(0.25)
            if run == "graph":
                g.replay()
            else:
                step()
            torch.cuda.synchronize()
            results.append((out.clone(), probs.clone(), imp.clone()))
        assert int(st.item()) == 0
        assert bool(torch.isfinite(results[0][0].float()).all())
        for a, b, what in zip(results[0], results[1], ("out", "probs", "importance")):
            assert torch.equal(_bits(a), _bits(b)), f"{what} differs from eager with lengths {lens}"


def test_chunked_prefill_replayed_at_new_positions():
    """Append + attend of a 96-token chunk of two sequences (the attention's
    cut units and merge pass included) captured with max_total_len 1024;
    replayed with other prior lengths and new token values: outputs, rotated
    queries and the cache equal the eager calls."""
    import causal_gqa_attention_rope_gb300 as na
    spec = W.Spec(H=8, KV=2, d=128, rd=128, qk_norm=True, out_gate=True,
                  rope=W.RopeParams(base=5e5))
    new = [64, 32]
    cap, max_total = 1024, 1024
    base = W.make_step(spec, [900, 700], new, cap, seed=203)
    dev = "cuda"
    cfg, rope = attn_cfg(spec), rope_cfg(spec)
    T = base.total_tokens
    cu = base.cu_seqlens.to(dev)
    lens = torch.empty(2, dtype=torch.int32, device=dev)
    q, k, v = (torch.empty_like(x, device=dev) for x in (base.q, base.k, base.v))
    gate = base.gate.to(dev)
    qw, kw = base.q_norm_w.to(dev), base.k_norm_w.to(dev)
    # every slot holds a real key and value, so any prior length attends data
    cg = torch.Generator().manual_seed(205)
    ck = torch.randn(base.cache_k.shape, generator=cg).to(torch.bfloat16).to(dev)
    cv = torch.randn(base.cache_v.shape, generator=cg).to(torch.bfloat16).to(dev)
    cache = na.KVCache(ck.clone(), cv.clone())
    q_out, out = torch.empty_like(q), torch.empty_like(q)
    ws = na.workspace(na.na_prefill_workspace_size(cfg, 2, T, max(new), max_total), dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        na.na_rope_append_kv(cfg, rope, cu, lens, q, k, v, q_out, cache, q_norm_w=qw,
                             k_norm_w=kw, status=st)
        na.na_attn_prefill_chunk(cfg, cu, lens, max(new), max_total, q_out, cache, out,
                                 gate=gate, workspace=ws, status=st)

    gen = torch.Generator().manual_seed(9)
    for x, y in ((q, base.q), (k, base.k), (v, base.v)):
        x.copy_(y)
    lens.copy_(torch.tensor([900, 700], dtype=torch.int32))
    g = _capture(step)
    for prior in ([900, 700], [960, 0], [100, 992], [0, 5]):
        vals = [torch.randn(x.shape, generator=gen).to(torch.bfloat16) for x in (base.q, base.k, base.v)]
        results = []
        for run in ("graph", "eager"):
            for x, y in zip((q, k, v), vals):
                x.copy_(y)
            lens.copy_(torch.tensor(prior, dtype=torch.int32))
            cache.k.copy_(ck)
            cache.v.copy_(cv)
            if run == "graph":
                g.replay()
            else:
                step()
            torch.cuda.synchronize()
            results.append((out.clone(), q_out.clone(), cache.k.clone(), cache.v.clone()))
        assert int(st.item()) == 0
        assert bool(torch.isfinite(results[0][0].float()).all())
        for a, b, what in zip(results[0], results[1], ("out", "q_out", "cache K", "cache V")):
            assert torch.equal(_bits(a), _bits(b)), f"{what} differs from eager with priors {prior}"


def test_calls_on_two_streams_at_once():
    """A decode on one stream and an append + attend on another, launched
    without waiting for each other (each with its own workspace and status):
    both equal the same calls run one after the other -- no device state is
    shared between calls."""
    import causal_gqa_attention_rope_gb300 as na
    dev = "cuda"
    # decode
    dspec = W.Spec(H=32, KV=8, d=128, rd=128)
    dec = W.make_decode(dspec, [4000, 17, 2500, 900], 4096, seed=211)
    dcfg = attn_cfg(dspec)
    dq, dkv = dec.q.to(dev), dec.kv_lens.to(dev)
    dcache = na.KVCache(dec.cache_k.to(dev), dec.cache_v.to(dev))
    dout = torch.empty_like(dq)
    dprobs = torch.zeros(4, dspec.H, 4000, device=dev)
    dws = na.workspace(na.na_decode_workspace_size(dcfg, 4, 4000), dev)
    dst = torch.zeros(1, dtype=torch.int32, device=dev)
    # prefill
    pspec = W.Spec(H=8, KV=2, d=64, rd=64, out_gate=True)
    step = W.make_step(pspec, [600, 40], [150, 70], 1024, seed=213)
    pcfg, prope = attn_cfg(pspec), rope_cfg(pspec)
    cu, lens = step.cu_seqlens.to(dev), step.cache_lens.to(dev)
    q, k, v, gate = (x.to(dev) for x in (step.q, step.k, step.v, step.gate))
    ck0, cv0 = step.cache_k.to(dev), step.cache_v.to(dev)
    pcache = na.KVCache(ck0.clone(), cv0.clone())
    q_out, pout = torch.empty_like(q), torch.empty_like(q)
    T = step.total_tokens
    pws = na.workspace(na.na_prefill_workspace_size(pcfg, 2, T, 150, 750), dev)
    pst = torch.zeros(1, dtype=torch.int32, device=dev)

    def decode():
        na.na_attn_decode(dcfg, dq, dcache, dkv, 4000, dout, probs=dprobs, workspace=dws,
                          status=dst)

    def prefill():
        na.na_rope_append_kv(pcfg, prope, cu, lens, q, k, v, q_out, pcache, status=pst)
        na.na_attn_prefill_chunk(pcfg, cu, lens, 150, 750, q_out, pcache, pout, gate=gate,
                                 workspace=pws, status=pst)

    def snapshot():
        torch.cuda.synchronize()
        return [t.clone() for t in (dout, dprobs, pout, q_out, pcache.k, pcache.v)]

    decode()
    prefill()
    ref = snapshot()
    for _ in range(3):
        dout.zero_()
        dprobs.zero_()
        pout.zero_()
        pcache.k.copy_(ck0)
        pcache.v.copy_(cv0)
        torch.cuda.synchronize()
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        with torch.cuda.stream(s1):
            decode()
        with torch.cuda.stream(s2):
            prefill()
        got = snapshot()
        assert int(dst.item()) == 0 and int(pst.item()) == 0
        for a, b in zip(got, ref):
            assert torch.equal(_bits(a), _bits(b))


def test_calls_from_several_host_threads():
    """Four host threads, each with its own stream, workspace and buffers, call
    the decode (two threads) and append + attend (two threads) ten times each
    at once (the binding releases the interpreter lock inside the library):
    every result equals the same call made alone."""
    import threading

    import causal_gqa_attention_rope_gb300 as na
    dev = "cuda"

    def make_decode_job(seed):
        spec = W.Spec(H=16, KV=4, d=128, rd=128)
        dec = W.make_decode(spec, [1500, 3, 777], 1536, seed=seed)
        cfg = attn_cfg(spec)
        q, kv = dec.q.to(dev), dec.kv_lens.to(dev)
        cache = na.KVCache(dec.cache_k.to(dev), dec.cache_v.to(dev))
        out = torch.empty_like(q)
        probs = torch.zeros(3, spec.H, 1500, device=dev)
        ws = na.workspace(na.na_decode_workspace_size(cfg, 3, 1500), dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)

        def run():
            na.na_attn_decode(cfg, q, cache, kv, 1500, out, probs=probs, workspace=ws, status=st)
            return [out, probs]
        return run, st

    def make_prefill_job(seed):
        spec = W.Spec(H=8, KV=2, d=64, rd=64, qk_norm=True)
        step = W.make_step(spec, [300, 0], [90, 40], 512, seed=seed)
        cfg, rope = attn_cfg(spec), rope_cfg(spec)
        cu, lens = step.cu_seqlens.to(dev), step.cache_lens.to(dev)
        q, k, v = (x.to(dev) for x in (step.q, step.k, step.v))
        qw, kw = step.q_norm_w.to(dev), step.k_norm_w.to(dev)
        ck0, cv0 = step.cache_k.to(dev), step.cache_v.to(dev)
        cache = na.KVCache(ck0.clone(), cv0.clone())
        q_out, out = torch.empty_like(q), torch.empty_like(q)
        ws = na.workspace(na.na_prefill_workspace_size(cfg, 2, step.total_tokens, 90, 390), dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)

        def run():
            cache.k.copy_(ck0)
            cache.v.copy_(cv0)
            na.na_rope_append_kv(cfg, rope, cu, lens, q, k, v, q_out, cache, q_norm_w=qw,
                                 k_norm_w=kw, status=st)
            na.na_attn_prefill_chunk(cfg, cu, lens, 90, 390, q_out, cache, out, workspace=ws,
                                     status=st)
            return [out, q_out, cache.k, cache.v]
        return run, st

    jobs = [make_decode_job(301), make_decode_job(302), make_prefill_job(303),
            make_prefill_job(304)]
    refs = []
    for run, _ in jobs:
        refs.append([t.clone() for t in run()])
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        run, _ = jobs[i]
        s = torch.cuda.Stream()
        try:
            with torch.cuda.stream(s):
                for _ in range(10):
                    got = run()
                    s.synchronize()
                    for a, b in zip(got, refs[i]):
                        if not torch.equal(_bits(a), _bits(b)):
                            errors.append(f"job {i} differs")
                            return
        except Exception as e:  # reported below
            errors.append(f"job {i}: {e}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for _, st in jobs:
        assert int(st.item()) == 0


def test_first_call_of_a_thread_inside_graph_capture():
    """A host thread whose very first library call is made while a CUDA graph
    is being captured (a serving thread that captures its step at once): the
    capture succeeds and its replay equals an eager call."""
    import threading

    import causal_gqa_attention_rope_gb300 as na
    dev = "cuda"
    spec = W.Spec(H=16, KV=4, d=128, rd=128)
    dec = W.make_decode(spec, [900, 31], 1024, seed=311)
    cfg = attn_cfg(spec)
    q, kv = dec.q.to(dev), dec.kv_lens.to(dev)
    cache = na.KVCache(dec.cache_k.to(dev), dec.cache_v.to(dev))
    out = torch.empty_like(q)
    probs = torch.zeros(2, spec.H, 900, device=dev)
    ws = na.workspace(na.na_decode_workspace_size(cfg, 2, 900), dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def call():
        na.na_attn_decode(cfg, q, cache, kv, 900, out, probs=probs, workspace=ws, status=st)

    result = {}

    def worker():
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call()
            g.replay()
            torch.cuda.synchronize()
            result["graph"] = (out.clone(), probs.clone())
        except Exception as e:  # reported below
            result["error"] = repr(e)

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert "error" not in result, result.get("error")
    out.zero_()
    probs.zero_()
    call()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(_bits(result["graph"][0]), _bits(out))
    assert torch.equal(_bits(result["graph"][1]), _bits(probs))


@pytest.mark.parametrize("first", ["prefill", "importance"])
def test_first_call_of_a_thread(first):
    """A fresh host thread whose first library call is the attention call (no
    append before it on that thread) or the importance pass: both encode
    tensor maps before they launch, and must bind the device's context first.
    The results equal the same call made on the main thread."""
    import threading

    import causal_gqa_attention_rope_gb300 as na
    dev = "cuda"
    if first == "prefill":
        spec = W.Spec(H=8, KV=2, d=128, rd=128)
        step = W.make_step(spec, [200, 0], [64, 30], 512, seed=321)
        cfg, rope = attn_cfg(spec), rope_cfg(spec)
        cu, lens = step.cu_seqlens.to(dev), step.cache_lens.to(dev)
        cache = na.KVCache(step.cache_k.to(dev), step.cache_v.to(dev))
        q_rot = torch.empty_like(step.q, device=dev)
        na.na_rope_append_kv(cfg, rope, cu, lens, step.q.to(dev), step.k.to(dev),
                             step.v.to(dev), q_rot, cache)
        out = torch.empty_like(q_rot)
        ws = na.workspace(na.na_prefill_workspace_size(cfg, 2, step.total_tokens, 64, 264), dev)

        def call():
            na.na_attn_prefill_chunk(cfg, cu, lens, 64, 264, q_rot, cache, out, workspace=ws)
            return out
    else:
        cfg = attn_cfg(W.Spec(H=16, KV=4, d=128, rd=128))
        gen = torch.Generator().manual_seed(323)
        probs = torch.rand((3, 16, 2048), generator=gen).to(dev)
        kv = torch.tensor([2048, 5, 1000], dtype=torch.int32, device=dev)
        imp = torch.zeros(3, 2048, device=dev)

        def call():  # overwrites imp (no accumulation): no torch op before it
            na.na_decode_importance(cfg, probs, kv, 2048, imp)
            return imp
    torch.cuda.synchronize()
    result = {}

    def worker():
        try:
            result["got"] = call().clone()
            torch.cuda.synchronize()
        except Exception as e:  # reported below
            result["error"] = repr(e)

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert "error" not in result, result.get("error")
    ref = call().clone()
    torch.cuda.synchronize()
    assert torch.equal(_bits(result["got"]), _bits(ref))

"""The seeded input generators follow the stated recipe: deterministic per
seed, lengths inside the stated closed ranges, unused cache slots holding the
sentinel, the stated distributions, and workload names that match their
shapes.  CPU only; shapes are kept small where the full ones are large."""
import re

import torch

import workloads as W


def test_same_seed_same_inputs_other_seed_differs():
    spec = W.Spec(H=4, KV=2, d=64, rd=64, qk_norm=True, out_gate=True, norm_w_mean=1.0,
                  norm_w_std=0.1)
    a = W.make_step(spec, [5, 0], [3, 7], 32, seed=11)
    b = W.make_step(spec, [5, 0], [3, 7], 32, seed=11)
    c = W.make_step(spec, [5, 0], [3, 7], 32, seed=12)
    for name in ("q", "k", "v", "gate", "q_norm_w", "k_norm_w", "cache_k", "cache_v"):
        x, y, z = getattr(a, name), getattr(b, name), getattr(c, name)
        assert torch.equal(x.view(torch.int16), y.view(torch.int16)), name
        assert not torch.equal(x.view(torch.int16), z.view(torch.int16)), name


def test_step_layout_and_sentinel_slots():
    spec = W.Spec(H=4, KV=2, d=64, rd=64)
    st = W.make_step(spec, [5, 0, 9], [3, 7, 1], 16, seed=1)
    assert st.cu_seqlens.tolist() == [0, 3, 10, 11] and st.total_tokens == 11
    assert st.q.shape == (11, 4, 64) and st.k.shape == (11, 2, 64)
    bits = st.cache_k.view(torch.int16)
    for b, n in enumerate([5, 0, 9]):
        assert bool((bits[b, :, n:] == W.SENTINEL_BITS).all()), "unused slots hold the sentinel"
        if n:
            assert not bool((bits[b, :, :n] == W.SENTINEL_BITS).any()), "history is drawn"


def test_varlen_lengths_in_stated_ranges():
    w = W.C5
    for seed in range(5):
        st = W.make_varlen_step(w, seed=seed, history=False)
        prior = st.cache_lens.tolist()
        new = (st.cu_seqlens[1:] - st.cu_seqlens[:-1]).tolist()
        assert len(prior) == w.batch
        assert all(w.prior_range[0] <= p <= w.prior_range[1] for p in prior)
        assert all(w.new_range[0] <= n <= w.new_range[1] for n in new)
        assert all(p + n <= w.capacity for p, n in zip(prior, new))


def test_decode_lengths_in_stated_range():
    w = W.C3
    gen = torch.Generator().manual_seed(0)
    lens = W.draw_lengths(gen, 10000, *w.kv_range)
    assert min(lens) >= w.kv_range[0] and max(lens) <= w.kv_range[1]
    assert min(lens) < w.kv_range[0] + 20 and max(lens) > w.kv_range[1] - 20  # both ends reached
    small = W.make_decode(W.Spec(H=4, KV=2, d=64, rd=64), [0, 3, 16], 16, seed=2)
    assert small.kv_lens.tolist() == [0, 3, 16]
    assert bool((small.cache_v.view(torch.int16)[0] == W.SENTINEL_BITS).all())


def test_chunked_prompt_chunks_cover_the_prompt_and_scale():
    w = W.C2
    p = W.make_chunked_prompt(w, seed=0)
    assert p.num_chunks == w.prompt_len // w.chunk
    covered = []
    for c in range(p.num_chunks):
        lo, hi = p.chunk_bounds(c)
        covered.extend(range(lo, hi))
    assert covered == list(range(w.prompt_len))
    std = float(p.q.float().std())
    assert abs(std - w.spec.std) < 0.01, std  # Q ~ 0.5 N(0, 1)


def test_norm_weights_and_gate_distributions():
    spec = W.C5.spec
    st = W.make_step(spec, [0], [512], 512, seed=3)
    w = torch.cat([st.q_norm_w.float(), st.k_norm_w.float()])
    assert abs(float(w.mean()) - 1.0) < 0.03 and abs(float(w.std()) - 0.1) < 0.03
    g = st.gate.float()
    assert abs(float(g.mean())) < 0.01 and abs(float(g.std()) - 1.0) < 0.01


def test_workload_names_match_their_shapes():
    for w in W.WORKLOADS.values():
        s = w.spec
        m = re.search(r"h(\d+)kv(\d+)d(\d+)", w.name)
        assert m and (int(m[1]), int(m[2]), int(m[3])) == (s.H, s.KV, s.d), w.name
        rd = re.search(r"_rd(\d+)", w.name)
        assert (int(rd[1]) if rd else s.d) == s.rd, w.name

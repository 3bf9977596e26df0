"""The README's example runs as written (on the GPU): no device error, a
finite decode output, probabilities over the 129 keys summing to 1 and the
running importance untouched past them."""
import os
import re

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "README has no python example"
    scope = {}
    exec(compile(blocks[0], "README example", "exec"), scope)
    import torch
    probs, kv_lens = scope["probs"], scope["kv_lens"]
    n = int(kv_lens[0])
    mass = probs[0, :, :n].double().sum(-1)
    assert torch.allclose(mass, torch.ones_like(mass), atol=1e-4)
    assert bool(torch.isfinite(scope["out1"].float()).all())
    assert bool((scope["imp"][0, n:] == 0).all())

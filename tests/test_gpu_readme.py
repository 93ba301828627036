"""The README's usage example runs as written on the GPU, and its stitch
matches the oracle on a sampled layer."""

import os
import re

import numpy as np
import pytest

import oracle
from gpu_util import bits

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example():
    text = open(os.path.join(ROOT, "README.md")).read()
    use = text.split("## Use", 1)[1]
    return re.search(r"```python\n(.*?)```", use, re.S).group(1)


def test_readme_example_runs_and_matches_the_oracle():
    scope = {}
    exec(compile(_example(), "README.md", "exec"), scope)
    torch, ridx, out = scope["torch"], scope["ridx"], scope["out"]
    torch.cuda.synchronize()
    # the recompute list: 4 positions at each of the three chunks (none is at position 0)
    starts = [128, 128 + 2048, 128 + 2048 + 1024]
    assert ridx.cpu().tolist() == [s + t for s in starts for t in range(4)]
    assert torch.isfinite(out).all()
    # layer 5 of the stitched keys against the oracle's rotation of the pool rows
    L, H, D, BS = scope["L"], scope["H"], scope["D"], scope["BS"]
    theta = oracle.model_inv_freq(D, 5e5, None)
    k_pool, k_cache, table = scope["k_pool"], scope["k_cache"], scope["table"]
    kp = oracle.bf16_bits_to_f64(bits(k_pool[5]))
    kc = oracle.bf16_bits_to_f64(bits(k_cache[5]))
    for c, (off, n), dst in ((2, (1536, 2048), 128), (0, (0, 1024), 2176), (1, (1024, 512), 3200)):
        want = oracle.rotate(kp[off:off + n], dst, theta, oracle.NEOX_HALF)
        pos = np.arange(dst, dst + n)
        got = kc[np.asarray(table)[pos // BS], pos % BS]
        assert np.all(np.abs(got - want) <= 2.0 ** -7 * np.abs(want) + 1e-3), c

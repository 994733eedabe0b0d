"""The README's usage example, run as written: it must work and give
attention over its 100 appended tokens (GQA: query head h reads KV head
h // 4), checked against the definition in float64."""

import os
import re

import numpy as np
import pytest

from harness import TOL, assert_close

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example(pa, cuda):
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    ns = {}
    exec(compile(code, "README.md", "exec"), ns)
    q = ns["q"].float().cpu().numpy().astype(np.float64)[0]     # [32, 128]
    k = ns["k"].float().cpu().numpy().astype(np.float64)        # [100, 8, 128], also the values
    want = np.zeros_like(q)
    for h in range(32):
        s = k[:, h // 4] @ q[h] * 128 ** -0.5
        w = np.exp(s - s.max())
        want[h] = w @ k[:, h // 4] / w.sum()
    assert_close(ns["out"].cpu().numpy()[0], want, TOL["bf16"], "README example")

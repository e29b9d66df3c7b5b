"""The Python usage example in README.md runs as written, and its allreduce
matches the oracle."""
import os
import re

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs_and_matches_oracle():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert len(blocks) == 1
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    ins = [x.cpu().numpy().view(np.uint16) for x in scope["ins"]]
    outs = [x.cpu().numpy().view(np.uint16) for x in scope["outs"]]
    want = oracle.allreduce(ins, "fp16")[0]
    for o in outs:
        assert np.array_equal(o, want)

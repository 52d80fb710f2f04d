"""The Python quick start in README.md runs as written: its block is executed verbatim on the
GPU, and the products it computes have the shapes the example states."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _quick_start() -> str:
    text = open(os.path.join(ROOT, "README.md"), encoding="utf-8").read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "README.md has no python block"
    return blocks[0]


def test_readme_quick_start_runs():
    import __graft_entry__
    __graft_entry__.build()
    scope = {}
    exec(compile(_quick_start(), "README.md", "exec"), scope)
    torch.cuda.synchronize()
    Y, dX, dW = scope["Y"], scope["dX"], scope["dW"]
    X, W, dY = scope["X"], scope["W"], scope["dY"]
    assert Y.shape == (X.shape[0], W.shape[0])
    assert dX.shape == X.shape
    assert dW.shape == W.shape
    for t in (Y, dX, dW):
        assert t.dtype == torch.bfloat16 and torch.isfinite(t.float()).all()

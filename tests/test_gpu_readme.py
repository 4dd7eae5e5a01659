"""The Python example in README.md runs as written and steps the parameters."""

import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "no python example in the README"
    env = {}
    exec(compile(blocks[0], "README.md example", "exec"), env)
    torch.cuda.synchronize()
    # zero gradients and zero weights: weight decay keeps zeros, so the step leaves every value 0,
    # and every rank's replica equals bf16 of the master weights
    assert all(torch.equal(r, env["replicas"][0]) for r in env["replicas"])
    assert torch.equal(env["replicas"][0].float(), env["master"])

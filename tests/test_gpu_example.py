"""The example step (tests/example_step.py, shown in the README) runs and steps the parameters."""

import pytest
import torch

import example_step

pytestmark = pytest.mark.gpu


def test_example_step_runs():
    env = example_step.run()
    torch.cuda.synchronize()
    # zero gradients and zero weights: weight decay keeps zeros, so the step leaves every value 0,
    # and every rank's replica equals bf16 of the master weights
    assert all(torch.equal(r, env["replicas"][0]) for r in env["replicas"])
    assert torch.equal(env["replicas"][0].float(), env["master"])

"""The Python example in README.md runs as written (its single-GPU part) and its stated
equality holds: step 1 from the tensor list gives the flat call's codes and scales."""
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1, "README.md holds one Python example"
    code = blocks[0]
    cut = code.index("# the same exchange across real ranks")  # needs torchrun
    return code[:cut]


@pytest.mark.gpu
def test_readme_example_runs():
    env = {}
    exec(compile(_example(), "README.md", "exec"), env)
    assert env["y"].dtype == torch.float16 and env["y"].numel() == env["x"].numel()
    assert env["avg"].shape == (env["N"] * env["M"], env["E"] // (env["N"] * env["M"]))
    assert torch.equal(env["t0"], env["c0"])
    assert torch.equal(env["ts0"].view(torch.int32), env["s0"].view(torch.int32))

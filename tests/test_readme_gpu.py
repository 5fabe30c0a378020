"""The README's usage example runs as written."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    text = open(os.path.join(ROOT, "README.md"), encoding="utf-8").read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert len(blocks) == 1
    env = {}
    exec(compile(blocks[0], "README.md", "exec"), env)
    rep = env["rep"]
    assert rep.t == 1 and rep.overflow == 0 and rep.current == 1
    env["graph"].replay()
    torch.cuda.synchronize()
    assert env["plan"].report().t == 3  # the step, the in-place step, the replay

"""The Python usage example in the repository's front-page documentation runs
as written: one gradient-sync step applied, not skipped."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_python_example_runs(capsys):
    from gradient_sync_rcc_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, re.S)
    assert blocks, "no python example found"
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    torch.cuda.synchronize()
    out = capsys.readouterr().out.split()
    assert len(out) == 4 and out[1] == "0" and out[2] == "1"   # not skipped, one step applied

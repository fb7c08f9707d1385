"""The README's Python example runs as written (on the GPU)."""
import os
import re

import pytest
import torch

from conftest import ROOT

pytestmark = pytest.mark.gpu


def test_readme_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    block = re.search(r"<!-- example -->\s*```python\n(.*?)```\s*<!-- /example -->", text, re.S)
    assert block, "README example block not found"
    exec(compile(block.group(1), "README example", "exec"), {})
    torch.cuda.synchronize()

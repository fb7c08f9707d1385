"""The package's usage example (tests/usage_example.py, printed in the user
documentation) runs as written on the GPU."""
import pytest
import torch

import usage_example

pytestmark = pytest.mark.gpu


def test_usage_example_runs():
    usage_example.run()
    torch.cuda.synchronize()

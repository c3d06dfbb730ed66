"""The quick start in README.md runs as written: every call it shows succeeds on the GPU,
returns the shapes it states and finite values, and the long-sequence call takes the
tensor-core pair kernel."""
import os
import re

import pytest
import torch

from linear_recurrence_sequence_chunkwise_b300 import binding as rb

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_quick_start_runs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1
    ns: dict = {}
    exec(compile(blocks[0], "README.md", "exec"), ns)
    torch.cuda.synchronize()
    b, H, N, dk, dv = ns["b"], ns["H"], ns["N"], ns["dk"], ns["dv"]
    assert ns["o"].shape == (b, H, N, dv) and ns["o"].dtype == torch.float32
    assert ns["y"].shape == (b, H, dv)
    assert ns["o_par"].shape == (b, H, 2048, dv)
    assert ns["dq"].shape == (b, H, N, dk) and ns["dv_"].shape == (b, H, N, dv)
    for name in ("o", "state", "y", "o_par", "dq", "dk_", "dv_"):
        assert torch.isfinite(ns[name]).all(), name
    rb.check_device_error()

"""The README's quick-start example runs as written and gives a sane step: clean
device status, finite outputs, refresh flags of 0 or 1, and top-k indices outside
the block."""
import os
import re

import pytest
import torch

from denoising_step_attention_qkv_b300 import capi

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def test_readme_quick_start_runs():
    text = open(README).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python block in the README"
    ns = {}
    exec(compile(blocks[0].replace("print(cache.status())", "status = cache.status()"), "README", "exec"), ns)
    torch.cuda.synchronize()
    assert ns["status"] == (capi.DLLM_OK, 0)
    assert torch.isfinite(ns["out"].float()).all()
    assert torch.isfinite(ns["cos"]).all() and (ns["cos"].abs() <= 1.0 + 1e-5).all()
    assert set(ns["refresh"].cpu().tolist()) <= {0, 1}
    idx = ns["idx"]
    assert ((idx < 512) | (idx >= 512 + ns["n"])).all() and (idx >= 0).all() and (idx < ns["S"]).all()

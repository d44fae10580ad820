"""fp64 CPU oracle for the cached-attention denoising step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path (``denoising_step_attention_qkv_b300``) and does not
import it.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against closed forms, invariants, brute force on
tiny inputs and one library routine (PyTorch's float8_e4m3fn cast for the FP8
code table).  No function is "parity unpinned".
"""
from .dllm_oracle import *  # noqa: F401,F403
from .dllm_oracle import __all__  # noqa: F401

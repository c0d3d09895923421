"""CPU oracle for the nanochat-style pretraining step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import anything under ``oracle/``.  The product path (the
CUDA library and its Python binding) never imports, links or calls it.

Every function is the plain fp64 definition of one step of the method; see
``nanochat_step.py`` (the forward + backward step) and ``optimizer.py`` (the
Muon + AdamW update that follows it) for the citations.  Parity is pinned by the ``not gpu``
tests in ``tests/test_oracle_*.py`` (closed forms, invariants, library special
cases, brute force and central differences; ``test_oracle_optimizer.py``:
closed-form AdamW steps, Newton-Schulz against an SVD-based scalar map).
"""
from .nanochat_step import (  # noqa: F401
    attention,
    attention_bwd,
    backward,
    cross_entropy,
    evaluate,
    forward,
    rmsnorm,
    rmsnorm_bwd,
    rope,
    rope_bwd,
    rope_tables,
    softcap,
    softcap_bwd,
    step,
)

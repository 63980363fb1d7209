"""CPU fp64 oracle for the tensor-parallel MLP path and the hidden-split LayerNorm.
TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and
``--impl reference``) may import this package. The library under
``tensor_sharded_linear_bias_gb300/`` never imports it, and this package imports nothing
from there.
"""
from .tp_mlp import *  # noqa: F401,F403
from .tp_layernorm import *  # noqa: F401,F403

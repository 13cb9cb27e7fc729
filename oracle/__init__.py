"""CPU oracle for the DeepSeekMoE layer with auxiliary-loss-free routing.

TEST INFRASTRUCTURE ONLY: ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` may import it; the CUDA library and its binding never do.  It shares no
code with them.  See ``moe_oracle`` for the definitions and the readings taken, and
``moe_backward`` for the gradients through the layer (bf16 and FP8 expert GEMMs).
"""
from . import fp8  # noqa: F401
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import __all__  # noqa: F401
from . import moe_backward  # noqa: F401

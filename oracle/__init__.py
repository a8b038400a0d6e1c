"""CPU oracle (test infrastructure only): the plain fp64 statement of the routed
MoE expert-MLP layer and its router step that the CUDA library is checked against.
Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
use it."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import silu_grad  # noqa: F401
from .router_oracle import *  # noqa: F401,F403

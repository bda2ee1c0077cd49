"""CPU oracle for the Switch top-1 MoE layer forward (test infrastructure).

This package is test infrastructure, not product code.  Only the tests, the
package's ``__graft_entry__.smoke()`` check and ``bench.py``'s CPU-baseline
leg may import it.  It shares no code with the CUDA library and imports
nothing from it.
"""
from .switch_moe_oracle import *  # noqa: F401,F403
from .switch_moe_oracle import __all__  # noqa: F401

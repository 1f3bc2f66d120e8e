"""CPU oracle for the single-GPU dropless MoE layer (test infrastructure only).

This package is the plain, slow, obviously-correct restatement of what the
layer computes.  It exists to check the CUDA library; it is not part of the
product.  Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference arm of ``bench.py`` may import it.  It shares no
code with the CUDA path and imports nothing from the ``ragged_grouped_gemm_gb300``
package.
"""
from .moe_oracle import *  # noqa: F401,F403
from .mxfp8 import *  # noqa: F401,F403

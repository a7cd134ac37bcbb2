"""Float64 CPU oracle for GPTQ layer quantization (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  It shares no code with the CUDA library.
"""

from . import gptq_oracle
from .gptq_oracle import *  # noqa: F401,F403

__all__ = list(gptq_oracle.__all__)

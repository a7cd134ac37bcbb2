"""GPTQ layer quantization on one NVIDIA GB300 (sm_103a).

The computation lives in ``libgptq_gb300.so`` (hand-written CUDA, C ABI in
``include/gptq.h``); ``gptq`` is its thin ctypes binding and ``api`` the Python-level
engine built on it.  Importing the package does not load the library; the first call
does, and fails loudly if it cannot.
"""

from .api import LayerEngine, QuantizedLayer, quantize_layer_from_host  # noqa: F401
from .shard import ShardedLayer, row_range, row_ranges, token_range  # noqa: F401

"""CPU oracle for INT8-QK attention. TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import anything here. The CUDA
library never calls, links or falls back to this code, and this code shares
nothing with it: no kernels, headers, tables or helpers.

See ``oracle/ia_oracle.py`` for the functions and the passages they follow.
"""
from .ia_oracle import (  # noqa: F401
    k_mean, quantize, row_validity, dequantize, attention, exact_attention, merge,
    quantize_and_attend, qk_prologue, round_to_16bit, PARITY_STATUS,
)

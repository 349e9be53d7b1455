"""CPU oracle for INT8-QK attention. TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import anything here. The CUDA
library never calls, links or falls back to this code, and this code shares
nothing with it: no kernels, headers, tables or helpers.

The arithmetic is plain C++ in ``oracle/ia_oracle.cpp`` (float64 attention,
IEEE float32 quantiser decisions, exact sums, ``std::thread`` over heads and
rows); ``oracle/ia_oracle.py`` marshals numpy arrays into it.
"""
from .ia_oracle import (  # noqa: F401
    k_mean, quantize, row_validity, attention, exact_attention, merge, quantize_and_attend,
    qk_prologue, round_to_16bit, exact_sum, set_threads, hardware_threads, PARITY_STATUS,
)

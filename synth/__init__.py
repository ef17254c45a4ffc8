"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This package draws random tensors and rounds them to their storage type.
It holds none of the FFN block's arithmetic: no normalisation, no
activation, no projection.  Both the tests and ``bench.py`` take their
inputs from here, so the oracle and the kernels always see the same bytes.
"""

from .ffn_inputs import *  # noqa: F401,F403

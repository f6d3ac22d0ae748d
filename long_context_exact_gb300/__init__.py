"""GB300-native blockwise ring attention.

The compute path is the C-ABI library built from ``csrc/`` (declared in
``include/ra.h``); ``binding`` marshals torch tensors into it.  ``inputs``
draws the seeded synthetic workloads; ``accounting`` holds the useful-FLOP
and byte formulas used for reporting.
"""

from .inputs import CONTIGUOUS, STRIPED, ZIGZAG  # noqa: F401

__all__ = ["CONTIGUOUS", "STRIPED", "ZIGZAG"]
__version__ = "0.1.0"

"""Seeded synthetic inputs for the selective-scan (S6) workloads.

This module is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark. It holds only the input recipes (shapes, distributions, seeds) and
the exact rounding of the drawn values to the storage dtype; none of the
selective-scan arithmetic lives here.
"""

from .configs import CONFIGS, ScanWorkload, DecodeWorkload, get_config  # noqa: F401
from .gen import make_scan_inputs, make_decode_steps, randn_blocks  # noqa: F401

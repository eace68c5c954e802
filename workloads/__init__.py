"""Seeded synthetic inputs for the RoPE + GQA decode step.

This package only *draws* inputs: shapes, N(0,1) values rounded to the
storage type, ragged lengths, block tables built from a seeded shuffle,
shared-prefix tables and NaN poisoning of every slot the step must not read.
It holds none of the step's arithmetic (no RoPE, no cache indexing beyond
laying out the drawn values, no attention), so both the float64 oracle
tests and the CUDA path can take their inputs from it without sharing code.
"""

from .configs import CONFIGS, WorkloadConfig, get_config, reduced  # noqa: F401
from .gen import DecodeInputs, make_inputs, make_structure, bf16_bits_from_f32  # noqa: F401

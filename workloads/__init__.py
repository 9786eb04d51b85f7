"""Seeded synthetic workloads for paged decode attention.

This module only draws random structure (context lengths, physical block
placement, sharing groups) and random values.  It holds none of the method's
arithmetic: no attention, no slot arithmetic, no softmax.  Both the oracle
tests and the CUDA path take their inputs from here, so neither depends on
the other for data.
"""

from .synth import (  # noqa: F401
    CONFIGS,
    SAMPLING,
    SAMPLING_ALIGNED,
    SAMPLINGS,
    DecodeConfig,
    DecodeCase,
    SamplingConfig,
    SamplingCase,
    make_codes,
    make_int4_pool,
    make_decode_case,
    make_sampling_case,
    make_values,
    sampling_tables,
)

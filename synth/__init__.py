"""Seeded synthetic inputs for the Engram memory read.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests.  It holds none of the Engram arithmetic (no hashing, no e4m3
decoding, no reduction, no gate, no projection): it only draws random
numbers and turns them into token streams, table bytes, scales and bf16
tensors with the distributions the workloads call for.

Random numbers come from one counter-based generator, Philox4x64-10
(Salmon, Moraes, Dror & Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
SC'11), implemented here in numpy and, bit-identically, in
``synth/csrc/synth_dev.cu`` so that tables of up to ~100 GB can be filled on
the device while any single row can still be regenerated on the host.
"""

from .philox import philox4x64, philox_u32  # noqa: F401
from .sampler import (  # noqa: F401
    CdfTable,
    e4m3_normal_table,
    bf16_normal_table,
    sample_codes,
    scale_from_u32,
)
from .configs import CONFIGS, EngramConfig, default_seeds  # noqa: F401

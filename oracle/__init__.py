"""fp64 CPU oracle for WISE block-sparse causal attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline arm, never by the library.
"""
from .wise_oracle import *  # noqa: F401,F403
from .wise_oracle import (FIXED_POINT_BITS, TIE_TOLERANCE, SUPPORT_SINK, SUPPORT_DIAG,  # noqa: F401
                          causal_attention, block_mass, block_mass_rows, step_support, working_set,
                          support_to_csr, csr_to_support, block_density, identification_margin,
                          retained_mass, discover, select, sparse, to_fixed, default_scale)

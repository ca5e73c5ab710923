"""Seeded synthetic workloads (sizes and input generators) for the decode path.

This package holds no arithmetic of the method; the CUDA path and the oracle
both take their inputs from it and share nothing else.
"""
from .configs import (ALL, LLAMA_128K, LLAMA_1M, LLAMA_32K, SWEEP_64K, TINY,  # noqa: F401
                      Workload, sweep_points)
from .gen import (make_A, make_B, make_decode_inputs, make_K_exact, make_layer, make_normal,  # noqa: F401
                  make_V, spike_chunks, storage_dtype, value_dtype)

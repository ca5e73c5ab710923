"""ShadowKV decode-step sparse attention for GB300 (sm_103a).

The compute path is libshadowkv.so (hand-written CUDA kernels behind the C
ABI in include/shadowkv.h); this package is its ctypes binding.
"""
from ._binding import (FIELDS, PHASES, SKV_BF16, SKV_F32, SKV_V_HBM, SKV_V_HOST,  # noqa: F401
                       HostBuffer, Layer, ShadowKVError, SkvConfig, fetch_probe, load, make_config, model,
                       sparse_attention_noalloc, sparse_attention_noalloc_setup,
                       sparse_attention_noalloc_status, strerror,
                       validate_config)

"""Paged KV-cache decode attention for one GB300 (sm_103a).

The computation lives in ``libpa.so`` (CUDA kernels behind the C ABI of
``include/pa.h``); this package is its ctypes binding plus the seeded
workload builder used by the tests and the benchmark.
"""
from .binding import (  # noqa: F401
    PA_DEV_ERR_BLOCK_ID, PA_DEV_ERR_PAIR, PA_DEV_ERR_SEQ_LEN, PA_DEV_ERR_SLOT,
    PA_DEV_ERR_TIMEOUT, DecodeStep, PAError, decode_workspace, lib, pa_copy_blocks, pa_decode,
    pa_decode_partition_tokens, pa_decode_workspace_bytes, pa_reshape_and_cache)

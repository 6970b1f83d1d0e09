"""libjolt for B300: JoLT KV-cache encode/decode (partial Tucker by ST-HOSVD,
Hadamard-rotated block-quantized residual, Lagrangian byte allocation).

The compute path is the C-ABI shared library libjolt.so (include/jolt.h),
built by `python -m partial_tucker_rotated_st_b300.build`; `jolt` holds the
ctypes bindings (same names as the C entry points), `codec` the buffer
management of a whole encode step.
"""
from . import jolt  # noqa: F401
from .jolt import (FULL, F32, BF16, F16, TOKEN_EXACT, TOKEN_RANDOMIZED,  # noqa: F401
                   COST_FORMULA, COST_SERIALIZED, JoltConfig, JoltBlobDesc, JoltError,
                   make_config, jolt_num_candidates, jolt_workspace_size, jolt_factor_group,
                   jolt_sweep_candidates, jolt_sweep_candidates_noalloc,
                   jolt_noalloc_scratch_bytes, jolt_allocate, jolt_blob_bytes, jolt_encode,
                   jolt_decode, jolt_read_status, jolt_status_string, jolt_launch_count)

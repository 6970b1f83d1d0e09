"""The oracle: a plain, slow float64 CPU statement of JoLT's encode/decode.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
baseline leg of bench.py may import it.  It shares no code with the CUDA
library (no kernels, headers, helpers or tables): its inputs come from the
seeded generator in kvgen/, and the CUDA side never calls into it.

Modules
  jacobi  - cyclic (round-robin order) Jacobi eigensolver, float64
  jolt    - the method: ST-HOSVD factors, Hadamard rotation, block quantizer,
            distortion table, byte cost, lambda bisection, blob codec
  run     - an encode pass over a workload's units

Parity-pin status of each function is recorded in tests/test_oracle_pins.py
(what independent fact pins it).
"""
from .jacobi import jacobi_eigh, round_robin_rounds  # noqa: F401
from . import jolt  # noqa: F401

"""fp64 CPU oracle for the KDA decode / speculative-replay / routed-MoE decode path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg import this package.  The CUDA library never
calls it, links it or shares a line of code with it, and it imports nothing
from the library: both sides receive the same seeded inputs and nothing else.

Everything here is plain numpy in float64, written to be checked against the
defining equations by eye; speed is not a goal.  Modules:

* ``numerics`` -- bfloat16 rounding (the storage format the kernels use) and
  the scalar nonlinearities (sigmoid, softplus, SiLU).
* ``kda``      -- the KDA recurrent-state step (gated delta rule), the
  speculative verify window, accepted-prefix bookkeeping and replay.
* ``moe``      -- RMSNorm, dense linear maps, the sigmoid top-k router and
  the SwiGLU routed + shared experts.
* ``layer``    -- the q/k/v/gate/beta projection epilogue and the composed
  hybrid decode layer.

Parity status: every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` (closed forms, hand-worked examples under
``tests/golden/``, brute force and invariants).  No function is unpinned.
"""

from . import numerics, kda, moe, layer  # noqa: F401

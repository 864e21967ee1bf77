"""The oracle: a plain, slow, obviously correct f64 CPU statement of what the
weight-streaming projection path computes.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline leg may import it.  The CUDA library never calls it, and
it shares no code with the CUDA side (no kernels, headers, helpers, tables or
constants); the only module both sides use is ``synth``, which draws inputs and
holds none of the method's arithmetic.

Every function follows the definition it cites from the cortiq-engine source pages
(``src/gpu_wgpu/nemotron_prefill.rs``, ``src/gpu_wgpu/gemma_batch.rs``,
``src/gpu_wgpu/embryo_wide.wgsl``) or, for the q8 block format, the workload
specification (int8 codes with a binary16 scale and offset per 32-element block
along the row).  Library primitives used as steps: numpy matmul and ``exp``,
binary16→f64 conversion (``astype``), stable sorting.

Parity pins: every function here is checked by ``tests/test_oracle_pins.py``
against closed forms, invariants, brute force on tiny inputs and the constants the
pages print; no function is unpinned.
"""
from .ref import *  # noqa: F401,F403

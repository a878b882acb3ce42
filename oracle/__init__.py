"""CPU FP64 oracle for the dynamic, unmerged LoRA linear and its siblings.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call, link or run
anything in this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares no code
with the CUDA library (no kernels, headers, tables or constant generators); both sides
read their inputs from ``workloads``, which holds no arithmetic of the method.

It is plain and slow on purpose: every stored input is decoded to its exact FP64
value, the method's definition is written out with ``numpy.matmul`` as the only
library step, and nothing is blocked, fused or reordered.

Modules
  numerics     bf16 <-> fp32/fp64 decoding and round-to-nearest-even encoding
  nf4          4-bit NormalFloat codebook, unpacking and dequantisation
  dense_patch  ``.diff`` / ``.diff_b`` additive deltas and ``.set_weight`` replacement
  lora         forward (single, multi-patch, grouped), closed-form backward, and the
               unfused bf16 reference chain used by the accuracy gate
  swiglu       the SwiGLU activation around the LoRA MLP and its backward, and the
               whole MLP's forward and closed-form gradients
  merge        baking adapters into a bf16 or 4-bit weight (rounded / re-encoded once,
               deterministically or stochastically)
  rng          Philox4x32-10, the counter-based generator of the stochastic re-encoding

Parity status: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (brute force, closed forms, invariants, library
special cases); none is "parity unpinned" except the claim that the NF4 codebook is
bit-identical to the one bitsandbytes ships (see ``nf4``).
"""
from . import numerics, nf4, dense_patch, lora, swiglu, merge, rng  # noqa: F401

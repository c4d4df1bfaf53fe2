"""CPU oracle for the slot-addressed MoE layer and its cache policy.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
restatement of what the layer computes, used to check the CUDA path.  Only
the test suite, the package smoke check and the benchmark's CPU-baseline leg
may import it.  The product path (``libmoe.so`` and its binding) never calls
into it and shares no code with it: the two sides meet only in the seeded
input generator ``serving_router_top_gb300.inputs``, which holds no layer
arithmetic.

Precision: every floating-point step of the layer is computed in fp64 from
the exact values of its bf16 / FP4 / FP8 inputs; the one fp32 rounding the
method defines (router logits feed top-k as fp32) is applied where stated.
The cache policy is defined on fp32 heat counters, so it is computed in the
exact fp32 operation sequence (numpy float32 arithmetic, one IEEE rounding
per add or multiply, no fused multiply-add).

Modules
  formats  -- E2M1 / E4M3 / bf16 decoding and NVFP4 row dequantisation
  layer    -- router, top-k, expert groups, residency lookup, SwiGLU expert,
              shared expert, combine, RMSNorm stack
  policy   -- heat counters, swap planning with decay, swap application
  side     -- the pages' share and q* arithmetic (self-checks)

Parity status (what pins each part is listed in the tests):
  share-update value 0.60 printed in the Strata log -- parity unpinned
    (the printed rule gives 0.62 from the printed inputs);
  swap execution timing -- parity unpinned (invariants only).
"""
from . import formats, layer, policy, side  # noqa: F401

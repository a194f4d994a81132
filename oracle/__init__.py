"""Plain CPU oracle for the Occult collaboration-aware MoE layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute anything in this package: only the test-suite, the smoke check in
``__graft_entry__`` and the benchmark's CPU-baseline leg use it.  It shares no
code with the CUDA path (no kernels, headers, helpers or tables); both sides
only receive the same tensors from the seeded generators in ``synth``.

Everything here is written from "Occult: Optimizing Collaborative Communication
across Experts for Accelerated Parallel MoE Training and Inference" (arXiv
2505.13345) and is deliberately slow and literal:

* ``routing``   -- Eq. 2 top-k softmax router; the device-limited pruning rule.
* ``brim``      -- Algorithm 3 (BRIM0), Algorithm 4 (dispatch), Algorithm 5
                   (BRIM1), the EPD layout they imply, Algorithms 6-9 (the staged
                   Occult pipeline) for stage-wise checks.
* ``expert``    -- Eq. 1 MoE output with SwiGLU experts (fp64), dense and sparse.
* ``coact``     -- Eq. 3 co-activation graph, Eq. 4 normalisation, C_T (Sec. 2.2,
                   Eq. 5 bounds), intra/inter collaboration (Sec. 3.2).
* ``placement`` -- Algorithm 1 expert placement.
* ``backward``  -- analytic fp64 gradients of Eq. 1 for the training workload.

Floating point is fp64 throughout, computed from the exact fp32/bf16 input
values.  Where floating point decides an integer (top-k choice) the decision is
taken on the fp32 inputs exactly as given, so both sides decide identically.
"""

"""fp64 CPU oracle for the sparse-MoE Dispatch-Compute-Combine layer with LoRA experts.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm) may import it.  The
CUDA library never calls it and shares no code with it: the only thing both sides consume is
the seeded input tensors.

Everything here is plain numpy in float64, written from the pages' definitions:

* "Adapting Trillion-Parameter MoE Models for LoRA Fine-Tuning: A Full-Stack Engineering
  Guide", section 2.1, equation 1 (the MoE layer ``y = sum_{i in TopK(x)} g_i(x) E_i(x)``)
  and section 3, equation 1 (the LoRA update ``W' = W0 + (alpha/r) B A``).
* "Day-Level Adaptation and LoRA Fine-Tuning of Ultra-Large-Scale Sparse MoE Models",
  section 2.1 (top-16 selection, auxiliary load-balancing loss, expert capacity control) and
  section 3.2 (``moe_router_topk=16``, ``expert_capacity=1.25``).
* "Trillion-Parameter MoE Model Training Adaptation: Full-Stack Optimization Practices",
  section 3 "Communication" and section 4.3 (permute -> grouped GEMM -> unpermute).

Parity status: every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (closed forms, brute force, special cases that reduce to a
textbook routine, finite differences, a hand-worked example).  Parity unpinned: the real
model's expert network and router (the pages do not publish them).
"""

from .moe_oracle import *  # noqa: F401,F403

"""Plain, slow CPU oracle of the MoonEP layer path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this package: only the test-suite, the package smoke check and the
benchmark's CPU-baseline / reference leg use it.  It shares no code with the
CUDA library (no headers, helpers, tables or constants) and never reads a value
the CUDA path produced.

Modules:

* ``planner`` -- histogram, global ordinals, the constructive balancing planner
  of Theorem 1 with a fixed tie-break, the per-rank expert-grouped buffer layout
  (``cu_seqlens``) and the destination / inverse permutation of every token
  copy.
* ``layer``   -- bf16 rounding, the per-expert GEMM, the gate-weighted combine
  and ``reduce_grad``.
* ``theory``  -- the imbalance metric (maxvio), Theorem 2's bound, and a brute
  force minimum-redundancy search (max-flow feasibility) for tiny inputs.

Parity status: every function above is pinned by tests against facts the
pages or mathematics fix.  For the planner the pages fix only invariants;
*which* copies move follows a tie-break the pages leave open (for the plain
policy: smallest-id underloaded and overloaded ranks, the donor's experts in
descending id, the highest ordinals first; for the largest-first policy: the
rule stated in planner.constructive_plan), and that tie-break is pinned by
plans worked by hand from those rules (tests/golden/hand_plans.json), not by
values the pages print.
"""
from . import planner, layer, theory  # noqa: F401

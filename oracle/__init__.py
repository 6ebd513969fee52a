"""CPU oracle for the Muon optimizer step -- TEST INFRASTRUCTURE ONLY.

A plain, slow, deliberately unoptimised restatement of what the GPU library
computes, written from the method's description and not from the library.
Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  The product path
(the CUDA library and its Python binding) never imports, calls or links
anything in this package, and the two share no code: the oracle reads the
same seeded inputs (``workloads``) and nothing else.

Sources, by page title (the pages are DeepSpeed pull requests about Muon
under ZeRO):

* "Support Muon in BF16_Optimizer with FP32 gradient accumulation" --
  PR description (Muon on the original matrices after reduction, owned
  intersections copied back, FP32 momentum partitioned like the master
  weights, alignment padding excluded), validation table (17x13 and 9x17
  matrices crossing partition boundaries; compiled NS checked at
  atol 1e-4 / rtol 1e-3).
* "Run Muon once per optimizer step under ZeRO-3, not once per micro-batch"
  -- "The problem" (momentum advances once per step, NS sees the
  accumulated gradient; NS call count), "The change" (order: overflow check,
  Muon, gradient norm taken over the Muon updates, clipping; a discarded
  step leaves momentum untouched), review thread (per-head Muon through
  ``muon_num_heads``; ``ns_method`` defaults to ``'gram'``).
* "Fix Muon optimizer under ZeRO CPU offload and bound gather buffers" --
  momentum kept in the master dtype (FP32), odd-numel padding.

The pages name the "standard" and "gram" Newton-Schulz methods but print no
formula.  The readings used here (quintic coefficients, step count, epsilon,
the Gram recurrence, the per-head split axis, clipping constants) are listed
in ``newton_schulz.py`` and ``muon.py`` where they are used.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against facts that do not come from this package (SVD closed forms,
calculus facts about the quintic, torch's bfloat16 conversion, brute-force
layouts, invariants the pages state).
"""
from . import bf16, newton_schulz, muon  # noqa: F401

"""CPU oracle for speculative verify and state commit.

TEST INFRASTRUCTURE ONLY.  This package defines the expected results that the
CUDA library is checked against.  Only the tests, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it; the library itself
never does, and it imports nothing from the library.

Parity status of each function (what pins it to something other than itself):
  philox.philox4x32_10   pinned: equals cuRAND's host PHILOX4_32_10 generator
                         output word for word (tests/test_oracle_philox.py).
  verify.target_distribution
                         pinned: closed forms (softmax, argmax), hand-worked
                         top-k/top-p cases, tie cases (tests/test_oracle_target.py).
  verify.verify_row      pinned: exact enumeration of the chain's outcome law
                         for tiny vocabularies, the marginal-preservation
                         theorem, chi-square at 40k trials, greedy = argmax,
                         alpha closed form, expected accept length against the
                         pages' table, the two-level race's winner law and its
                         two-entry closed form (tests/test_oracle_chain.py).
  commit.commit          pinned: explicit per-element loops
                         (tests/test_oracle_commit.py).
"""

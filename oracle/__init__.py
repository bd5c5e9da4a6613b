"""CPU oracle for Ozaki-scheme FP64 GEMM emulation.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  The product path (``fp64_gemm_emulation_gb300``)
never imports it, and this package never imports the product path: the two
share no code, no tables and no constants.  Inputs reach the oracle as plain
numpy arrays; the seeded generators live in their own module and hold none of
the method's arithmetic.

The oracle is plain and slow on purpose.  Integer steps use exact Python
integers or float64 arithmetic on integer values small enough to be exact
(|value| < 2**53); nothing is blocked, fused or reordered beyond what the
method's own definition states.

Pages cited (by title, section, equation or table):

* "Ozaki Scheme II: mapping high-precision GEMM to a few INT8 GEMMs with CRT"
  (explainer of Ozaki, Uchino, Imamura, arXiv:2504.08009), cited as
  ``[Ozaki II, §n]``; its Algorithm 1 is cited as ``[Ozaki II, §7 step n]``.
* "Ozaki Scheme" course notes (SplitFP, SplitINT, RN split, group-wise EF,
  Hybrid), cited as ``[Ozaki notes, <algorithm> step n]``.

Modules:

* :mod:`oracle.ozaki2` -- Scheme II: parameter choice, scaling, truncation,
  symmetric residues, exact per-modulus products, CRT, range reduction and the
  single final rounding; plus the direct definition of the same result.
* :mod:`oracle.ozaki1` -- Scheme I: RN / SplitFP slicing, the triangular slice
  products and the fixed-order FP64 accumulation.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against closed forms, invariants, brute force on tiny inputs and values the
pages print.  No function is "parity unpinned".
"""

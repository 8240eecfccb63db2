"""Float64 CPU oracle for the paged split-KV append + decode attention path.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. The CUDA library never calls
it, and it never calls the CUDA library: the two share no code. The only module
both sides use is ``workloads`` (seeded inputs, no arithmetic of the method).

Contents:

- ``formats``: the cache formats written from their definitions: bf16
  round-to-nearest-even from fp32 and OCP FP8 E4M3 (bias 7, max 448, no
  infinities) round-to-nearest-even with saturation to the largest finite value.
- ``paged``: the slot-mapping append (cast on store), the read of one sequence
  through its block table, decode attention as the plain definition
  softmax(scale * q K^T) V in float64, per-split partials (m, l, acc) and their
  fixed-order merge, and the split rule.

Every function cites the passage of the pages it follows (page title, section).
Pins (tests/test_oracle_*.py, run with ``-m "not gpu"``): torch-CPU library casts
and full decode tables for the formats; brute-force float64 attention on
contiguous tensors (torch's scaled_dot_product_attention); closed forms (one key
returns its value, identical keys return the mean of the values, a two-key
worked example); merge of arbitrary partitions; page-permutation and GQA
invariances; and planted mistakes that must make those pins fail.
"""

from . import formats, paged  # noqa: F401

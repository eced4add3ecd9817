"""CPU oracle for column-wise-masked exact attention (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package. The product path never does, and this package imports
nothing from the product package: the two share only the seeded input
generators, which hold none of the method's arithmetic.

Everything here is plain, slow fp64 NumPy that follows the definitions:

* ``attention``: softmax(Q K^T * scale + M) V and its gradients, with the dense
  mask M materialised from the four boundary vectors one row block at a time
  ("FlashMask: Efficient and Rich Mask Extension of FlashAttention", abstract:
  exact result, column-wise sparse mask; "FlashMask-3", abstract: four
  query-axis boundary vectors indexed by key position).
* ``tiles``: brute-force three-way tile labels and per-key-block min/max tables
  over the materialised mask.
* ``masks_independent``: dense masks built straight from each mask family's
  definition, never from boundary vectors, to pin the encoding.

Pins (tests/test_oracle_*.py): torch fp64 scaled_dot_product_attention with a
dense boolean mask and its autograd; scipy logsumexp; central finite
differences; closed forms (one visible key, Q=0, no mask); rows of P summing to
one; the fully-masked-row convention; hand-worked tile labels and closed-form
tile counts. No function here is "parity unpinned".
"""

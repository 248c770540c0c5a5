"""CPU oracle for masked flash-attention (forward) -- TEST INFRASTRUCTURE ONLY.

This package is the plain, slow, obviously-correct definition that the CUDA
library is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it.  The library
(``masked_flash_attention_gb300``) never imports, calls or links anything from
here, and it has no CPU fallback: the two share no code, only the seeded
inputs drawn by ``workloads``.

Contents
  attention  -- numpy fp64 definition: per (batch, q-head) it materialises the
                whole masked logit matrix, takes its softmax, multiplies by V.
  brute      -- pure-Python scalar loops over the same definition, for tiny
                inputs; used to pin ``attention``.
  backward   -- gradients dQ, dK, dV of the forward (softmax Jacobian, the
                soft-cap's derivative, grouped-query sums); pinned by finite
                differences of ``attention`` in ``tests/test_oracle_backward.py``.
  kvcache    -- keys from two sources (cached rows, then the step's active
                rows) and the cache append, built on ``attention``; pinned in
                ``tests/test_oracle_kvcache.py``.

Parity pins (all in ``tests/test_oracle.py``): the ExecuTorch sliding-window
worked example, the all -inf chunk, causal equal to a lower-triangular mask and
to torch's fp64 scaled-dot-product attention, bottom-right alignment, GQA equal
to explicit K/V repetition, varlen/paged equal to per-sequence dense, softcap
limits, closed forms (uniform scores, single key), brute force on tiny inputs
(including every 0/-inf mask of a 4x4 tile and flash-sparse-attention's
1,1,4,4,keep=2 example), and hand-derived golden kept sets under
``tests/golden/``.  No function here is "parity unpinned".
"""
from . import attention, brute  # noqa: F401  (modules, not re-exported names)

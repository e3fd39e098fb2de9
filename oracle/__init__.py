"""Binary64 CPU oracle for the per-row vocabulary sampling stage (top-k / top-p / min-p / Gumbel-max).

TEST INFRASTRUCTURE -- not part of the product path. Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import or run anything under ``oracle/``. The oracle shares
no code with the CUDA path: the two sides meet only in the seeded input generators of ``workloads``,
which hold none of the method's arithmetic.

Modules:

* ``oracle.philox``  -- Philox4x32-10 from its published definition (Salmon et al., SC'11).
* ``oracle.sampler`` -- the per-row stage in binary64: canonical order, max-subtracted weights, fsum
  normaliser, top-k, compensated top-p scan with an fsum-certified boundary, min-p, Gumbel-max draw
  from the same Philox counters, selected-token log-probability; plus the stand-alone top-k select.

Every function is pinned by ``tests/test_oracle_pins.py``; none is "parity unpinned".
"""
from .philox import philox4x32_10, philox4x32_10_np, token_words  # noqa: F401
from .sampler import (  # noqa: F401
    STATUS_OK, STATUS_INVALID_ARG, STATUS_NONFINITE, BAND_REL, TIE_REL,
    RowResult, sample_row, kept_mask, softmax_lse_row, logprob_row, topk_select_row,
    order_key, canonical_order, draw, draw_many, gumbel_scores, uniform_from_word,
    gumbel_from_uniform, argmax_lowest, nucleus_count, neumaier_scan, widen,
)

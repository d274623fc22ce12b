"""Oracle for the join verdicts built from the restricted head's argmax. Test
infrastructure.

Source: "Motor de inferência Quail atinge 1 bilhão de tokens por minuto por GPU", section
"Como funciona", zero-decode bullet (a boolean AI.IF needs one token from the last prefill
pass) and cascade bullet (the output vocabulary is cut to 8 options); the AI_JOIN example of
"Quail: یک میلیارد توکن در دقیقه روی یک GPU" (the join keeps the pairs for which AI.IF
holds). Reading: suffix s (one (anchor, candidate) pair) passes when the head's argmax is
the option that stands for "true"; the join's result is the passing suffixes in
increasing order (anchor-major, since an anchor's suffixes are contiguous), with a count
per anchor.
"""
from __future__ import annotations

import numpy as np


def join_select(argmax, anchor_suffix_ptr, true_index):
    """Returns (verdict uint8 [S], selected suffix ids int32 (increasing), count per
    anchor int32 [A])."""
    am = np.asarray(argmax)
    asp = np.asarray(anchor_suffix_ptr, dtype=np.int64)
    verdict = (am == true_index).astype(np.uint8)
    selected = np.flatnonzero(verdict).astype(np.int32)
    counts = np.array([int(verdict[asp[a]:asp[a + 1]].sum()) for a in range(asp.size - 1)],
                      dtype=np.int32)
    return verdict, selected, counts

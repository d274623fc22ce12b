"""Oracle for the zero-decode restricted head (float64, numpy, CPU). Test infrastructure.

Definition followed: [P1] "Motor de inferência Quail atinge 1 bilhão de tokens por minuto
por GPU", section "Como funciona": a boolean AI.IF needs only the final prefill pass,
which emits a single token (zero-decode bullet), and the output head is cut to 8 options,
shrinking the final unembedding matrix (cascade-attention bullet); [P2] "Quail: یک
میلیارد توکن در دقیقه روی یک GPU", key points: the language head is limited to 8 output
tokens. The final RMSNorm before the head is the Qwen3 architecture's (the pages name the
model, Qwen3-4B, but not its layers): y_k = h_k * (mean_k h_k^2 + eps)^(-1/2) * gamma_k.
"""
from __future__ import annotations

import numpy as np


def rmsnorm(h, gamma, eps):
    """y = h * (mean(h^2) + eps)^(-1/2) * gamma over the last axis, in float64."""
    h = np.asarray(h, np.float64)
    r = 1.0 / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)
    return h * r * np.asarray(gamma, np.float64)


def restricted_head(h, gamma, w8, eps, row_index=None):
    """logits[n, j] = sum_k y[n, k] w8[j, k] for the 8 retained vocabulary columns, and the
    argmax (lowest index among equal maxima). `row_index` selects rows of h first (the
    last token of each suffix)."""
    h = np.asarray(h, np.float64)
    if row_index is not None:
        h = h[np.asarray(row_index, np.int64)]
    w8 = np.asarray(w8, np.float64)
    if w8.shape[0] != 8:
        raise ValueError("the restricted head has exactly 8 columns")
    logits = rmsnorm(h, gamma, eps) @ w8.T
    return logits, np.argmax(logits, axis=-1).astype(np.int32)


def top2_margin(logits):
    """Gap between the largest and second largest logit of each row."""
    s = np.sort(np.asarray(logits, np.float64), axis=-1)
    return s[:, -1] - s[:, -2]

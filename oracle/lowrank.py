"""Low-rank residual prefill in float64 (test infrastructure only).

An agent whose prompt prefix is already in the shared base cache but whose
adapter has no residual rows for it computes only the rank-``r`` factor of
its LoRA keys and values over that prefix (ForkKV guide, "Two-Tier Lookup
Mechanics", case B; LRAgent summary, section 2 "BaseShared"):
``Lk = X A_k`` and ``Lv = X A_v``, with ``X`` the layer's input hidden
states ``[n, d_model]`` and ``A`` the adapter's down-projection
``[d_model, r]`` (ForkKV guide, "Mathematical Decomposition of LoRA KV
Activations": ``W = W0 + s A B`` gives ``X W = X W0 + s (X A) B``, and the
residual cache keeps ``X A``).

The product is one library matmul in float64 on the exact values of the
(bf16) inputs; nothing is blocked or reordered.
"""
from __future__ import annotations

import numpy as np

from .residual_attention import _f64


def lowrank_projection(x, a) -> np.ndarray:
    """``X A`` in float64: ``x [n, d_model]``, ``a [d_model, r]`` -> ``[n, r]``."""
    x, a = _f64(x), _f64(a)
    if x.ndim != 2 or a.ndim != 2 or x.shape[1] != a.shape[0]:
        raise ValueError("expected x [n, d_model] and a [d_model, r]")
    return x @ a


def lora_projection(x, w0, a, b, s: float) -> np.ndarray:
    """The merged-weight LoRA projection ``X (W0 + s A B)`` in float64
    (``w0 [d_model, m]``, ``a [d_model, r]``, ``b [r, m]``): the quantity the
    base cache plus the low-rank factor reconstruct."""
    x, w0, a, b = _f64(x), _f64(w0), _f64(a), _f64(b)
    return x @ (w0 + float(s) * (a @ b))

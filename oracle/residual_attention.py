"""Materialised residual attention in float64 (test infrastructure only).

The definition followed here:

* LoRA on the key/value projections, ``W = W0 + (alpha/r) A B`` with
  ``s = alpha/r`` (ForkKV guide, "Mathematical Decomposition of LoRA KV
  Activations", first equation).
* The keys/values of adapter ``i`` split into a base part that depends only
  on ``W0`` and a residual ``s X A B`` (same section, the ``K^(i)`` and
  ``V^(i)`` decompositions); the residual cache keeps the rank-``r`` factor
  ``X A`` and applies ``B`` when needed (ForkKV guide, "The Disaggregated
  Memory Layout", item 2; LRAgent summary, section 2 "BaseShared").
* Scores ``q k^T / sqrt(d)`` over ``k = k_base + dk`` (ForkKV guide,
  "Mathematical Formulation of ResidualAttention"), then softmax and the
  value sum ("On-the-Fly Register Fusion", item 4).

Readings where the pages are silent:

* RoPE: rotate-half pairing ``(i, i + d/2)``, ``theta_i = base^(-2i/d)``,
  angle ``t * theta_i`` in float64 with ``t`` the 0-based position in the
  agent's own sequence.  The base cache holds post-RoPE keys, so only the
  residual is rotated here: ``RoPE_t(X W0 + s X A B) = Kb + s RoPE_t(Lk Bk)``
  because RoPE is linear.
* GQA: query head ``hq`` reads kv head ``hq // G`` with ``G = H_q / H_kv``.
* ``Lk`` is per layer and shared by all kv heads; ``Bk`` is ``[r, H_kv*d]``
  (a LoRA on ``k_proj``); head ``h`` uses columns ``h*d .. (h+1)*d``.
* ``s`` scales the residual only.
* Query row ``c`` of an agent with ``T`` keys and ``C`` query rows sits at
  position ``T - C + c``; with ``causal`` it sees keys ``t <= T - C + c``,
  otherwise all ``T`` keys.  Queries arrive post-RoPE.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np


def _f64(x) -> np.ndarray:
    """Inputs may be NumPy arrays or CPU torch tensors (bf16 included)."""
    if hasattr(x, "detach"):
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def rope_inv_freq(d: int, base: float) -> np.ndarray:
    """``theta_i = base^(-2i/d)`` for ``i = 0 .. d/2-1`` (float64)."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / float(d))


def rope(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotate-half RoPE of ``x[..., T, d]`` at integer positions ``pos[T]``.

    ``x'_i = x_i cos(t theta_i) - x_{i+d/2} sin(t theta_i)`` and
    ``x'_{i+d/2} = x_{i+d/2} cos(t theta_i) + x_i sin(t theta_i)``.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq(d, base)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def agent_kv(kb: np.ndarray, vb: np.ndarray, lk: np.ndarray, lv: np.ndarray,
             bk: np.ndarray, bv: np.ndarray, s: float, h: int,
             pos: np.ndarray, base: float) -> Tuple[np.ndarray, np.ndarray]:
    """Materialise ``K_a`` and ``V_a`` ``[T, d]`` of one agent and kv head.

    ``kb``/``vb``: ``[T, d]`` base rows of head ``h``; ``lk``/``lv``:
    ``[T, r]``; ``bk``/``bv``: ``[r, H_kv*d]``.
    """
    d = kb.shape[-1]
    bk_h = bk[:, h * d:(h + 1) * d]
    bv_h = bv[:, h * d:(h + 1) * d]
    u = lk @ bk_h                                   # [T, d]
    k = kb + s * rope(u, pos, base)
    v = vb + s * (lv @ bv_h)
    return k, v


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                      allowed: np.ndarray) -> np.ndarray:
    """Textbook scaled-dot-product attention.

    ``q [n, d]``, ``k [T, d]``, ``v [T, d]``, ``allowed [n, T]`` bool.  Each
    row must allow at least one key.
    """
    d = q.shape[-1]
    scores = (q @ k.T) / math.sqrt(d)
    scores = np.where(allowed, scores, -np.inf)
    m = scores.max(axis=-1, keepdims=True)
    p = np.exp(scores - m)
    p = p / p.sum(axis=-1, keepdims=True)
    return p @ v


def gather_agent_base(pages_k, pages_v, block_table_row: np.ndarray, T: int,
                      P: int) -> Tuple[np.ndarray, np.ndarray]:
    """Base ``Kb``/``Vb`` ``[T, H_kv, d]`` of one agent through its block
    table: token ``t`` is row ``t % P`` of page ``block_table_row[t // P]``."""
    pk = _f64(pages_k)
    pv = _f64(pages_v)
    t = np.arange(T)
    slots = np.asarray(block_table_row)[t // P]
    if np.any(slots < 0):
        raise ValueError("block table names no page for a live token")
    return pk[slots, t % P], pv[slots, t % P]


def query_positions(T: int, C: int) -> np.ndarray:
    """Position of each of an agent's ``C`` query rows: ``T - C + c``."""
    return np.arange(T - C, T, dtype=np.int64)


def residual_attention(pages_k, pages_v, block_table, seq_lens, lk, lv, bk,
                       bv, q, s: float, rope_base: float, causal: bool,
                       P: int = 16,
                       pairs: Optional[Iterable[Tuple[int, int]]] = None
                       ) -> np.ndarray:
    """Output ``[A, C, H_q, d]`` (float64) of every agent's query rows.

    ``pages_k``/``pages_v``: ``[n_pages, P, H_kv, d]``; ``block_table``
    ``[A, max_pages]``; ``seq_lens [A]``; ``lk[a]``/``lv[a]`` ``[T_a, r_a]``;
    ``bk[a]``/``bv[a]`` ``[r_a, H_kv*d]``; ``q [A, C, H_q, d]``.

    ``pairs`` restricts the work to some ``(agent, kv_head)`` pairs (the rest
    of the output is NaN); used to sample very large workloads.
    """
    qf = _f64(q)
    A, C, H_q, d = qf.shape
    H_kv = _f64(pages_k[:1]).shape[2]
    G = H_q // H_kv
    out = np.full((A, C, H_q, d), np.nan)
    want: Dict[int, List[int]] = {}
    if pairs is None:
        for a in range(A):
            want[a] = list(range(H_kv))
    else:
        for a, h in pairs:
            want.setdefault(int(a), []).append(int(h))
    bt = np.asarray(block_table)
    for a, heads in sorted(want.items()):
        T = int(seq_lens[a])
        kb_all, vb_all = gather_agent_base(pages_k, pages_v, bt[a], T, P)
        lk_a, lv_a = _f64(lk[a]), _f64(lv[a])
        bk_a, bv_a = _f64(bk[a]), _f64(bv[a])
        pos_k = np.arange(T, dtype=np.int64)
        pos_q = query_positions(T, C)
        if causal:
            allowed_c = pos_k[None, :] <= pos_q[:, None]       # [C, T]
        else:
            allowed_c = np.ones((C, T), dtype=bool)
        for h in heads:
            k, v = agent_kv(kb_all[:, h], vb_all[:, h], lk_a, lv_a, bk_a,
                            bv_a, s, h, pos_k, rope_base)
            for g in range(G):
                hq = h * G + g
                out[a, :, hq] = softmax_attention(qf[a, :, hq], k, v,
                                                  allowed_c)
    return out

"""Seeded synthetic inputs for shared-base residual attention.

This module only draws numbers and lays out page tables.  It holds none of
the method's arithmetic (no RoPE, no attention, no quantisation), so that the
CPU oracle (``oracle/``) and the CUDA path can both be fed from it without
sharing any code with each other.

Workload shapes follow the ForkKV guide's running example (Llama-3-8B style
layers, rank-16 LoRA on k_proj/v_proj, 16-token pages; section
"Fused ResidualAttention"), the PolyKV page's 15-agent / 4K shared pool
(section 2), and the Qwen-2.5-72B scale the ForkKV guide names in its
introduction.  All tensors are drawn with a seeded ``torch.Generator`` as fp32
``randn * std`` and rounded once to bf16 (round-to-nearest-even), so every
value handed to either side is exactly representable in bf16.

Logical model of one layer:

* ``pages_k`` / ``pages_v``: ``[n_slots, P, H_kv, d]`` bf16 base cache pages
  (post-RoPE ``Kb``/``Vb``), in *generator slot* order.  Slots are placed at
  seeded random positions so block tables are not the identity.
* ``block_table``: ``[A, max_pages]`` int32, logical page -> slot, ``-1`` past
  the end of an agent's sequence.  A shared prefix is one set of slots named
  by every agent; a page the prefix only partly fills is forked per agent
  that appends past it (copy-on-write), as is every private suffix page.
* ``lk[a]`` / ``lv[a]``: ``[T_a, r_a]`` bf16 residual cache of agent ``a``
  (``X A_k``, ``X A_v``) for the agent's whole sequence.
* ``bk[a]`` / ``bv[a]``: ``[r_a, H_kv*d]`` bf16 LoRA up-projections.
* ``q``: ``[A, C, H_q, d]`` bf16 post-RoPE queries; row ``c`` of agent ``a``
  sits at position ``T_a - C + c``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

PAGE = 16

# Published shapes used for synthetic stand-ins (all sizes are per layer).
CONFIGS: Dict[str, dict] = {
    # 4 agents over a 256-token prefix, GQA 8/2, d=64, rank 8, every tensor
    # N(0,1)*0.5.
    "tiny": dict(seed=1001, n_layers=1, A=4, C=1, H_q=8, H_kv=2, d=64,
                 prefix=256, suffix=(0, 0), ranks=(8,), s=2.0,
                 std_base=0.5, std_q=0.5, std_l=0.5, std_b=0.5),
    # Llama-3-8B layer shapes, 8 agents sharing a 32,768-token prefix.
    "llama8b_32k": dict(seed=1002, n_layers=1, A=8, C=1, H_q=32, H_kv=8,
                        d=128, prefix=32768, suffix=(0, 0), ranks=(16,),
                        s=2.0, std_base=1.0, std_q=1.0, std_l=0.1,
                        std_b=0.02),
    # 32 agents x 32 layers, 8,192 shared + uniform 0..512 private tokens,
    # ranks drawn from {8,16,32,64}.
    "agents32_layers32": dict(seed=1003, n_layers=32, A=32, C=1, H_q=32,
                              H_kv=8, d=128, prefix=8192, suffix=(0, 512),
                              ranks=(8, 16, 32, 64), s=2.0, std_base=1.0,
                              std_q=1.0, std_l=0.1, std_b=0.02),
    # Qwen2.5-72B layer shapes, 16 agents over 65,536 shared tokens, a
    # 32-token causal chunk per agent.
    "qwen72b_chunk": dict(seed=1004, n_layers=1, A=16, C=32, H_q=64, H_kv=8,
                          d=128, prefix=65536, suffix=(32, 32), ranks=(64,),
                          s=2.0, std_base=1.0, std_q=1.0, std_l=0.1,
                          std_b=0.02, causal=True),
    # Llama-3-8B shapes, 15 agents over 4,096 shared tokens, compressed pool.
    "compressed": dict(seed=1005, n_layers=1, A=15, C=1, H_q=32, H_kv=8,
                       d=128, prefix=4096, suffix=(0, 0), ranks=(16,), s=2.0,
                       std_base=1.0, std_q=1.0, std_l=0.1, std_b=0.02,
                       compressed=True),
}

VARIANTS = ("base", "peaked", "strong")


@dataclasses.dataclass
class LayerData:
    pages_k: torch.Tensor          # [n_slots, P, H_kv, d] bf16
    pages_v: torch.Tensor          # [n_slots, P, H_kv, d] bf16
    lk: List[torch.Tensor]         # A x [T_a, r_a] bf16
    lv: List[torch.Tensor]
    bk: List[torch.Tensor]         # A x [r_a, H_kv*d] bf16
    bv: List[torch.Tensor]
    q: torch.Tensor                # [A, C, H_q, d] bf16


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    variant: str
    n_layers: int
    A: int
    C: int
    H_q: int
    H_kv: int
    d: int
    P: int
    s: float
    rope_base: float
    causal: bool
    compressed: bool
    prefix: int
    suffix_lens: np.ndarray        # [A] int
    seq_lens: np.ndarray           # [A] int32
    ranks: np.ndarray              # [A] int
    block_table: np.ndarray        # [A, max_pages] int32 (slots, -1 unused)
    n_slots: int
    slot_fill: np.ndarray          # [n_slots] tokens held by each slot
    slot_owner: np.ndarray         # [n_slots] -1 shared, else agent index
    std: dict
    _cache: Dict[int, LayerData] = dataclasses.field(default_factory=dict,
                                                     repr=False)

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def max_pages(self) -> int:
        return self.block_table.shape[1]

    def layer(self, l: int) -> LayerData:
        if l not in self._cache:
            self._cache[l] = _draw_layer(self, l)
        return self._cache[l]

    def drop(self, l: Optional[int] = None) -> None:
        if l is None:
            self._cache.clear()
        else:
            self._cache.pop(l, None)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _randn(g: torch.Generator, shape, std: float) -> torch.Tensor:
    return (torch.randn(*shape, generator=g, dtype=torch.float32)
            * float(std)).to(torch.bfloat16)


def make_workload(name: str, variant: str = "base", *,
                  prefix: Optional[int] = None,
                  suffix: Optional[tuple] = None,
                  A: Optional[int] = None,
                  n_layers: Optional[int] = None,
                  ranks: Optional[tuple] = None,
                  C: Optional[int] = None,
                  seed: Optional[int] = None,
                  heads: Optional[tuple] = None) -> Workload:
    """Build the page tables of workload ``name`` (see ``CONFIGS``).

    Keyword overrides shrink a workload for tests (same shapes per token,
    fewer tokens / agents / layers); ``heads`` = (H_q, H_kv, d) changes the
    head shapes (calls that other attention kernels serve).  ``variant`` selects the stress inputs:
    ``peaked`` doubles q and plants, per agent, keys aligned with that
    agent's queries; ``strong`` draws the LoRA up-projections with std 0.5 so
    the residual is as large as the base.
    """
    if name not in CONFIGS:
        raise KeyError(f"unknown workload {name!r}; have {sorted(CONFIGS)}")
    if variant not in VARIANTS:
        raise KeyError(f"unknown variant {variant!r}")
    cfg = dict(CONFIGS[name])
    for key, val in (("prefix", prefix), ("suffix", suffix), ("A", A),
                     ("n_layers", n_layers), ("ranks", ranks), ("C", C),
                     ("seed", seed)):
        if val is not None:
            cfg[key] = val
    if heads is not None:               # (H_q, H_kv, d): other head shapes
        cfg["H_q"], cfg["H_kv"], cfg["d"] = (int(x) for x in heads)
    P = PAGE
    A_ = int(cfg["A"])
    g = _gen(cfg["seed"])
    lo, hi = cfg["suffix"]
    if hi > lo:
        suffix_lens = torch.randint(lo, hi + 1, (A_,), generator=g).numpy()
    else:
        suffix_lens = np.full(A_, lo, dtype=np.int64)
    rank_choices = tuple(cfg["ranks"])
    if len(rank_choices) > 1:
        idx = torch.randint(0, len(rank_choices), (A_,), generator=g).numpy()
        ranks = np.array([rank_choices[i] for i in idx], dtype=np.int64)
    else:
        ranks = np.full(A_, rank_choices[0], dtype=np.int64)
    prefix_len = int(cfg["prefix"])
    seq_lens = (prefix_len + suffix_lens).astype(np.int32)
    C_ = int(cfg["C"])
    if np.any(seq_lens < C_) or np.any(seq_lens < 1):
        raise ValueError("every agent needs at least C >= 1 tokens")

    # Slot plan: shared full prefix pages, a shared partial prefix page for
    # agents that never write past it, and private pages (forks of the
    # partial page + suffix pages) for the others.
    n_full = prefix_len // P
    part = prefix_len % P
    slots_fill: List[int] = []
    slots_owner: List[int] = []
    shared_full = list(range(n_full))
    slots_fill += [P] * n_full
    slots_owner += [-1] * n_full
    shared_part = -1
    if part and np.any(suffix_lens == 0):
        shared_part = len(slots_fill)
        slots_fill.append(part)
        slots_owner.append(-1)
    max_pages = int(math.ceil(int(seq_lens.max()) / P))
    bt = np.full((A_, max_pages), -1, dtype=np.int64)
    for a in range(A_):
        bt[a, :n_full] = shared_full
        T_a = int(seq_lens[a])
        n_pages_a = int(math.ceil(T_a / P))
        for lp in range(n_full, n_pages_a):
            if lp == n_full and part and suffix_lens[a] == 0:
                bt[a, lp] = shared_part
                continue
            bt[a, lp] = len(slots_fill)
            slots_fill.append(min(P, T_a - lp * P))
            slots_owner.append(a)
    n_slots = len(slots_fill)
    # Seeded random physical placement of the slots.
    perm = torch.randperm(n_slots, generator=g).numpy()
    inv_fill = np.zeros(n_slots, dtype=np.int64)
    inv_owner = np.zeros(n_slots, dtype=np.int64)
    inv_fill[perm] = np.asarray(slots_fill)
    inv_owner[perm] = np.asarray(slots_owner)
    bt = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)

    std = dict(base=cfg["std_base"], q=cfg["std_q"], l=cfg["std_l"],
               b=cfg["std_b"])
    if variant == "strong":
        std["b"] = 0.5
    if variant == "peaked":
        std["q"] = 2.0 * cfg["std_q"]
    return Workload(
        name=name, seed=int(cfg["seed"]), variant=variant,
        n_layers=int(cfg["n_layers"]), A=A_, C=C_, H_q=int(cfg["H_q"]),
        H_kv=int(cfg["H_kv"]), d=int(cfg["d"]), P=P, s=float(cfg["s"]),
        rope_base=10000.0, causal=bool(cfg.get("causal", False)),
        compressed=bool(cfg.get("compressed", False)), prefix=prefix_len,
        suffix_lens=suffix_lens, seq_lens=seq_lens, ranks=ranks,
        block_table=bt, n_slots=n_slots, slot_fill=inv_fill,
        slot_owner=inv_owner, std=std)


def _draw_layer(w: Workload, l: int) -> LayerData:
    g = _gen(w.seed * 1000 + 17 * l + VARIANTS.index(w.variant))
    H, d, P = w.H_kv, w.d, w.P
    # Base values: the shared prefix once, each agent's private tokens once.
    pre_k = _randn(g, (w.prefix, H, d), w.std["base"])
    pre_v = _randn(g, (w.prefix, H, d), w.std["base"])
    suf_k = [_randn(g, (int(n), H, d), w.std["base"]) for n in w.suffix_lens]
    suf_v = [_randn(g, (int(n), H, d), w.std["base"]) for n in w.suffix_lens]
    lk = [_randn(g, (int(T), int(r)), w.std["l"])
          for T, r in zip(w.seq_lens, w.ranks)]
    lv = [_randn(g, (int(T), int(r)), w.std["l"])
          for T, r in zip(w.seq_lens, w.ranks)]
    bk = [_randn(g, (int(r), H * d), w.std["b"]) for r in w.ranks]
    bv = [_randn(g, (int(r), H * d), w.std["b"]) for r in w.ranks]
    q = _randn(g, (w.A, w.C, w.H_q, d), w.std["q"])

    if w.variant == "peaked":
        # Per agent, three keys pointing along the mean of the agent's
        # queries of each kv head, with norm sqrt(d): their scores are about
        # |q|, far above the bulk, so attention is sharply peaked.
        G = w.G
        for a in range(w.A):
            T_a = int(w.seq_lens[a])
            pos = torch.randint(0, T_a, (3,), generator=g).tolist()
            qa = q[a].to(torch.float32).reshape(w.C, H, G, d).mean(dim=(0, 2))
            dirn = qa / qa.norm(dim=-1, keepdim=True).clamp_min(1e-6)
            key = (dirn * math.sqrt(d)).to(torch.bfloat16)
            for t in pos:
                if t < w.prefix:
                    pre_k[t] = key
                else:
                    suf_k[a][t - w.prefix] = key

    pages_k = torch.zeros((w.n_slots, P, H, d), dtype=torch.bfloat16)
    pages_v = torch.zeros((w.n_slots, P, H, d), dtype=torch.bfloat16)
    for a in range(w.A):
        T_a = int(w.seq_lens[a])
        full_k = torch.cat([pre_k, suf_k[a]], dim=0)
        full_v = torch.cat([pre_v, suf_v[a]], dim=0)
        for lp in range(int(math.ceil(T_a / P))):
            slot = int(w.block_table[a, lp])
            n = min(P, T_a - lp * P)
            pages_k[slot, :n] = full_k[lp * P: lp * P + n]
            pages_v[slot, :n] = full_v[lp * P: lp * P + n]
    return LayerData(pages_k=pages_k, pages_v=pages_v, lk=lk, lv=lv, bk=bk,
                     bv=bv, q=q)


def logical_kv(w: Workload, layer: LayerData, a: int):
    """Agent ``a``'s base K/V ``[T_a, H_kv, d]`` read through its block table.

    Pure indexing (gather), used by tests to check that what the pool holds
    equals what was appended.
    """
    T_a = int(w.seq_lens[a])
    idx = np.arange(T_a)
    slots = w.block_table[a, idx // w.P]
    rows = idx % w.P
    return layer.pages_k[slots, rows], layer.pages_v[slots, rows]

"""CPU oracle for shared-base residual attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import, call or run anything in this package.  The
library (``shared_base_kv_gb300``) never does, and it fails loudly when its
CUDA library is missing instead of falling back here.

What it computes, in plain float64 NumPy, with every agent's keys and values
materialised (no blocking, fusion or reordering):

* ``residual_attention`` -- for agent ``a`` and kv head ``h``,
  ``K_a[t] = Kb[t] + s * RoPE_t(Lk_a[t] Bk_a[:, h])`` and
  ``V_a[t] = Vb[t] + s * Lv_a[t] Bv_a[:, h]``, then textbook softmax
  attention of each query row over ``K_a``/``V_a``
  (ForkKV guide, "Mathematical Decomposition of LoRA KV Activations" and
  "Mathematical Formulation of ResidualAttention"; LRAgent summary, section 2
  "BaseShared").
* ``compress`` -- int8 per-tensor keys and 3-bit FWHT + Lloyd-Max values with
  a per-vector norm (PolyKV summary, section 2B).
* ``lowrank`` -- the residual prefill ``Lk = X A_k``, ``Lv = X A_v`` of an
  agent over a prefix the base cache already holds (ForkKV guide, "Two-Tier
  Lookup Mechanics", case B).
* ``paging`` -- the sharing classes of a block table (which agents name the
  same physical page at the same logical page; ForkKV guide, "Two-Tier Lookup
  Mechanics" and "The Copy-on-Write Paradigm").

Readings where the pages are silent (RoPE pairing, GQA head map, rounding and
tie rules, bit packing) are stated in each function's docstring.  Every
function here is pinned by a ``-m "not gpu"`` test against something other
than itself (a library routine, a closed form, brute force, or a value the
pages print).
"""
from .residual_attention import (  # noqa: F401
    rope_inv_freq, rope, agent_kv, softmax_attention, gather_agent_base,
    residual_attention, query_positions)
from .compress import (  # noqa: F401
    LLOYD_MAX_N01_8, LLOYD_MAX_BOUNDARIES, fwht, k_int8_scale, k_int8_encode,
    k_int8_decode, v3_encode, v3_decode, pack_planes, unpack_planes,
    compression_ratio, encode_pages, decode_pages)
from .paging import page_classes, coverage  # noqa: F401
from .lowrank import lowrank_projection, lora_projection  # noqa: F401

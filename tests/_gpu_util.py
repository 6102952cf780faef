"""Helpers shared by the GPU tests: oracle runs on workload data and
decoders of the pool's documented page layouts (pure indexing)."""
import numpy as np
import torch

import oracle

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
MAX_ABS_COMPRESSED = 5e-2


def oracle_out(w, layer, pairs=None, **over):
    ld = w.layer(layer)
    kw = dict(pages_k=ld.pages_k, pages_v=ld.pages_v, block_table=w.block_table,
              seq_lens=w.seq_lens, lk=ld.lk, lv=ld.lv, bk=ld.bk, bv=ld.bv, q=ld.q, s=w.s,
              rope_base=w.rope_base, causal=w.causal, P=w.P, pairs=pairs)
    kw.update(over)
    return oracle.residual_attention(**kw)


def oracle_codes(w, layer):
    ld = w.layer(layer)
    kq, ks, vc, vn = oracle.encode_pages(ld.pages_k, ld.pages_v, w.slot_fill)
    return kq, ks, vc, vn


def errors(out, ref):
    mask = ~np.isnan(ref)
    d = np.abs(out[mask] - ref[mask])
    rel = np.linalg.norm(out[mask] - ref[mask]) / max(np.linalg.norm(ref[mask]), 1e-30)
    return float(d.max()), float(d.mean()), float(rel)


def bf16_bits_to_f32(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32)


def pool_u16(pool, region):
    return pool.region(region).cpu().numpy().view(np.uint16)


def decode_base(u16, L, NP, H, d, layer, page, head, values: bool):
    """[16, d] bf16 bits of one (layer, page, head) block of the key or value
    store.  Keys: [token-group][d-chunk][token][8 d]; values: [token-chunk]
    [d-group][d][8 tokens]."""
    blk = u16[(((layer * NP + page) * H + head) * 16 * d):(((layer * NP + page) * H + head + 1) * 16 * d)]
    core = blk.reshape(2, d // 8, 8, 8)
    if values:
        return core.transpose(0, 3, 1, 2).reshape(16, d)     # [tok-chunk, tok, d-group, d]
    return core.transpose(0, 2, 1, 3).reshape(16, d)         # [tok-group, tok, d-chunk, d]


def decode_lk(u8, rp, T):
    core = u8.view(np.uint16)[: T // 8 * 8 * rp].reshape(T // 8, rp // 8, 8, 8)
    return core.transpose(0, 2, 1, 3).reshape(T // 8 * 8, rp)


def decode_lv(u8, rp, T):
    core = u8.view(np.uint16)[: T // 8 * 8 * rp].reshape(T // 8, rp // 8, 8, 8)
    return core.transpose(0, 3, 1, 2).reshape(T // 8 * 8, rp)


def as_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

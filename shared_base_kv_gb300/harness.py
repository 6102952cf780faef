"""Load a workload description into a device pool through the C ABI.

A workload (see ``workloads.py`` at the repository root) names base pages
by *slot*, each agent's logical pages by a block table of slots, and holds
per-layer base pages, residual rows, up-projections and queries on the host.
``DeviceWorkload`` allocates one pool page per slot, appends every slot's
tokens with ``fk_base_append``, registers the agents, appends their residual
rows, translates the block tables to pool page ids, and then serves
``fk_residual_attention`` calls.  It holds no attention arithmetic; only
marshalling.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import (Pool, fk_agent_register, fk_agent_register_shared, fk_base_append, fk_check, fk_fork, fk_last_launch_count,
               fk_pages_alloc, fk_pages_release, fk_pool_compress, fk_pool_load_compressed,
               fk_residual_append, fk_residual_attention)


class DeviceWorkload:
    def __init__(self, w, *, layers: Optional[list] = None, device: str = "cuda",
                 compressed: Optional[str] = None, codes: Optional[dict] = None,
                 spare_pages: int = 0, workspace_bytes: int = 0,
                 page_shuffle_seed: Optional[int] = None, shared_a: bool = False):
        """``compressed``: None, ``"gpu"`` (encode with fk_pool_compress) or
        ``"codes"`` (load the per-layer codes in ``codes[layer] = (kq,
        k_scale, vcodes_packed, vnorm)``, slot-ordered host arrays).
        ``shared_a``: True (every agent but 0 reads agent 0's low-rank rows)
        or a dict {agent: source agent} (Shared-A registration)."""
        self.w = w
        self.dev = torch.device(device)
        self.layers = list(range(w.n_layers)) if layers is None else list(layers)
        self.compressed = compressed
        if shared_a is True:
            self.share_src = {a: 0 for a in range(1, w.A)}
        else:
            self.share_src = dict(shared_a or {})
        self.shared_a = bool(self.share_src)
        rmax = int(np.max(w.ranks))
        self.pool = Pool(n_layers=w.n_layers, n_q_heads=w.H_q, n_kv_heads=w.H_kv, head_dim=w.d,
                         num_pages=w.n_slots + spare_pages, max_agents=w.A, max_rank=rmax,
                         max_tokens=int(np.max(w.seq_lens)), rope_base=w.rope_base,
                         compressed=compressed is not None, device=self.dev,
                         workspace_bytes=workspace_bytes)
        h = self.pool.h
        if page_shuffle_seed is None:
            self.slot_page = fk_pages_alloc(h, w.n_slots)        # slot -> pool page id
        else:
            # take every page, place the slots on a seeded random subset
            ids = fk_pages_alloc(h, w.n_slots + spare_pages)
            order = np.random.default_rng(page_shuffle_seed).permutation(ids.size)
            self.slot_page = ids[order[:w.n_slots]].astype(np.int32)
            if spare_pages:
                fk_pages_release(h, ids[order[w.n_slots:]])
        bt = w.block_table
        self.block_table = np.where(bt >= 0, self.slot_page[np.maximum(bt, 0)], -1).astype(np.int32)
        # Agents: register with all layers' up-projections.
        for a in range(w.A):
            r = int(w.ranks[a])
            Bk = torch.stack([w.layer(l).bk[a] for l in range(w.n_layers)]).to(self.dev)
            Bv = torch.stack([w.layer(l).bv[a] for l in range(w.n_layers)]).to(self.dev)
            if a in self.share_src:
                # Shared-A: the agent reads its source agent's low-rank rows
                # (the workload's lk/lv must then be the same for both)
                fk_agent_register_shared(h, a, self.share_src[a], w.s, Bk.contiguous(),
                                         Bv.contiguous())
            else:
                fk_agent_register(h, a, r, w.s, Bk.contiguous(), Bv.contiguous())
        for l in self.layers:
            self._load_layer(l, codes)
        # Reference counts: one per agent naming a page.
        for a in range(w.A):
            n = int(np.ceil(w.seq_lens[a] / w.P))
            fk_fork(h, self.block_table[a, :n])
        fk_pages_release(h, self.slot_page)
        torch.cuda.synchronize(self.dev)

    def _load_layer(self, l: int, codes) -> None:
        w, h = self.w, self.pool.h
        ld = w.layer(l)
        pk = ld.pages_k.to(self.dev)
        pv = ld.pages_v.to(self.dev)
        for slot in range(w.n_slots):
            n = int(w.slot_fill[slot])
            row = np.array([self.slot_page[slot]], dtype=np.int32)
            fk_base_append(h, l, row, 0, pk[slot, :n].contiguous(), pv[slot, :n].contiguous())
        for a in range(w.A):
            if a in self.share_src:
                continue
            fk_residual_append(h, l, a, 0, ld.lk[a].to(self.dev).contiguous(),
                               ld.lv[a].to(self.dev).contiguous())
        if self.compressed == "gpu":
            fk_pool_compress(h, l)
        elif self.compressed == "codes":
            kq, k_scale, vcp, vn = codes[l]
            fk_pool_load_compressed(h, l, self.slot_page,
                                    torch.from_numpy(np.ascontiguousarray(kq)).to(self.dev),
                                    torch.from_numpy(np.ascontiguousarray(vcp)).to(self.dev),
                                    torch.from_numpy(np.ascontiguousarray(vn)).to(self.dev),
                                    float(k_scale))
        torch.cuda.synchronize(self.dev)

    def queries(self, l: int) -> torch.Tensor:
        return self.w.layer(l).q.to(self.dev).contiguous()

    def attention(self, l: int, q: Optional[torch.Tensor] = None,
                  out: Optional[torch.Tensor] = None, stream=None,
                  compressed: Optional[bool] = None) -> torch.Tensor:
        w = self.w
        if q is None:
            q = self.queries(l)
        if out is None:
            out = torch.empty_like(q)
        comp = (self.compressed is not None) if compressed is None else compressed
        fk_residual_attention(self.pool.h, l, q, np.arange(w.A, dtype=np.int32),
                              self.block_table, w.seq_lens, w.causal, comp, out, stream)
        return out

    def check(self) -> None:
        fk_check(self.pool.h)

    def last_launches(self) -> int:
        return fk_last_launch_count(self.pool.h)


def main(argv=None) -> int:
    """Run one workload's attention call a few times on cuda:0 (for profilers):
    ``python -m shared_base_kv_gb300.harness compressed --calls 4``."""
    import argparse
    import os
    import sys
    ap = argparse.ArgumentParser()
    ap.add_argument("workload")
    ap.add_argument("--calls", type=int, default=4)
    args = ap.parse_args(argv)
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import workloads
    w = workloads.make_workload(args.workload)
    dw = DeviceWorkload(w, compressed="gpu" if w.compressed else None)
    q = dw.queries(0)
    out = torch.empty_like(q)
    for _ in range(args.calls):
        dw.attention(0, q, out)
    torch.cuda.synchronize()
    dw.check()
    print(f"{args.workload}: {args.calls} calls, {dw.last_launches()} launches each")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())

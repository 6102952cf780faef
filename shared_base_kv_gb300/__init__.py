"""Python binding of libforkkv (residual attention over a shared base KV cache).

Thin ctypes marshalling over the C ABI in ``include/forkkv.h``: every
``fk_*`` function here has the same name and arguments as its C
counterpart, with torch tensors standing in for device pointers and NumPy
arrays for host arrays.  All computation happens in the CUDA library; if
``libforkkv.so`` is missing or cannot be loaded, every call raises -- there
is no fallback.  ``Pool`` bundles a pool handle with the device carve-out
(a torch uint8 tensor) it lives in.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libforkkv.so")

FK_OK = 0
FK_ERR_INVALID_ARG = 1
FK_ERR_OUT_OF_PAGES = 2
FK_ERR_OOM = 3
FK_ERR_UNSUPPORTED = 4
FK_ERR_CUDA = 5
FK_ERR_DEVICE_CHECK = 6
FK_ERR_TIMEOUT = 7

FK_REGION_KB, FK_REGION_VB, FK_REGION_RC, FK_REGION_KQ, FK_REGION_VC, \
    FK_REGION_VN, FK_REGION_KS = range(7)

# Every symbol include/forkkv.h declares (checked by the CPU tests).
EXPORTS = (
    "fk_last_error", "fk_version", "fk_pool_bytes", "fk_pool_create",
    "fk_pool_destroy", "fk_pool_region", "fk_pages_alloc", "fk_pages_release",
    "fk_fork", "fk_page_refcount", "fk_agent_register", "fk_agent_release",
    "fk_base_append", "fk_residual_append", "fk_pool_compress",
    "fk_pool_load_compressed", "fk_residual_attention", "fk_last_launch_count",
    "fk_check", "fk_plan_host", "fk_plan_host_slots8", "fk_pool_set_profile_event",
    "fk_pool_set_test_stall",
    "fk_agent_rcache",
    "fk_residual_attention_noalloc", "fk_agent_register_shared",
    "fk_radix_create", "fk_radix_destroy", "fk_radix_match", "fk_radix_insert",
    "fk_radix_adapter_get", "fk_radix_adapter_attach", "fk_radix_adapter_detach",
    "fk_radix_evict", "fk_radix_stats", "fk_radix_node_ref", "fk_residual_prefill",
    "fk_radix_priority_assign", "fk_radix_priority_release", "fk_radix_priority_clear",
    "fk_radix_node_priority", "fk_radix_evict_workflow", "fk_workflow_steps",
    "fk_plan_chunk_host",
)


class FKError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"forkkv error {code}: {msg}")
        self.code = code


class fk_pool_config(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("max_agents", ctypes.c_int32), ("max_rank", ctypes.c_int32),
        ("max_tokens", ctypes.c_int32), ("rcache_rank_budget", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64), ("rope_base", ctypes.c_float),
        ("compressed", ctypes.c_int32),
    ]


class fk_work_item(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "head", "row_begin", "n_rows", "page_begin", "n_pages", "lp_begin",
        "agent_begin", "n_agents", "partial_begin", "sum_rank")]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it was never built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        P32 = ctypes.POINTER(ctypes.c_int32)
        sig = {
            "fk_last_error": (ctypes.c_char_p, []),
            "fk_version": (ctypes.c_char_p, []),
            "fk_pool_bytes": (ctypes.c_size_t, [ctypes.POINTER(fk_pool_config)]),
            "fk_pool_create": (i32, [ctypes.POINTER(fk_pool_config), vp, ctypes.c_size_t,
                                     ctypes.POINTER(vp)]),
            "fk_pool_destroy": (i32, [vp]),
            "fk_pool_region": (i32, [vp, i32, ctypes.POINTER(ctypes.c_size_t),
                                     ctypes.POINTER(ctypes.c_size_t)]),
            "fk_pages_alloc": (i32, [vp, i32, P32]),
            "fk_pages_release": (i32, [vp, i32, P32]),
            "fk_fork": (i32, [vp, P32, i32, P32]),
            "fk_page_refcount": (i32, [vp, ctypes.c_int32]),
            "fk_agent_register": (i32, [vp, i32, i32, ctypes.c_float, vp, vp, vp]),
            "fk_agent_release": (i32, [vp, i32]),
            "fk_agent_register_shared": (i32, [vp, i32, i32, ctypes.c_float, vp, vp, vp]),
            "fk_base_append": (i32, [vp, i32, P32, i32, i32, i32, vp, vp, vp]),
            "fk_residual_append": (i32, [vp, i32, i32, i32, i32, vp, vp, vp]),
            "fk_residual_prefill": (i32, [vp, i32, i32, i32, i32, vp, vp, vp, i32, vp]),
            "fk_pool_compress": (i32, [vp, i32, vp]),
            "fk_pool_load_compressed": (i32, [vp, i32, P32, i32, vp, vp, vp, ctypes.c_float, vp]),
            "fk_residual_attention": (i32, [vp, i32, vp, P32, P32, i32, P32, i32, i32, i32,
                                            i32, vp, vp]),
            "fk_residual_attention_noalloc": (i32, [vp, i32, vp, P32, P32, i32, P32, i32, i32,
                                                    i32, i32, vp, vp]),
            "fk_last_launch_count": (i32, [vp]),
            "fk_check": (i32, [vp, vp]),
            "fk_pool_set_profile_event": (i32, [vp, vp]),
            "fk_pool_set_test_stall": (i32, [vp, i32]),
            "fk_agent_rcache": (i32, [vp, i32, ctypes.POINTER(ctypes.c_size_t),
                                      ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(i32)]),
            "fk_plan_host": (i32, [i32, i32, i32, i32, i32, P32, i32, P32, P32, i32, i32, i32,
                                   ctypes.POINTER(fk_work_item), i32, P32,
                                   P32, P32, i32, P32, P32, i32, P32, P32, i32, P32]),
            "fk_plan_host_slots8": (i32, [i32, i32, i32, i32, i32, P32, i32, P32, P32, i32,
                                          ctypes.POINTER(fk_work_item), i32, P32,
                                          P32, P32, i32, P32, P32, i32, P32, P32, i32, P32]),
            "fk_radix_create": (i32, [i32, ctypes.POINTER(vp)]),
            "fk_radix_destroy": (None, [vp]),
            "fk_radix_match": (i32, [vp, P32, i32, P32, i32, ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_int64)]),
            "fk_radix_insert": (i32, [vp, P32, i32, P32, i32, ctypes.POINTER(ctypes.c_int64)]),
            "fk_radix_adapter_get": (i32, [vp, i64, ctypes.c_int32, P32]),
            "fk_radix_adapter_attach": (i32, [vp, i64, ctypes.c_int32, ctypes.c_int32]),
            "fk_radix_adapter_detach": (i32, [vp, i64, ctypes.c_int32, P32]),
            "fk_radix_evict": (i32, [vp, i32, P32, i32, ctypes.POINTER(i32)]),
            "fk_radix_stats": (i32, [vp, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
            "fk_radix_node_ref": (i32, [vp, i64, ctypes.POINTER(ctypes.c_int64)]),
            "fk_radix_priority_assign": (i32, [vp, i64, i32]),
            "fk_radix_priority_release": (i32, [vp, i64, i32]),
            "fk_radix_priority_clear": (i32, [vp]),
            "fk_radix_node_priority": (i32, [vp, i64, ctypes.POINTER(i32)]),
            "fk_radix_evict_workflow": (i32, [vp, i32, P32, i32, ctypes.POINTER(i32)]),
            "fk_workflow_steps": (i32, [i32, P32, P32, P32, P32, P32]),
            "fk_plan_chunk_host": (i32, [i32, i32, i32, i32, P32, i32, P32, i32,
                                         ctypes.POINTER(fk_work_item), i32, ctypes.POINTER(i32), P32, i32,
                                         ctypes.POINTER(i32), P32, i32, ctypes.POINTER(i32), P32,
                                         i32, P32, i32, ctypes.POINTER(i32)]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(code: int) -> None:
    if code != FK_OK:
        raise FKError(code, lib().fk_last_error().decode())


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p32(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _dev(t) -> int:
    """Device pointer of a contiguous CUDA tensor."""
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ------------------------------------------------------------- the ABI ----

def fk_version() -> str:
    return lib().fk_version().decode()


def fk_pool_bytes(cfg: fk_pool_config) -> int:
    n = lib().fk_pool_bytes(ctypes.byref(cfg))
    if n == 0:
        raise FKError(FK_ERR_INVALID_ARG, lib().fk_last_error().decode())
    return n


def fk_pool_create(cfg: fk_pool_config, dev_buf, nbytes: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().fk_pool_create(ctypes.byref(cfg), ctypes.c_void_p(_dev(dev_buf)), nbytes,
                                ctypes.byref(h)))
    return h


def fk_pool_destroy(h) -> None:
    _check(lib().fk_pool_destroy(h))


def fk_pool_region(h, region: int):
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().fk_pool_region(h, region, ctypes.byref(off), ctypes.byref(nb)))
    return off.value, nb.value


def fk_pages_alloc(h, n: int) -> np.ndarray:
    ids = np.zeros(max(n, 1), dtype=np.int32)
    _check(lib().fk_pages_alloc(h, n, _p32(ids)))
    return ids[:n]


def fk_pages_release(h, ids) -> None:
    a = _i32(ids)
    _check(lib().fk_pages_release(h, a.size, _p32(a)))


def fk_fork(h, parent_row) -> np.ndarray:
    a = _i32(parent_row)
    child = np.zeros_like(a)
    _check(lib().fk_fork(h, _p32(a), a.size, _p32(child)))
    return child


def fk_page_refcount(h, page_id: int) -> int:
    return lib().fk_page_refcount(h, int(page_id))


def fk_agent_register(h, agent: int, rank: int, s: float, Bk, Bv, stream=None) -> None:
    _check(lib().fk_agent_register(h, agent, rank, float(s), _dev(Bk), _dev(Bv), _stream(stream)))


def fk_agent_register_shared(h, agent: int, src: int, s: float, Bk, Bv, stream=None) -> None:
    """Shared-A: `agent` reads live agent `src`'s low-rank rows."""
    _check(lib().fk_agent_register_shared(h, agent, src, float(s), _dev(Bk), _dev(Bv),
                                          _stream(stream)))


def fk_agent_release(h, agent: int) -> None:
    _check(lib().fk_agent_release(h, agent))


def fk_agent_rcache(h, agent: int):
    """(byte offset of layer-0 Lk, bytes per layer of Lk+Lv, padded rank)."""
    off, lb, rp = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_int()
    _check(lib().fk_agent_rcache(h, agent, ctypes.byref(off), ctypes.byref(lb), ctypes.byref(rp)))
    return off.value, lb.value, rp.value


def fk_base_append(h, layer: int, block_table_row: np.ndarray, pos: int, Kb, Vb,
                   stream=None) -> None:
    """``block_table_row`` (int32 NumPy) is updated in place (new pages,
    copy-on-write)."""
    if block_table_row.dtype != np.int32 or not block_table_row.flags.c_contiguous:
        raise ValueError("block_table_row must be a contiguous int32 array")
    n = int(Kb.shape[0])
    _check(lib().fk_base_append(h, layer, _p32(block_table_row), block_table_row.size, pos, n,
                                _dev(Kb), _dev(Vb), _stream(stream)))


def fk_residual_append(h, layer: int, agent: int, pos: int, Lk, Lv, stream=None) -> None:
    _check(lib().fk_residual_append(h, layer, agent, pos, int(Lk.shape[0]), _dev(Lk), _dev(Lv),
                                    _stream(stream)))


def fk_residual_prefill(h, layer: int, agent: int, pos: int, X, Ak, Av, stream=None) -> None:
    """Lk = X Ak, Lv = X Av (X: bf16 [n][d_model], Ak/Av: bf16
    [d_model][rank]) computed on the device into the agent's rCache rows
    pos..pos+n-1."""
    _check(lib().fk_residual_prefill(h, layer, agent, pos, int(X.shape[0]), _dev(X), _dev(Ak),
                                     _dev(Av), int(X.shape[1]), _stream(stream)))


def fk_pool_compress(h, layer: int, stream=None) -> None:
    _check(lib().fk_pool_compress(h, layer, _stream(stream)))


def fk_pool_load_compressed(h, layer: int, page_ids, kq, vcodes, vnorm, k_scale: float,
                            stream=None) -> None:
    ids = _i32(page_ids)
    _check(lib().fk_pool_load_compressed(h, layer, _p32(ids), ids.size, _dev(kq), _dev(vcodes),
                                         _dev(vnorm), float(k_scale), _stream(stream)))


def fk_residual_attention(h, layer: int, q, agents, block_table, seq_lens, causal: bool,
                          compressed: bool, out, stream=None) -> None:
    """``q``/``out``: CUDA bf16 ``[A, C, H_q, d]``; tables are host arrays."""
    ag, bt, sl = _i32(agents), _i32(block_table), _i32(seq_lens)
    A, C = int(q.shape[0]), int(q.shape[1])
    if bt.ndim != 2 or bt.shape[0] != A:
        raise ValueError("block_table must be [A, max_pages]")
    _check(lib().fk_residual_attention(h, layer, _dev(q), _p32(ag), _p32(bt), bt.shape[1],
                                       _p32(sl), A, C, int(bool(causal)), int(bool(compressed)),
                                       _dev(out), _stream(stream)))


FK_NOALLOC_SCRATCH_BYTES = 16 << 20


def fk_residual_attention_noalloc(h, layer: int, q, agents, block_table, seq_lens, causal: bool,
                                  compressed: bool, out, stream=None) -> None:
    """fk_residual_attention for callers that must not allocate device
    memory: its scratch is a fixed 16 MiB array inside the library (see the
    header); the first call on a device sets it up, so make it before any
    stream capture, and do not overlap two such calls on the GPU."""
    ag, bt, sl = _i32(agents), _i32(block_table), _i32(seq_lens)
    A, C = int(q.shape[0]), int(q.shape[1])
    if bt.ndim != 2 or bt.shape[0] != A:
        raise ValueError("block_table must be [A, max_pages]")
    _check(lib().fk_residual_attention_noalloc(h, layer, _dev(q), _p32(ag), _p32(bt), bt.shape[1],
                                               _p32(sl), A, C, int(bool(causal)),
                                               int(bool(compressed)), _dev(out), _stream(stream)))


def fk_last_launch_count(h) -> int:
    return lib().fk_last_launch_count(h)


def fk_pool_set_profile_event(h, event) -> None:
    """``event``: a torch.cuda.Event (recorded after the main kernel) or None."""
    ptr = None if event is None else event.cuda_event
    _check(lib().fk_pool_set_profile_event(h, ptr))


def fk_pool_set_test_stall(h, on: bool) -> None:
    """Failure-detection test hook (see include/forkkv.h)."""
    _check(lib().fk_pool_set_test_stall(h, 1 if on else 0))


def fk_check(h, stream=None) -> None:
    _check(lib().fk_check(h, _stream(stream)))


def fk_plan_host(A: int, C: int, H_q: int, H_kv: int, block_table, seq_lens, ranks,
                 target_items: int, max_rows: int = 64, max_rank_sum: int = 64):
    """Work list for a call shape, built by the library on the host."""
    bt, sl, rk = _i32(block_table), _i32(seq_lens), _i32(ranks)
    n_it, n_rw, n_pg, n_ta = (ctypes.c_int() for _ in range(4))
    L = lib()
    code = L.fk_plan_host(A, C, H_q, H_kv, 16, _p32(bt), bt.shape[1], _p32(sl), _p32(rk),
                          max_rows, max_rank_sum, target_items, None, 0, ctypes.byref(n_it),
                          None, None, 0, ctypes.byref(n_rw), None, 0, ctypes.byref(n_pg),
                          None, 0, ctypes.byref(n_ta))
    if code not in (FK_OK, FK_ERR_OOM):
        _check(code)
    items = (fk_work_item * max(n_it.value, 1))()
    ra, rc = np.zeros(max(n_rw.value, 1), np.int32), np.zeros(max(n_rw.value, 1), np.int32)
    pg, ta = np.zeros(max(n_pg.value, 1), np.int32), np.zeros(max(n_ta.value, 1), np.int32)
    _check(L.fk_plan_host(A, C, H_q, H_kv, 16, _p32(bt), bt.shape[1], _p32(sl), _p32(rk),
                          max_rows, max_rank_sum, target_items, items, n_it.value,
                          ctypes.byref(n_it), _p32(ra), _p32(rc), n_rw.value,
                          ctypes.byref(n_rw), _p32(pg), n_pg.value, ctypes.byref(n_pg),
                          _p32(ta), n_ta.value, ctypes.byref(n_ta)))
    its = [{f: getattr(items[i], f) for f, _ in fk_work_item._fields_} for i in range(n_it.value)]
    return its, ra[:n_rw.value], rc[:n_rw.value], pg[:n_pg.value], ta[:n_ta.value]


def fk_plan_host_slots8(A: int, C: int, H_q: int, H_kv: int, block_table, seq_lens, ranks,
                        target_items: int):
    """The eight-slot decode kernel's work list for a call shape (host only)."""
    bt, sl, rk = _i32(block_table), _i32(seq_lens), _i32(ranks)
    n_it, n_rw, n_pg, n_ta = (ctypes.c_int() for _ in range(4))
    L = lib()
    code = L.fk_plan_host_slots8(A, C, H_q, H_kv, 16, _p32(bt), bt.shape[1], _p32(sl), _p32(rk),
                                 target_items, None, 0, ctypes.byref(n_it), None, None, 0,
                                 ctypes.byref(n_rw), None, 0, ctypes.byref(n_pg), None, 0,
                                 ctypes.byref(n_ta))
    if code not in (FK_OK, FK_ERR_OOM):
        _check(code)
    items = (fk_work_item * max(n_it.value, 1))()
    ra, rc = np.zeros(max(n_rw.value, 1), np.int32), np.zeros(max(n_rw.value, 1), np.int32)
    pg, ta = np.zeros(max(n_pg.value, 1), np.int32), np.zeros(max(n_ta.value, 1), np.int32)
    _check(L.fk_plan_host_slots8(A, C, H_q, H_kv, 16, _p32(bt), bt.shape[1], _p32(sl), _p32(rk),
                                 target_items, items, n_it.value, ctypes.byref(n_it), _p32(ra),
                                 _p32(rc), n_rw.value, ctypes.byref(n_rw), _p32(pg), n_pg.value,
                                 ctypes.byref(n_pg), _p32(ta), n_ta.value, ctypes.byref(n_ta)))
    its = [{f: getattr(items[i], f) for f, _ in fk_work_item._fields_} for i in range(n_it.value)]
    return its, ra[:n_rw.value], rc[:n_rw.value], pg[:n_pg.value], ta[:n_ta.value]


def fk_plan_chunk_host(A: int, C: int, H_q: int, H_kv: int, block_table, seq_lens, n_ctas: int):
    """The chunk kernel's work list for a call shape (host only): items,
    CTA ranges, page ids, and the combine lists (csr_ptr, csr_slots)."""
    bt, sl = _i32(block_table), _i32(seq_lens)
    counts = [ctypes.c_int() for _ in range(4)]
    L = lib()
    args = lambda it, ni, cb, nc, pg, np_, cp, ncp, cs, ns: (
        A, C, H_q, H_kv, _p32(bt), bt.shape[1], _p32(sl), n_ctas, it, ni, ctypes.byref(counts[0]),
        cb, nc, ctypes.byref(counts[1]), pg, np_, ctypes.byref(counts[2]), cp, ncp, cs, ns,
        ctypes.byref(counts[3]))
    code = L.fk_plan_chunk_host(*args(None, 0, None, 0, None, 0, None, 0, None, 0))
    if code not in (FK_OK, FK_ERR_OOM):
        _check(code)
    n_it, n_cta, n_pg, n_sl = (c.value for c in counts)
    items = (fk_work_item * max(n_it, 1))()
    cta = np.zeros(max(n_cta, 1), np.int32)
    pg = np.zeros(max(n_pg, 1), np.int32)
    ptr = np.zeros(A * C * H_q + 1, np.int32)
    slots = np.zeros(max(n_sl, 1), np.int32)
    _check(L.fk_plan_chunk_host(*args(items, n_it, _p32(cta), n_cta, _p32(pg), n_pg, _p32(ptr),
                                      ptr.size, _p32(slots), n_sl)))
    its = [{f: getattr(items[i], f) for f, _ in fk_work_item._fields_} for i in range(n_it)]
    return its, cta[:n_cta], pg[:n_pg], ptr, slots[:n_sl]


# ------------------------------------------------------- two-tier index --

class RadixIndex:
    """The library's two-tier prefix index (tier 1: token prefixes to bCache
    pages; tier 2: adapter leaves).  Argument marshalling only."""

    def __init__(self, page_size: int = 16):
        h = ctypes.c_void_p()
        _check(lib().fk_radix_create(int(page_size), ctypes.byref(h)))
        self.h = h
        self.page_size = int(page_size)

    def close(self) -> None:
        if self.h:
            lib().fk_radix_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def match(self, tokens):
        """(pages matched, their page ids, node handle)."""
        t = _i32(tokens)
        cap = t.size // self.page_size
        pages = np.zeros(max(cap, 1), np.int32)
        n = ctypes.c_int()
        node = ctypes.c_int64()
        _check(lib().fk_radix_match(self.h, _p32(t), t.size, _p32(pages), cap, ctypes.byref(n),
                                    ctypes.byref(node)))
        return n.value, pages[:n.value].copy(), node.value

    def insert(self, tokens, new_pages) -> int:
        t, p = _i32(tokens), _i32(new_pages)
        node = ctypes.c_int64()
        _check(lib().fk_radix_insert(self.h, _p32(t), t.size, _p32(p), p.size, ctypes.byref(node)))
        return node.value

    def adapter_get(self, node: int, adapter: int) -> int:
        o = ctypes.c_int32()
        _check(lib().fk_radix_adapter_get(self.h, int(node), int(adapter), ctypes.byref(o)))
        return o.value

    def adapter_attach(self, node: int, adapter: int, owner: int) -> None:
        _check(lib().fk_radix_adapter_attach(self.h, int(node), int(adapter), int(owner)))

    def adapter_detach(self, node: int, adapter: int) -> int:
        o = ctypes.c_int32()
        _check(lib().fk_radix_adapter_detach(self.h, int(node), int(adapter), ctypes.byref(o)))
        return o.value

    def evict(self, want_pages: int, cap: int = 1 << 16) -> np.ndarray:
        out = np.zeros(max(cap, 1), np.int32)
        n = ctypes.c_int()
        _check(lib().fk_radix_evict(self.h, int(want_pages), _p32(out), int(cap), ctypes.byref(n)))
        return out[:n.value].copy()

    def stats(self):
        a, b = ctypes.c_int64(), ctypes.c_int64()
        _check(lib().fk_radix_stats(self.h, ctypes.byref(a), ctypes.byref(b)))
        return a.value, b.value

    def node_ref(self, node: int) -> int:
        r = ctypes.c_int64()
        _check(lib().fk_radix_node_ref(self.h, int(node), ctypes.byref(r)))
        return r.value

    def priority_assign(self, node: int, step: int) -> None:
        _check(lib().fk_radix_priority_assign(self.h, int(node), int(step)))

    def priority_release(self, node: int, step: int) -> None:
        _check(lib().fk_radix_priority_release(self.h, int(node), int(step)))

    def priority_clear(self) -> None:
        _check(lib().fk_radix_priority_clear(self.h))

    def node_priority(self, node: int) -> Optional[int]:
        """The node's priority, or None if no agent marks it."""
        p = ctypes.c_int32()
        _check(lib().fk_radix_node_priority(self.h, int(node), ctypes.byref(p)))
        return None if p.value < 0 else p.value

    def evict_workflow(self, want_pages: int, cap: int = 1 << 16) -> np.ndarray:
        out = np.zeros(max(cap, 1), np.int32)
        n = ctypes.c_int()
        _check(lib().fk_radix_evict_workflow(self.h, int(want_pages), _p32(out), int(cap),
                                             ctypes.byref(n)))
        return out[:n.value].copy()


FK_JOIN_AND, FK_JOIN_OR = 0, 1


def workflow_steps(preds, join, fixed):
    """Steps-to-execution of every agent of an agent step graph:
    ``preds[i]`` lists agent i's predecessors, ``join[i]`` is FK_JOIN_AND or
    FK_JOIN_OR, ``fixed[i]`` a given value or None.  Returns a list with
    None for agents that never run."""
    n = len(preds)
    off = np.zeros(n + 1, np.int32)
    for i, p in enumerate(preds):
        off[i + 1] = off[i] + len(p)
    flat = _i32([int(x) for p in preds for x in p] or [0])
    j = _i32([int(x) for x in join] or [0])
    f = _i32([-1 if v is None else int(v) for v in fixed] or [0])
    out = np.zeros(max(n, 1), np.int32)
    _check(lib().fk_workflow_steps(n, _p32(off), _p32(flat), _p32(j), _p32(f), _p32(out)))
    return [None if v < 0 else int(v) for v in out[:n]]


# ------------------------------------------------------------ conveniences --

class Pool:
    """A pool handle plus the torch uint8 carve-out it lives in."""

    def __init__(self, *, n_layers: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                 num_pages: int, max_agents: int, max_rank: int, max_tokens: int,
                 rope_base: float = 10000.0, compressed: bool = False,
                 rcache_rank_budget: int = 0, workspace_bytes: int = 0, device=None):
        import torch
        self.cfg = fk_pool_config(n_layers, n_q_heads, n_kv_heads, head_dim, 16, num_pages,
                                  max_agents, max_rank, max_tokens, rcache_rank_budget,
                                  workspace_bytes, rope_base, int(bool(compressed)))
        self.nbytes = fk_pool_bytes(self.cfg)
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8,
                               device=device or torch.device("cuda"))
        pad = (-self.buf.data_ptr()) % 256
        self.mem = self.buf[pad:pad + self.nbytes]
        self.h = fk_pool_create(self.cfg, self.mem, self.nbytes)

    def close(self) -> None:
        if getattr(self, "h", None) is not None:
            fk_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def region(self, region: int):
        """A uint8 view of one region of the carve-out."""
        off, nb = fk_pool_region(self.h, region)
        return self.mem[off:off + nb]

"""GPU residual attention (through the C ABI) against the fp64 CPU oracle.

Reduced sizes compare every output element; full sizes (the workloads the
benchmark times) compare sampled (agent, kv-head) rows the oracle can afford.
Tolerances: max-abs 2e-2 and mean-abs 2e-3 on bf16 outputs; 5e-2 max for
the compressed pool, compared with the oracle run on the same codes.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from shared_base_kv_gb300 import fk_last_launch_count, harness
from _gpu_util import (MAX_ABS, MAX_ABS_COMPRESSED, MEAN_ABS, errors, oracle_codes,
                       oracle_out)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(params=["4", "8"])
def slots(request, monkeypatch):
    """Agents per decode tile, fixed when a pool is created: four (the
    default) or eight slots (d = 128, uncompressed pool)."""
    monkeypatch.setenv("FORKKV_DECODE_SLOTS", request.param)
    return request.param


REDUCED = {
    # several 128-token tiles, a ragged last page, two 4-agent row tiles
    "llama8b_32k": dict(prefix=1000, A=8),
    # private suffixes (CoW-forked partial pages), mixed ranks 8..64
    "agents32_layers32": dict(prefix=200, suffix=(0, 40), A=9, n_layers=2),
    # 32-row causal chunk per agent: 256 rows per head split in 4 tiles
    "qwen72b_chunk": dict(prefix=300, A=3),
    "tiny": {},
}


def _run(w, layer=0, **dw_kw):
    dw = harness.DeviceWorkload(w, **dw_kw)
    out = dw.attention(layer).float().cpu().numpy()
    dw.check()
    return dw, out


@pytest.mark.parametrize("variant", ["base", "peaked", "strong"])
@pytest.mark.parametrize("name", list(REDUCED))
def test_parity_reduced(name, variant, slots):
    w = workloads.make_workload(name, variant, **REDUCED[name])
    dw = harness.DeviceWorkload(w)
    for layer in range(w.n_layers):
        out = dw.attention(layer).float().cpu().numpy()
        ref = oracle_out(w, layer)
        mx, mean, rel = errors(out, ref)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (name, variant, layer, mx, mean, rel)
        assert rel < 2e-2
    dw.check()
    # decode-shaped calls (four query rows per agent) add the M-build grid
    # of the four-agent decode kernel; the eight-slot decode kernel (d = 128)
    # builds M itself
    decode_shaped = (w.H_q // w.H_kv) * w.C == 4
    eight = slots == "8" and w.d == 128
    assert fk_last_launch_count(dw.pool.h) == (3 if decode_shaped and not eight else 2)


@pytest.mark.parametrize("variant", ["base", "peaked", "strong"])
def test_parity_compressed_reduced(variant):
    w = workloads.make_workload("compressed", variant, prefix=500, A=15)
    kq, ks, vc, vn = oracle_codes(w, 0)
    dw, out = _run(w, compressed="codes", codes={0: (kq, ks, oracle.pack_planes(vc), vn)})
    kh, vh = oracle.decode_pages(kq, ks, vc, vn)
    ref = oracle_out(w, 0, pages_k=kh, pages_v=vh)
    mx, mean, rel = errors(out, ref)
    assert mx <= MAX_ABS_COMPRESSED and mean <= MEAN_ABS, (variant, mx, mean, rel)


def _sampled_pairs(w, n, seed):
    rng = np.random.default_rng(seed)
    pairs = {(0, 0), (w.A - 1, w.H_kv - 1)}
    while len(pairs) < n:
        pairs.add((int(rng.integers(w.A)), int(rng.integers(w.H_kv))))
    return sorted(pairs)


def _check_pairs(out, ref, w, pairs, max_abs=MAX_ABS):
    G = w.H_q // w.H_kv
    for a, h in pairs:
        o = out[a, :, h * G:(h + 1) * G]
        r = ref[a, :, h * G:(h + 1) * G]
        mx, mean, rel = errors(o, r)
        assert mx <= max_abs and mean <= MEAN_ABS, (a, h, mx, mean, rel)


def test_parity_full_llama8b_32k(slots):
    w = workloads.make_workload("llama8b_32k")
    dw, out = _run(w)
    pairs = _sampled_pairs(w, 6, 7)
    _check_pairs(out, oracle_out(w, 0, pairs=pairs), w, pairs)


def test_parity_full_llama8b_32k_strong(slots):
    w = workloads.make_workload("llama8b_32k", "strong")
    dw, out = _run(w)
    pairs = _sampled_pairs(w, 4, 8)
    _check_pairs(out, oracle_out(w, 0, pairs=pairs), w, pairs)


def test_parity_full_llama8b_32k_peaked(slots):
    # the variant whose planted keys make a row's weight sit in a few keys,
    # merged across the most split partials at full length
    w = workloads.make_workload("llama8b_32k", "peaked")
    dw, out = _run(w)
    pairs = _sampled_pairs(w, 4, 10)
    _check_pairs(out, oracle_out(w, 0, pairs=pairs), w, pairs)


def test_parity_full_qwen72b_chunk():
    w = workloads.make_workload("qwen72b_chunk")
    dw, out = _run(w)
    pairs = _sampled_pairs(w, 3, 9)
    _check_pairs(out, oracle_out(w, 0, pairs=pairs), w, pairs)


def test_parity_full_agents32_layers32(slots):
    w = workloads.make_workload("agents32_layers32")
    dw = harness.DeviceWorkload(w)
    outs = {}
    for layer in range(w.n_layers):
        o = dw.attention(layer)
        if layer in (0, 17, 31):
            outs[layer] = o.float().cpu().numpy()
    dw.check()
    for layer, seed in ((0, 1), (17, 2), (31, 3)):
        pairs = _sampled_pairs(w, 4, seed)
        _check_pairs(outs[layer], oracle_out(w, layer, pairs=pairs), w, pairs)


def test_parity_full_compressed():
    w = workloads.make_workload("compressed")
    kq, ks, vc, vn = oracle_codes(w, 0)
    dw, out = _run(w, compressed="codes", codes={0: (kq, ks, oracle.pack_planes(vc), vn)})
    kh, vh = oracle.decode_pages(kq, ks, vc, vn)
    ref = oracle_out(w, 0, pages_k=kh, pages_v=vh)
    mx, mean, rel = errors(out, ref)
    assert mx <= MAX_ABS_COMPRESSED and mean <= MEAN_ABS, (mx, mean, rel)
    # the quantisation error against the uncompressed oracle is reported, not gated
    full = oracle_out(w, 0)
    print("compressed vs uncompressed oracle:", errors(out, full))


def test_parity_full_tiny_stress_both():
    w = workloads.make_workload("tiny", "peaked")
    dw, out = _run(w)
    mx, mean, rel = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS


# ------------------------------------------------------- general kernel --
# Calls that are neither decode-shaped (G * C == 4) nor chunk-shaped
# (G * C >= 128 with d = 128 on the uncompressed pool) run the general
# attention kernel: a GQA group of eight, two query rows per agent, the
# compressed pool with C = 2, and d = 64 with 128 rows per agent and head.
GENERAL = {
    "gqa8_decode": dict(name="llama8b_32k", kw=dict(prefix=700, A=5, heads=(64, 8, 128))),
    "c2_gqa4": dict(name="llama8b_32k", kw=dict(prefix=500, suffix=(0, 40), A=4, C=2)),
    "c2_causal_gqa8": dict(name="qwen72b_chunk", kw=dict(prefix=300, A=3, C=2)),
    "d64_c32": dict(name="tiny", kw=dict(prefix=200, A=3, C=32)),
}


@pytest.mark.parametrize("variant", ["base", "peaked", "strong"])
@pytest.mark.parametrize("case", list(GENERAL))
def test_parity_general_kernel(case, variant):
    spec = GENERAL[case]
    w = workloads.make_workload(spec["name"], variant, **spec["kw"])
    G = w.H_q // w.H_kv
    assert G * w.C != 4 and (G * w.C < 128 or w.d != 128)    # the general kernel's shapes
    dw, out = _run(w)
    mx, mean, rel = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (case, variant, mx, mean, rel)
    assert fk_last_launch_count(dw.pool.h) == 2             # attention kernel + combine


@pytest.mark.parametrize("variant", ["base", "peaked", "strong"])
def test_parity_general_kernel_compressed_c2(variant):
    w = workloads.make_workload("compressed", variant, prefix=500, A=5, C=2)
    kq, ks, vc, vn = oracle_codes(w, 0)
    dw, out = _run(w, compressed="codes", codes={0: (kq, ks, oracle.pack_planes(vc), vn)})
    kh, vh = oracle.decode_pages(kq, ks, vc, vn)
    ref = oracle_out(w, 0, pages_k=kh, pages_v=vh)
    mx, mean, rel = errors(out, ref)
    assert mx <= MAX_ABS_COMPRESSED and mean <= MEAN_ABS, (variant, mx, mean, rel)


# ------------------------------------------------------------ edge cases --

def test_single_key_and_short_sequences(slots):
    w = workloads.make_workload("agents32_layers32", prefix=1, suffix=(0, 20), A=7, n_layers=1)
    assert w.seq_lens.min() >= 1
    dw, out = _run(w)
    mx, mean, _ = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS


@pytest.mark.parametrize("ranks,A", [((64,), 1), ((8,), 8), ((64, 8), 5)])
def test_decode_tile_shapes(slots, ranks, A):
    # one rank-64 agent (an eight-slot tile with an empty half), eight
    # rank-8 agents (one Z chunk per warpgroup), and a rank mix that leaves
    # slots empty
    w = workloads.make_workload("llama8b_32k", "strong", prefix=450, A=A, ranks=ranks)
    dw, out = _run(w)
    mx, mean, _ = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (ranks, A, mx, mean)


@pytest.mark.parametrize("name,ranks,A", [
    ("llama8b_32k", (32,), 2),     # two rank-32 agents: one tile, both in its first half
    ("llama8b_32k", (64,), 3),     # three rank-64 agents, each alone in its tile
    ("tiny", (64,), 2),            # d = 64
])
def test_split_items(slots, name, ranks, A):
    # tiles of one or two agents with 48 or more ranks: the second compute
    # warpgroup of the four-agent decode kernel takes half of the rank groups
    # and hands its sums over through tensor memory
    w = workloads.make_workload(name, "strong", prefix=700, A=A, ranks=ranks)
    assert all(int(r) == ranks[0] for r in w.ranks)
    dw, out = _run(w)
    mx, mean, rel = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS and rel < 2e-2, (name, ranks, A, mx, mean, rel)


@pytest.mark.parametrize("ranks", [(8, 64), (16,)])
def test_chunk_kernel_ranks(ranks):
    # the chunk kernel with padded ranks below its 64-rank stage (rank 8 and
    # 16 agents next to rank 64 ones)
    w = workloads.make_workload("qwen72b_chunk", "strong", prefix=250, A=3, ranks=ranks)
    dw, out = _run(w)
    mx, mean, _ = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (ranks, mx, mean)


@pytest.mark.parametrize("name,heads", [("qwen72b_chunk", (16, 8, 128)), ("qwen72b_chunk", (4, 2, 64))])
def test_causal_decode_shaped_two_tokens(slots, name, heads):
    # G = 2 query heads per kv head and C = 2 causal chunk tokens: four rows
    # per agent (the decode kernels), each with its own causal limit
    w = workloads.make_workload(name, "peaked", prefix=300, A=5, C=2, heads=heads)
    assert w.causal and (w.H_q // w.H_kv) * w.C == 4
    dw, out = _run(w)
    mx, mean, _ = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (heads, mx, mean)


def test_compressed_pool_with_private_pages():
    # partial shared page forked per agent, private suffix pages: unfilled
    # rows carry no codes and are masked
    w = workloads.make_workload("compressed", "strong", prefix=300, suffix=(0, 40), A=6)
    kq, ks, vc, vn = oracle_codes(w, 0)
    dw, out = _run(w, compressed="codes", codes={0: (kq, ks, oracle.pack_planes(vc), vn)})
    kh, vh = oracle.decode_pages(kq, ks, vc, vn)
    mx, mean, rel = errors(out, oracle_out(w, 0, pages_k=kh, pages_v=vh))
    assert mx <= MAX_ABS_COMPRESSED and mean <= MEAN_ABS, (mx, mean, rel)


def test_causal_chunk_covering_whole_sequence():
    w = workloads.make_workload("qwen72b_chunk", prefix=0, A=2)     # T == C == 32
    assert list(w.seq_lens) == [32, 32]
    dw, out = _run(w)
    mx, mean, _ = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS


def test_many_agents_many_row_tiles(slots):
    w = workloads.make_workload("llama8b_32k", "strong", prefix=300, A=40)
    dw, out = _run(w)
    mx, mean, _ = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS


def test_head_dim_64_ragged():
    w = workloads.make_workload("tiny", prefix=203, A=5)
    dw, out = _run(w)
    mx, mean, _ = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS


# ------------------------------------------------------------ invariants --

def test_repeated_calls_are_bit_identical(slots):
    w = workloads.make_workload("llama8b_32k", prefix=700, A=6)
    dw = harness.DeviceWorkload(w)
    a = dw.attention(0).clone()
    b = dw.attention(0).clone()
    assert torch.equal(a, b)


def test_physical_page_placement_is_invisible(slots):
    w = workloads.make_workload("llama8b_32k", "strong", prefix=900, A=5)
    a = harness.DeviceWorkload(w).attention(0).cpu()
    dw2 = harness.DeviceWorkload(w, spare_pages=37, page_shuffle_seed=5)
    b = dw2.attention(0).cpu()
    assert torch.equal(a, b)


def test_identical_adapters_give_identical_agents():
    w = workloads.make_workload("llama8b_32k", prefix=640, A=4)
    ld = w.layer(0)
    for a in range(1, w.A):
        ld.lk[a] = ld.lk[0].clone()
        ld.lv[a] = ld.lv[0].clone()
        ld.bk[a] = ld.bk[0].clone()
        ld.bv[a] = ld.bv[0].clone()
    ld.q[:] = ld.q[0:1]
    out = harness.DeviceWorkload(w).attention(0).cpu()
    for a in range(1, w.A):
        assert torch.equal(out[a], out[0])


def _permuted_call(dw, w, perm):
    from shared_base_kv_gb300 import fk_residual_attention
    q = dw.queries(0)[torch.from_numpy(perm).long()].contiguous()
    out = torch.empty_like(q)
    fk_residual_attention(dw.pool.h, 0, q, perm, dw.block_table[perm], w.seq_lens[perm],
                          False, False, out)
    return out.cpu()


def test_agent_order_within_tiles_is_bit_exact():
    # Six agents over one prefix form a tile of the first four and one of the
    # last two (in call order).  Reordering agents inside their tiles keeps
    # every tile, work item and split: only the agents' slots change, and
    # every row is computed from its own columns, so outputs are identical.
    w = workloads.make_workload("llama8b_32k", "strong", prefix=500, A=6)
    dw = harness.DeviceWorkload(w)
    base = dw.attention(0).cpu()
    perm = np.array([3, 1, 0, 2, 5, 4], dtype=np.int32)
    got = _permuted_call(dw, w, perm)
    assert torch.equal(got, base[torch.from_numpy(perm).long()])


def test_agent_order_across_tiles_permutes_outputs():
    # Moving an agent into another tile changes that tile's weight, so the
    # planner may cut its page run into other work items: the agent's split
    # partials are then merged in another grouping.  Equal up to rounding,
    # not bit for bit.
    w = workloads.make_workload("llama8b_32k", "strong", prefix=500, A=6)
    dw = harness.DeviceWorkload(w)
    base = dw.attention(0).float().cpu().numpy()
    perm = np.array([3, 1, 5, 0, 2, 4], dtype=np.int32)
    got = _permuted_call(dw, w, perm).float().numpy()
    assert np.abs(got - base[perm]).max() <= 2e-3


def test_parity_shared_a_mixed_tiles(slots):
    """Shared-A agents next to agents with rows of their own in one tile: 2
    and 3 read the rows of 0 and 1 (same tile), 5 reads 0's from the other
    tile.  The four-agent kernel copies each shared block once."""
    w = workloads.make_workload("llama8b_32k", "strong", prefix=700, suffix=(0, 0), A=6)
    share = {2: 0, 3: 1, 5: 0}
    ld = w.layer(0)
    for a, src in share.items():
        ld.lk[a] = ld.lk[src]
        ld.lv[a] = ld.lv[src]
    dw, out = _run(w, shared_a=share)
    mx, mean, rel = errors(out, oracle_out(w, 0))
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean, rel)
    assert np.abs(out[0] - out[2]).max() > 1e-3          # same rows, other B


def test_parity_shared_a_agents_read_one_low_rank_cache():
    """Shared-A (LRAgent summary, "BaseLRShared"): every agent has its own B
    but reads agent 0's low-rank rows; the oracle is given those same rows
    for every agent."""
    w = workloads.make_workload("llama8b_32k", prefix=1000, A=8)
    ld = w.layer(0)
    for a in range(1, w.A):
        ld.lk[a] = ld.lk[0]
        ld.lv[a] = ld.lv[0]
    dw, out = _run(w, shared_a=True)
    ref = oracle_out(w, 0)
    mx, mean, rel = errors(out, ref)
    assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean, rel)
    # agents differ only through B: their outputs must differ
    assert np.abs(out[0] - out[1]).max() > 1e-3

"""Low-rank residual prefill on the device (ForkKV guide, "Two-Tier Lookup
Mechanics", case B: the base cache holds the prefix, so only the adapter's
factor X A is computed) against the float64 oracle, read back from the
rCache's documented layout.

Tolerance, from the arithmetic: the kernel multiplies the exact bf16 inputs,
accumulates in fp32 over d_model and rounds once to bf16 (nearest even).
The rounding costs at most 2^-9 |y|; an fp32 sum of d_model products is
within d_model * 2^-24 * sum_k |x_k a_k| of the exact sum (recursive
summation bound), taken here with a factor 4 for the tensor core's own
accumulation order.  So each element is checked against
    2^-8 |ref| + d_model * 2^-22 * sum_k |x_k a_k|
and, on top, the relative Frobenius error of the whole factor must stay
below 4e-3 (bf16 rounding alone gives about 1.1e-3), which a dropped or
doubled K-chunk would break."""
import numpy as np
import pytest
import torch

import oracle
import shared_base_kv_gb300 as fk
from _gpu_util import as_u16, bf16_bits_to_f32, decode_lk, decode_lv

pytestmark = pytest.mark.gpu

L, HQ, H, D = 2, 8, 2, 128


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _pool(agents=4, max_rank=64, max_tokens=600):
    return fk.Pool(n_layers=L, n_q_heads=HQ, n_kv_heads=H, head_dim=D, num_pages=4,
                   max_agents=agents, max_rank=max_rank, max_tokens=max_tokens)


def _hidden(n, dm, seed):
    """Hidden states after the layer norm: unit-variance rows."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn(n, dm, generator=g).to(torch.bfloat16)


def _down(dm, r, seed):
    """A LoRA down-projection scaled so that X A has unit variance."""
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(dm, r, generator=g) / dm ** 0.5).to(torch.bfloat16)


def _read_factors(pool, agent, layer, T):
    off, layer_bytes, rp = fk.fk_agent_rcache(pool.h, agent)
    mem = pool.mem.cpu().numpy()
    base = off + layer * layer_bytes
    lk = decode_lk(mem[base: base + layer_bytes // 2], rp, T)
    lv = decode_lv(mem[base + layer_bytes // 2: base + layer_bytes], rp, T)
    return lk, lv, rp


def _check_factor(got_u16, X, A):
    ref = oracle.lowrank_projection(X, A)
    got = bf16_bits_to_f32(got_u16).astype(np.float64)
    dm = X.shape[1]
    mag = np.abs(X.double().numpy()) @ np.abs(A.double().numpy())
    bound = 2.0 ** -8 * np.abs(ref) + dm * 2.0 ** -22 * mag
    err = np.abs(got - ref)
    assert (err <= bound).all(), float((err / bound).max())
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 4e-3, rel


@pytest.mark.parametrize("ranks", [(8, 24, 40, 64), (16, 32, 48, 56)])
@pytest.mark.parametrize("dm", [128, 384])
def test_prefill_matches_oracle_for_every_rank(dm, ranks):
    # every rank the kernel instantiates (padded ranks 16, 32, 48, 64, with
    # and without padding columns); 300 tokens = two whole 128-token tiles
    # and a ragged tail, starting at a position that is not a multiple of 8
    pool = _pool()
    pos, n, layer = 37, 300, 1
    for agent, r in enumerate(ranks):
        B = torch.zeros(L, r, H * D, dtype=torch.bfloat16).cuda()
        fk.fk_agent_register(pool.h, agent, r, 1.0, B, B)
        X = _hidden(n, dm, 100 + agent)
        Ak, Av = _down(dm, r, 200 + agent), _down(dm, r, 300 + agent)
        fk.fk_residual_prefill(pool.h, layer, agent, pos, X.cuda(), Ak.cuda(), Av.cuda())
        torch.cuda.synchronize()
        fk.fk_check(pool.h)
        lk, lv, rp = _read_factors(pool, agent, layer, 344)
        _check_factor(lk[pos:pos + n, :r], X, Ak)
        _check_factor(lv[pos:pos + n, :r], X, Av)
        assert not lk[:pos].any() and not lv[:pos].any()              # rows before pos
        assert not lk[pos + n:].any() and not lv[pos + n:].any()      # rows after the run
        assert not lk[:, r:].any() and not lv[:, r:].any()            # rank padding stays zero
        lk0, lv0, _ = _read_factors(pool, agent, 0, 344)              # the other layer
        assert not lk0.any() and not lv0.any()
    pool.close()


def test_prefill_at_llama_width_and_one_token():
    # d_model 4096 (32 K-chunks), rank 16; then a single-token run appended
    # after it (a decode step's residual) lands in its own row
    pool = _pool(agents=1, max_rank=16, max_tokens=1200)
    dm, r, n = 4096, 16, 1000
    B = torch.zeros(L, r, H * D, dtype=torch.bfloat16).cuda()
    fk.fk_agent_register(pool.h, 0, r, 1.0, B, B)
    X = _hidden(n + 1, dm, 7)
    Ak, Av = _down(dm, r, 8), _down(dm, r, 9)
    fk.fk_residual_prefill(pool.h, 0, 0, 0, X[:n].contiguous().cuda(), Ak.cuda(), Av.cuda())
    fk.fk_residual_prefill(pool.h, 0, 0, n, X[n:].contiguous().cuda(), Ak.cuda(), Av.cuda())
    torch.cuda.synchronize()
    fk.fk_check(pool.h)
    lk, lv, _ = _read_factors(pool, 0, 0, 1008)
    _check_factor(lk[:n + 1, :r], X, Ak)
    _check_factor(lv[:n + 1, :r], X, Av)
    assert not lk[n + 1:].any()
    pool.close()


def test_prefill_and_append_agree_on_the_layout():
    # the same bf16 factor written by the append path and rebuilt by the
    # prefill with an identity down-projection (X = the factor itself,
    # d_model = 128, A = [I_r; 0]) leaves the same bytes
    pool = _pool(agents=2, max_rank=32)
    r, n = 32, 130
    B = torch.zeros(L, r, H * D, dtype=torch.bfloat16).cuda()
    for a in (0, 1):
        fk.fk_agent_register(pool.h, a, r, 1.0, B, B)
    g = torch.Generator().manual_seed(5)
    F = torch.randn(n, r, generator=g).to(torch.bfloat16)
    X = torch.zeros(n, 128, dtype=torch.bfloat16)
    X[:, :r] = F
    A = torch.zeros(128, r, dtype=torch.bfloat16)
    A[:r] = torch.eye(r, dtype=torch.bfloat16)
    fk.fk_residual_append(pool.h, 1, 0, 3, F.cuda(), F.cuda())
    fk.fk_residual_prefill(pool.h, 1, 1, 3, X.cuda(), A.cuda(), A.cuda())
    torch.cuda.synchronize()
    lk0, lv0, _ = _read_factors(pool, 0, 1, 136)
    lk1, lv1, _ = _read_factors(pool, 1, 1, 136)
    assert np.array_equal(lk0, lk1) and np.array_equal(lv0, lv1)
    assert np.array_equal(lk1[3:3 + n, :r], as_u16(F))
    pool.close()


def test_prefill_through_a_shared_a_agent_fills_the_shared_rows():
    pool = _pool(agents=2, max_rank=16)
    r, dm, n = 16, 256, 64
    B = torch.zeros(L, r, H * D, dtype=torch.bfloat16).cuda()
    fk.fk_agent_register(pool.h, 0, r, 1.0, B, B)
    fk.fk_agent_register_shared(pool.h, 1, 0, 0.5, B, B)
    X, Ak, Av = _hidden(n, dm, 1), _down(dm, r, 2), _down(dm, r, 3)
    fk.fk_residual_prefill(pool.h, 0, 1, 0, X.cuda(), Ak.cuda(), Av.cuda())
    torch.cuda.synchronize()
    lk, lv, _ = _read_factors(pool, 0, 0, 64)
    _check_factor(lk[:, :r], X, Ak)
    _check_factor(lv[:, :r], X, Av)
    pool.close()


def test_prefill_argument_errors():
    pool = _pool(agents=2, max_rank=16, max_tokens=200)
    r = 16
    B = torch.zeros(L, r, H * D, dtype=torch.bfloat16).cuda()
    fk.fk_agent_register(pool.h, 0, r, 1.0, B, B)
    X = _hidden(40, 256, 1).cuda()
    A = _down(256, r, 2).cuda()
    with pytest.raises(fk.FKError):
        fk.fk_residual_prefill(pool.h, 0, 1, 0, X, A, A)                  # unregistered agent
    with pytest.raises(fk.FKError):
        fk.fk_residual_prefill(pool.h, 2, 0, 0, X, A, A)                  # layer out of range
    with pytest.raises(fk.FKError):
        fk.fk_residual_prefill(pool.h, 0, 0, 180, X, A, A)                # past max_tokens
    with pytest.raises(fk.FKError):
        fk.fk_residual_prefill(pool.h, 0, 0, 0, X[:, :200].contiguous(), A[:200].contiguous(),
                               A[:200].contiguous())                     # d_model % 128 != 0
    flat = torch.zeros(40 * 256 + 8, dtype=torch.bfloat16, device="cuda")
    Xmis = flat[1:1 + 40 * 256].view(40, 256)                            # 2-byte aligned
    with pytest.raises(fk.FKError):
        fk.fk_residual_prefill(pool.h, 0, 0, 0, Xmis, A, A)
    fk.fk_residual_prefill(pool.h, 0, 0, 0, X[:0], A, A)                 # empty run: no-op
    torch.cuda.synchronize()
    fk.fk_check(pool.h)
    lk, lv, _ = _read_factors(pool, 0, 0, 200)
    assert not lk.any() and not lv.any()
    pool.close()


@pytest.mark.parametrize("n", [1, 127, 128, 129])
def test_prefill_runs_ending_at_the_capacity(n):
    # a run whose last token is the rCache's last row (max_tokens = 640 =
    # the padded capacity), one tile boundary either side of 128 tokens
    pool = _pool(agents=1, max_rank=32, max_tokens=640)
    r, dm = 24, 256
    B = torch.zeros(L, r, H * D, dtype=torch.bfloat16).cuda()
    fk.fk_agent_register(pool.h, 0, r, 1.0, B, B)
    X, Ak, Av = _hidden(n, dm, 50 + n), _down(dm, r, 60), _down(dm, r, 61)
    pos = 640 - n
    fk.fk_residual_prefill(pool.h, 1, 0, pos, X.cuda(), Ak.cuda(), Av.cuda())
    torch.cuda.synchronize()
    fk.fk_check(pool.h)
    lk, lv, _ = _read_factors(pool, 0, 1, 640)
    _check_factor(lk[pos:, :r], X, Ak)
    _check_factor(lv[pos:, :r], X, Av)
    assert not lk[:pos].any() and not lv[:pos].any()
    with pytest.raises(fk.FKError):                           # one row past the capacity
        fk.fk_residual_prefill(pool.h, 1, 0, pos + 1, X.cuda(), Ak.cuda(), Av.cuda())
    pool.close()


def test_prefill_wide_hidden_state():
    # d_model 8192: 64 chunks through the stage ring, rank 64 (padded rank
    # equal to the rank: no padding columns)
    pool = _pool(agents=1, max_rank=64, max_tokens=256)
    r, dm, n = 64, 8192, 200
    B = torch.zeros(L, r, H * D, dtype=torch.bfloat16).cuda()
    fk.fk_agent_register(pool.h, 0, r, 1.0, B, B)
    X, Ak, Av = _hidden(n, dm, 70), _down(dm, r, 71), _down(dm, r, 72)
    fk.fk_residual_prefill(pool.h, 0, 0, 0, X.cuda(), Ak.cuda(), Av.cuda())
    torch.cuda.synchronize()
    fk.fk_check(pool.h)
    lk, lv, _ = _read_factors(pool, 0, 0, 200)
    _check_factor(lk[:, :r], X, Ak)
    _check_factor(lv[:, :r], X, Av)
    pool.close()

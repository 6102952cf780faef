"""Pins of the CPU oracle against things other than itself (no GPU).

Each test checks one oracle function against a library routine, a closed
form, brute force on tiny inputs, or a value the pages print, chosen so that
a dropped term, a sign or index slip, or a transposed operand fails one of
them.
"""
import cmath
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import compress as oc
import importlib
ora = importlib.import_module("oracle.residual_attention")
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            vals[k] = float(v)
    return vals


# ---------------------------------------------------------------- RoPE ----

def test_rope_inv_freq_closed_form():
    th = oracle.rope_inv_freq(4, 10000.0)
    assert th.tolist() == [1.0, 0.01]
    th = oracle.rope_inv_freq(128, 10000.0)
    assert th[0] == 1.0
    assert abs(th[-1] - 10000.0 ** (-126.0 / 128.0)) < 1e-18


def test_rope_equals_complex_rotation():
    # Independent formulation: pair (x_i, x_{i+d/2}) as x_i + j x_{i+d/2}
    # and multiply by exp(j t theta_i).
    rng = _rng(1)
    d, T, base = 8, 6, 10000.0
    x = rng.standard_normal((T, d))
    pos = np.array([0, 1, 5, 17, 1000, 65535])
    got = oracle.rope(x, pos, base)
    for ti, t in enumerate(pos):
        for i in range(d // 2):
            theta = base ** (-2.0 * i / d)
            z = complex(x[ti, i], x[ti, i + d // 2]) * cmath.exp(1j * t * theta)
            assert abs(got[ti, i] - z.real) < 1e-12
            assert abs(got[ti, i + d // 2] - z.imag) < 1e-12


def test_rope_two_dims_is_rotation_matrix():
    x = np.array([[0.3, -1.2]])
    for t in (0, 1, 7):
        rot = np.array([[math.cos(t), -math.sin(t)], [math.sin(t), math.cos(t)]])
        assert np.allclose(oracle.rope(x, np.array([t]), 10000.0)[0],
                           rot @ x[0], atol=1e-14)


def test_rope_norm_and_relative_position():
    rng = _rng(2)
    d = 16
    q = rng.standard_normal(d)
    k = rng.standard_normal(d)
    for t in (0, 3, 999):
        r = oracle.rope(q[None], np.array([t]), 500.0)[0]
        assert abs(np.linalg.norm(r) - np.linalg.norm(q)) < 1e-12
    dots = []
    for m, n in ((5, 2), (103, 100), (4003, 4000)):
        dots.append(oracle.rope(q[None], np.array([m]), 500.0)[0]
                    @ oracle.rope(k[None], np.array([n]), 500.0)[0])
    assert max(dots) - min(dots) < 1e-9


def test_rope_linearity_makes_post_rope_base_shareable():
    # RoPE_t(X (W0 + s A B)) = RoPE_t(X W0) + s RoPE_t(X A B): the post-RoPE
    # base cache plus a rotated residual equals the adapted post-RoPE key.
    rng = _rng(3)
    T, din, d, r, s = 7, 12, 8, 3, 2.0
    X = rng.standard_normal((T, din))
    W0 = rng.standard_normal((din, d))
    A = rng.standard_normal((din, r))
    B = rng.standard_normal((r, d))
    pos = np.arange(T) + 40
    lhs = oracle.rope(X @ (W0 + s * A @ B), pos, 10000.0)
    rhs = oracle.rope(X @ W0, pos, 10000.0) + s * oracle.rope(X @ A @ B, pos, 10000.0)
    assert np.allclose(lhs, rhs, atol=1e-12)


# ------------------------------------------------------ low-rank prefill ----

def test_lowrank_projection_brute_force_integers():
    # small integers: every product and sum is exact, so the sums written
    # out by hand must agree to the last bit
    rng = _rng(21)
    X = rng.integers(-4, 5, (3, 5)).astype(np.float64)
    A = rng.integers(-4, 5, (5, 2)).astype(np.float64)
    got = oracle.lowrank_projection(X, A)
    assert got.shape == (3, 2)
    for i in range(3):
        for j in range(2):
            acc = 0.0
            for k in range(5):
                acc += X[i, k] * A[k, j]
            assert got[i, j] == acc


def test_lowrank_projection_special_cases():
    rng = _rng(22)
    X = rng.standard_normal((6, 8))
    assert np.array_equal(oracle.lowrank_projection(X, np.eye(8)), X)        # A = I
    assert not oracle.lowrank_projection(X, np.zeros((8, 3))).any()          # A = 0
    A = rng.standard_normal((8, 4))
    perm = np.array([2, 0, 3, 1])
    # permuting A's columns permutes the factor's columns; scaling X's rows
    # scales the factor's rows
    assert np.allclose(oracle.lowrank_projection(X, A[:, perm]),
                       oracle.lowrank_projection(X, A)[:, perm], atol=1e-13)
    dsc = np.arange(1.0, 7.0)
    assert np.allclose(oracle.lowrank_projection(dsc[:, None] * X, A),
                       dsc[:, None] * oracle.lowrank_projection(X, A), atol=1e-12)
    with pytest.raises(ValueError):
        oracle.lowrank_projection(X, A.T)                                     # transposed operand
    # bf16 inputs are taken at their exact values
    xb = torch.tensor(X, dtype=torch.bfloat16)
    ab = torch.tensor(A, dtype=torch.bfloat16)
    assert np.array_equal(oracle.lowrank_projection(xb, ab),
                          xb.double().numpy() @ ab.double().numpy())


def test_lowrank_factor_rebuilds_lora_keys_and_values():
    # base cache (post-RoPE X W0 per head) + the prefill's factor X A through
    # the oracle's residual materialisation equals the merged-weight LoRA
    # projection X (W0 + s A B), rotated for keys (ForkKV guide, "Mathematical
    # Decomposition of LoRA KV Activations")
    rng = _rng(23)
    T, dm, H_kv, d, r, s, base = 9, 16, 2, 8, 3, 0.75, 10000.0
    X = rng.standard_normal((T, dm))
    W0k, W0v = rng.standard_normal((dm, H_kv * d)), rng.standard_normal((dm, H_kv * d))
    Ak, Av = rng.standard_normal((dm, r)), rng.standard_normal((dm, r))
    Bk, Bv = rng.standard_normal((r, H_kv * d)), rng.standard_normal((r, H_kv * d))
    pos = np.arange(T)
    lk, lv = oracle.lowrank_projection(X, Ak), oracle.lowrank_projection(X, Av)
    full_k = oracle.lora_projection(X, W0k, Ak, Bk, s)
    full_v = oracle.lora_projection(X, W0v, Av, Bv, s)
    for h in range(H_kv):
        cols = slice(h * d, (h + 1) * d)
        kb = oracle.rope(X @ W0k[:, cols], pos, base)
        vb = X @ W0v[:, cols]
        k, v = oracle.agent_kv(kb, vb, lk, lv, Bk, Bv, s, h, pos, base)
        assert np.allclose(k, oracle.rope(full_k[:, cols], pos, base), atol=1e-10)
        assert np.allclose(v, full_v[:, cols], atol=1e-10)
    # the factors of the two projections are not interchangeable
    k_swapped, _ = oracle.agent_kv(oracle.rope(X @ W0k[:, :d], pos, base), X @ W0v[:, :d],
                                   lv, lk, Bk, Bv, s, 0, pos, base)
    assert not np.allclose(k_swapped, oracle.rope(full_k[:, :d], pos, base), atol=1e-3)


# ----------------------------------------------------------- attention ----

def _tiny_inputs(seed, A=2, T=(5, 3), H_q=4, H_kv=2, d=8, r=(2, 3), P=4,
                 C=1, zero_b=False):
    rng = _rng(seed)
    n_pages = sum((t + P - 1) // P for t in T)
    pages_k = rng.standard_normal((n_pages, P, H_kv, d))
    pages_v = rng.standard_normal((n_pages, P, H_kv, d))
    maxp = max((t + P - 1) // P for t in T)
    bt = np.full((A, maxp), -1)
    perm = rng.permutation(n_pages)
    k = 0
    for a in range(A):
        for lp in range((T[a] + P - 1) // P):
            bt[a, lp] = perm[k]
            k += 1
    lk = [rng.standard_normal((T[a], r[a])) for a in range(A)]
    lv = [rng.standard_normal((T[a], r[a])) for a in range(A)]
    scale_b = 0.0 if zero_b else 1.0
    bk = [scale_b * rng.standard_normal((r[a], H_kv * d)) for a in range(A)]
    bv = [scale_b * rng.standard_normal((r[a], H_kv * d)) for a in range(A)]
    q = rng.standard_normal((A, C, H_q, d))
    return dict(pages_k=pages_k, pages_v=pages_v, block_table=bt,
                seq_lens=np.array(T), lk=lk, lv=lv, bk=bk, bv=bv, q=q, P=P)


@pytest.mark.parametrize("causal,C", [(False, 1), (True, 3), (False, 3)])
def test_zero_adapter_reduces_to_library_sdpa(causal, C):
    inp = _tiny_inputs(10, T=(9, 6), C=C, zero_b=True)
    out = oracle.residual_attention(s=2.0, rope_base=10000.0, causal=causal,
                                    **inp)
    A, _, H_q, d = inp["q"].shape
    H_kv = inp["pages_k"].shape[2]
    G = H_q // H_kv
    for a in range(A):
        T = int(inp["seq_lens"][a])
        kb, vb = oracle.gather_agent_base(inp["pages_k"], inp["pages_v"],
                                          inp["block_table"][a], T, inp["P"])
        # repeat_kv: query head hq reads kv head hq // G
        k = torch.from_numpy(kb).permute(1, 0, 2).repeat_interleave(G, dim=0)
        v = torch.from_numpy(vb).permute(1, 0, 2).repeat_interleave(G, dim=0)
        q = torch.from_numpy(inp["q"][a]).permute(1, 0, 2)      # [H_q, C, d]
        mask = None
        if causal:
            qpos = torch.arange(T - C, T)[:, None]
            mask = torch.arange(T)[None, :] <= qpos
        ref = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=mask)
        assert np.allclose(out[a], ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_single_key_returns_its_value():
    inp = _tiny_inputs(11, T=(1, 1), H_q=2, H_kv=1, d=8, r=(2, 2))
    s = 1.5
    out = oracle.residual_attention(s=s, rope_base=10000.0, causal=False, **inp)
    for a in range(2):
        slot = inp["block_table"][a, 0]
        v = inp["pages_v"][slot, 0, 0] + s * inp["lv"][a][0] @ inp["bv"][a]
        assert np.allclose(out[a, 0, 0], v, atol=1e-12)
        assert np.allclose(out[a, 0, 1], v, atol=1e-12)


def test_equal_keys_give_mean_value():
    inp = _tiny_inputs(12, T=(7, 5), zero_b=False)
    inp["pages_k"][:] = inp["pages_k"][0, 0][None, None]   # every Kb equal
    for a in range(2):
        inp["bk"][a][:] = 0.0                              # no key residual
    s = 2.0
    out = oracle.residual_attention(s=s, rope_base=10000.0, causal=False, **inp)
    d = inp["q"].shape[-1]
    for a in range(2):
        T = int(inp["seq_lens"][a])
        _, vb = oracle.gather_agent_base(inp["pages_k"], inp["pages_v"],
                                         inp["block_table"][a], T, inp["P"])
        for h in range(2):
            v = vb[:, h] + s * inp["lv"][a] @ inp["bv"][a][:, h * d:(h + 1) * d]
            for g in range(2):
                assert np.allclose(out[a, 0, h * 2 + g], v.mean(0), atol=1e-12)


def _bruteforce_factored(inp, s, base, causal):
    """Scalar loops, factored forms: score = (q.Kb + s q.RoPE(Lk Bk)) / sqrt d
    with RoPE as complex rotation; out = sum p Vb + s (sum p Lv) Bv."""
    q = inp["q"]
    A, C, H_q, d = q.shape
    H_kv = inp["pages_k"].shape[2]
    G = H_q // H_kv
    P = inp["P"]
    out = np.zeros_like(q)
    for a in range(A):
        T = int(inp["seq_lens"][a])
        r = inp["lk"][a].shape[1]
        for c in range(C):
            pos_q = T - C + c
            for hq in range(H_q):
                h = hq // G
                scores = []
                for t in range(T):
                    if causal and t > pos_q:
                        continue
                    slot = inp["block_table"][a, t // P]
                    kb = inp["pages_k"][slot, t % P, h]
                    base_dot = sum(q[a, c, hq, j] * kb[j] for j in range(d))
                    u = [sum(inp["lk"][a][t, k] * inp["bk"][a][k, h * d + j]
                             for k in range(r)) for j in range(d)]
                    res_dot = 0.0
                    for i in range(d // 2):
                        th = base ** (-2.0 * i / d)
                        z = complex(u[i], u[i + d // 2]) * cmath.exp(1j * t * th)
                        res_dot += q[a, c, hq, i] * z.real + q[a, c, hq, i + d // 2] * z.imag
                    scores.append((t, (base_dot + s * res_dot) / math.sqrt(d)))
                m = max(sc for _, sc in scores)
                w = [(t, math.exp(sc - m)) for t, sc in scores]
                tot = sum(x for _, x in w)
                o_base = np.zeros(d)
                o_lr = np.zeros(r)
                for t, x in w:
                    slot = inp["block_table"][a, t // P]
                    o_base += (x / tot) * inp["pages_v"][slot, t % P, h]
                    o_lr += (x / tot) * inp["lv"][a][t]
                up = np.array([sum(o_lr[k] * inp["bv"][a][k, h * d + j]
                                   for k in range(r)) for j in range(d)])
                out[a, c, hq] = o_base + s * up
    return out


@pytest.mark.parametrize("causal,C", [(False, 1), (True, 2)])
def test_materialised_equals_bruteforce_factored(causal, C):
    inp = _tiny_inputs(13, T=(5, 4), C=C, r=(2, 3))
    s, base = 1.75, 100.0
    got = oracle.residual_attention(s=s, rope_base=base, causal=causal, **inp)
    ref = _bruteforce_factored(inp, s, base, causal)
    assert np.allclose(got, ref, atol=1e-12)


def test_bruteforce_detects_dropped_rope():
    # Power check: the brute-force pin must tell a RoPE-free residual apart.
    inp = _tiny_inputs(14, T=(5, 4))
    ref = _bruteforce_factored(inp, 2.0, 10.0, False)
    a = oracle.residual_attention(s=2.0, rope_base=10.0, causal=False, **inp)
    saved = ora.rope
    try:
        ora.rope = lambda x, pos, base: np.asarray(x, dtype=np.float64)
        b = oracle.residual_attention(s=2.0, rope_base=10.0, causal=False, **inp)
    finally:
        ora.rope = saved
    assert np.allclose(a, ref, atol=1e-12)
    assert not np.allclose(b, ref, atol=1e-3)


def test_physical_page_permutation_invariance():
    inp = _tiny_inputs(15, T=(9, 7))
    out1 = oracle.residual_attention(s=2.0, rope_base=10000.0, causal=False, **inp)
    n = inp["pages_k"].shape[0]
    perm = _rng(0).permutation(n)
    inv = np.argsort(perm)
    inp2 = dict(inp)
    inp2["pages_k"] = inp["pages_k"][perm]
    inp2["pages_v"] = inp["pages_v"][perm]
    inp2["block_table"] = np.where(inp["block_table"] >= 0,
                                   inv[np.maximum(inp["block_table"], 0)], -1)
    out2 = oracle.residual_attention(s=2.0, rope_base=10000.0, causal=False, **inp2)
    assert np.array_equal(out1, out2)


# -------------------------------------------------------- compression ----

def test_compression_ratio_matches_page():
    g = _read_golden("polykv_compression_ratio.txt")
    r = oc.compression_ratio(int(g["base_bits"]), int(g["k_bits"]), int(g["v_bits"]))
    assert r == g["base_bits"] / g["denominator"]
    assert round(r, 2) == g["ratio_printed"]


def test_lloyd_max_levels_are_a_lloyd_fixed_point():
    from scipy.stats import norm
    c = oc.LLOYD_MAX_N01_8
    b = np.concatenate([[-np.inf], oc.LLOYD_MAX_BOUNDARIES, [np.inf]])
    for j in range(8):
        lo, hi = b[j], b[j + 1]
        cond_mean = (norm.pdf(lo) - norm.pdf(hi)) / (norm.cdf(hi) - norm.cdf(lo))
        assert abs(cond_mean - c[j]) < 5e-5
    assert np.allclose(oc.LLOYD_MAX_BOUNDARIES,
                       [(c[j] + c[j + 1]) / 2 for j in range(7)])


def test_lloyd_max_distortion_is_classical_value():
    from scipy import integrate
    from scipy.stats import norm
    c = oc.LLOYD_MAX_N01_8
    b = np.concatenate([[-np.inf], oc.LLOYD_MAX_BOUNDARIES, [np.inf]])
    mse = sum(integrate.quad(lambda x, cj=c[j]: (x - cj) ** 2 * norm.pdf(x),
                             b[j], b[j + 1])[0] for j in range(8))
    assert abs(mse - 0.03455) < 1e-4


def test_fwht_equals_library_hadamard():
    from scipy.linalg import hadamard
    rng = _rng(20)
    for n in (2, 8, 128):
        x = rng.standard_normal((3, n))
        assert np.allclose(oc.fwht(x), x @ hadamard(n), atol=1e-12)


def test_fwht_round_trip_and_parseval():
    rng = _rng(21)
    x = rng.standard_normal((4, 128))
    y = oc.fwht(x)
    assert np.allclose(oc.fwht(y) / 128.0, x, atol=1e-12)
    assert np.allclose((y * y).sum(-1), 128.0 * (x * x).sum(-1))


def test_int8_keys_within_half_step():
    rng = _rng(22)
    k = rng.standard_normal((64, 8, 128)) * 3.0
    scale = oc.k_int8_scale(k)
    assert scale.dtype == np.float32
    assert scale == np.float32(np.abs(k).max() / 127.0)
    qk = oc.k_int8_encode(k, scale)
    assert qk.dtype == np.int8 and qk.min() >= -127 and qk.max() <= 127
    err = np.abs(oc.k_int8_decode(qk, scale) - k)
    assert err.max() <= float(scale) / 2 * (1 + 1e-6)
    i = np.unravel_index(np.argmax(np.abs(k)), k.shape)
    assert abs(int(qk[i])) == 127
    assert oc.k_int8_scale(np.zeros(5)) == np.float32(1.0)


def test_encode_pages_scale_over_filled_rows_only():
    # PolyKV summary, section 2B: one key scale per tensor, max|K| / 127.  The
    # layer's key tensor is the filled rows of its pages; rows past a page's
    # fill (and empty pages) hold no token and must neither set the scale
    # nor carry codes.
    rng = _rng(41)
    n, P, H, d = 3, 16, 2, 128
    pk = rng.uniform(-1.0, 1.0, (n, P, H, d))
    pv = rng.standard_normal((n, P, H, d))
    fill = np.array([16, 5, 0])
    pk[0, 3, 1, 7] = -3.0                  # the largest filled magnitude
    pk[1, 5:] = 1000.0                     # past page 1's fill
    pk[2] = -1000.0                        # an empty page
    kq, scale, codes, norms = oc.encode_pages(pk, pv, fill)
    assert scale == np.float32(3.0 / 127.0)
    assert kq[0, 3, 1, 7] == -127
    live = np.arange(P)[None, :] < fill[:, None]
    assert not np.any(kq[~live]) and not np.any(codes[~live]) and not np.any(norms[~live])
    # a filled row keeps its own codes: |K / scale| rounds to within half a
    # step, and each value row's norm is its length
    dec = kq[live].astype(np.float64) * float(scale)
    assert np.abs(dec - pk[live]).max() <= float(scale) / 2 * (1 + 1e-6)
    assert np.allclose(norms[live], np.linalg.norm(pv[live], axis=-1), rtol=1e-6)


def test_int8_round_half_even():
    scale = np.float32(0.5)
    k = np.array([0.25, 0.75, -0.25, 1.25])          # K/scale = .5, 1.5, -.5, 2.5
    assert oc.k_int8_encode(k, scale).tolist() == [0, 2, 0, 2]


def test_v3_codes_are_nearest_level():
    rng = _rng(23)
    v = rng.standard_normal((50, 128)) * 2.0
    codes, norms = oc.v3_encode(v)
    from scipy.linalg import hadamard
    z = v @ hadamard(128) / np.linalg.norm(v, axis=-1, keepdims=True)
    nearest = np.argmin(np.abs(z[..., None] - oc.LLOYD_MAX_N01_8), axis=-1)
    assert np.array_equal(codes, nearest)
    assert norms.dtype == np.float32
    assert np.allclose(norms, np.linalg.norm(v, axis=-1), rtol=1e-7)


def test_v3_tie_goes_up_and_zero_vector():
    b = oc.LLOYD_MAX_BOUNDARIES
    idx = np.searchsorted(b, b, side="right")
    assert idx.tolist() == list(range(1, 8))
    codes, norms = oc.v3_encode(np.zeros((1, 128)))
    assert norms[0] == 0 and np.all(oc.v3_decode(codes, norms) == 0)


def test_v3_decode_error_is_parseval_of_code_error():
    from scipy.linalg import hadamard
    rng = _rng(24)
    v = rng.standard_normal((20, 128))
    codes, norms = oc.v3_encode(v)
    vh = oc.v3_decode(codes, norms)
    n = np.linalg.norm(v, axis=-1)
    z = v @ hadamard(128) / n[:, None]
    zh = oc.LLOYD_MAX_N01_8[codes]
    # decoded with the fp32 norm: v_hat = n32 H zh / d
    assert np.allclose(vh, norms[:, None].astype(np.float64) * (zh @ hadamard(128)) / 128,
                       atol=1e-12)
    lhs = ((v - n[:, None] * (zh @ hadamard(128)) / 128) ** 2).sum(-1)
    rhs = n ** 2 * ((z - zh) ** 2).sum(-1) / 128
    assert np.allclose(lhs, rhs, rtol=1e-9)


def test_pack_planes_round_trip_and_bit_order():
    rng = _rng(25)
    codes = rng.integers(0, 8, size=(7, 128)).astype(np.uint8)
    packed = oc.pack_planes(codes)
    assert packed.shape == (7, 48)
    assert np.array_equal(oc.unpack_planes(packed, 128), codes)
    one = np.zeros((1, 128), np.uint8)
    one[0, 9] = 5                      # bits 0 and 2 of code 9
    p = oc.pack_planes(one)[0]
    assert p[1] == 2 and p[16 + 1] == 0 and p[32 + 1] == 2
    assert p.sum() == 4


# ------------------------------------------------------------- paging ----

def test_page_classes_by_hand():
    bt = np.array([[7, 3, 9, -1],
                   [7, 3, 4, 5],
                   [7, 2, -1, -1]])
    seq = np.array([40, 64, 20])
    P = 16
    got = oracle.page_classes(bt, seq, P)
    assert got == [(0, 7, (0, 1, 2)), (1, 2, (2,)), (1, 3, (0, 1)),
                   (2, 4, (1,)), (2, 9, (0,)), (3, 5, (1,))]
    cov = oracle.coverage(bt, seq, P)
    assert len(cov) == 3 + 4 + 2


def test_workload_tables_follow_copy_on_write():
    w = workloads.make_workload("agents32_layers32", prefix=40, n_layers=1,
                                A=6, suffix=(0, 20))
    classes = oracle.page_classes(w.block_table, w.seq_lens, w.P)
    for lp, ph, agents in classes:
        if lp < w.prefix // w.P:
            assert agents == tuple(range(w.A))          # full prefix pages shared
        elif len(agents) > 1:
            # only a partial prefix page may stay shared, by agents that
            # never wrote past the prefix
            assert lp == w.prefix // w.P
            assert all(w.suffix_lens[a] == 0 for a in agents)


# ------------------------------------------------ null-kernel sanity gate ----

def _oracle_out(w, layer, **over):
    ld = w.layer(layer)
    kw = dict(pages_k=ld.pages_k, pages_v=ld.pages_v, block_table=w.block_table,
              seq_lens=w.seq_lens, lk=ld.lk, lv=ld.lv, bk=ld.bk, bv=ld.bv,
              q=ld.q, s=w.s, rope_base=w.rope_base, causal=w.causal, P=w.P)
    kw.update(over)
    return oracle.residual_attention(**kw)


@pytest.mark.parametrize("variant", ["peaked", "strong"])
def test_stress_variants_reject_null_and_base_only_kernels(variant):
    # A kernel that writes zeros, or ignores the adapters, must fail the
    # parity tolerance (max-abs 2e-2) on the stress inputs.
    w = workloads.make_workload("llama8b_32k", variant, prefix=512, A=3)
    ref = _oracle_out(w, 0)
    ld = w.layer(0)
    base_only = _oracle_out(w, 0, bk=[b * 0 for b in ld.bk], bv=[b * 0 for b in ld.bv])
    assert np.abs(ref).max() > 2e-2
    assert np.abs(base_only - ref).max() > 2e-2


def test_tiny_workload_residual_is_visible():
    w = workloads.make_workload("tiny")
    ref = _oracle_out(w, 0)
    ld = w.layer(0)
    base_only = _oracle_out(w, 0, bk=[b * 0 for b in ld.bk], bv=[b * 0 for b in ld.bv])
    assert np.abs(base_only - ref).max() > 2e-2
    assert np.abs(base_only - ref).mean() > 2e-3

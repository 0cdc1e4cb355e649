"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to a closed form, a worked example printed on the
ShadowKV review page, an invariant of the mathematics, a brute-force answer on
a tiny input, or an independent library routine for a special case.
"""
import itertools
import math

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import shadowkv_oracle as O


def _complex_rope(x, pos, theta):
    """RoPE written as multiplication by exp(i * pos * freq) on the complex pair
    (x_i + i x_{i+d/2}) -- an independent formulation of rotate-half RoPE."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    half = d // 2
    freq = np.array([theta ** (-2.0 * i / d) for i in range(half)])
    z = x[..., :half] + 1j * x[..., half:]
    z = z * np.exp(1j * np.asarray(pos, np.float64)[..., None] * freq)
    return np.concatenate([z.real, z.imag], axis=-1)


# ---------------------------------------------------------------- RoPE (P8)
def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 5, 16))
    pos = rng.integers(0, 300000, size=(3, 5))
    np.testing.assert_allclose(O.rope(x, pos, 5e5), _complex_rope(x, pos, 5e5), atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((2, 64))
    # identity at position 0
    np.testing.assert_allclose(O.rope(q, 0, 1e4), q, atol=0)
    # norm preserved
    for p in (1, 7, 1023, 262143):
        assert abs(np.linalg.norm(O.rope(q, p, 1e4)) - np.linalg.norm(q)) < 1e-12
    # inner product depends only on the position difference
    a = O.rope(q, 100, 1e4) @ O.rope(k, 37, 1e4)
    b = O.rope(q, 1063, 1e4) @ O.rope(k, 1000, 1e4)
    assert abs(a - b) < 1e-9
    # rotate-half pairing: a vector on dimension 0 only moves into dimension d/2
    e0 = np.zeros(64)
    e0[0] = 1.0
    r = O.rope(e0, 1, 1e4)
    assert abs(r[0] - math.cos(1.0)) < 1e-15 and abs(r[32] - math.sin(1.0)) < 1e-15
    assert np.count_nonzero(np.abs(r) > 1e-15) == 2


# ------------------------------------------------------- chunk stats (P9)
def test_chunk_mean_closed_form_and_constant_chunk():
    rng = np.random.default_rng(3)
    c, d, n = 8, 16, 5
    centers = rng.standard_normal((n, d))
    dev = rng.standard_normal((n, c, d))
    dev -= dev.mean(axis=1, keepdims=True)          # deviations sum to zero
    k = (centers[:, None, :] + 0.1 * dev).reshape(n * c, d)
    k[2 * c:3 * c] = centers[2]                    # chunk 2 is constant
    L = O.chunk_landmarks(k, c, n)
    np.testing.assert_allclose(L, centers, atol=1e-14)
    m = O.chunk_min_cosine(k, L, c)
    assert abs(m[2] - 1.0) < 1e-14
    assert np.all(m <= 1.0 + 1e-15) and np.all(m >= -1.0 - 1e-15)


def test_chunk_min_cos_anti_aligned_token():
    # chunk of 4 copies of v and one -v among 8 tokens -> mean (6v)/8, min cos = -1
    v = np.arange(1.0, 9.0)
    k = np.tile(v, (8, 1))
    k[5] = -v
    m = O.chunk_min_cosine(k, O.chunk_landmarks(k, 8, 1), 8)
    assert abs(m[0] + 1.0) < 1e-14


# ---------------------------------------------------------- top-k (P7)
def _is_valid_topk(scores, chosen, k):
    chosen = list(chosen)
    if len(chosen) != k or len(set(chosen)) != k or chosen != sorted(chosen):
        return False
    rest = [j for j in range(len(scores)) if j not in chosen]
    for i in chosen:
        for j in rest:
            if scores[i] < scores[j] or (scores[i] == scores[j] and i > j):
                return False
    return True


@pytest.mark.parametrize("seed", range(6))
def test_argtopk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    n, k = 9, 4
    scores = rng.integers(0, 4, size=n).astype(float)     # many planted ties
    got = O.argtopk(scores, k)
    assert _is_valid_topk(scores, got, k)
    # exhaustive: exactly one k-subset satisfies the definition
    valid = [s for s in itertools.combinations(range(n), k) if _is_valid_topk(scores, s, k)]
    assert valid == [tuple(got)]


def test_argtopk_respects_validity_mask():
    scores = np.array([5.0, 9.0, 1.0, 9.0, 3.0])
    valid = np.array([True, False, True, True, True])
    assert list(O.argtopk(scores, 2, valid=valid)) == [0, 3]


# ------------------------------------------------------ outliers (P4)
def test_planted_outlier_chunks_detected():
    rng = np.random.default_rng(4)
    b, h, d, c, w = 1, 2, 32, 8, 16
    n = 24
    s = n * c + w
    # smooth pre-RoPE keys: a slowly varying direction along the sequence
    base = rng.standard_normal((b, h, 1, d))
    drift = np.cumsum(0.01 * rng.standard_normal((b, h, s, d)), axis=2)
    k_pre = base + drift
    planted = [3, 11, 20]
    for j in planted:
        k_pre[:, :, j * c + 4] *= -1.0                    # anti-aligned token
    v = rng.standard_normal((b, h, s, d))
    st = O.prefill(k_pre, v, c=c, r=8, o=3, w=w, theta=1e4)
    for hi in range(h):
        assert sorted(st.outlier_ids[0, hi].tolist()) == planted


# ---------------------------------------------------------- SVD (P2, P3)
def test_svd_exact_low_rank_reconstruction():
    rng = np.random.default_rng(5)
    b, h, s, d, r = 2, 2, 96, 16, 6
    U = rng.standard_normal((b, s, r))
    W = rng.standard_normal((b, r, h * d))
    M = U @ W
    k_pre = M.reshape(b, s, h, d).transpose(0, 2, 1, 3)
    A, B, _ = O.svd_factors(k_pre, r)
    for bi in range(b):
        rec = A[bi] @ B[bi].transpose(1, 0, 2).reshape(r, h * d)
        assert np.linalg.norm(rec - M[bi]) / np.linalg.norm(M[bi]) < 1e-12


def test_svd_eckart_young_closed_form():
    rng = np.random.default_rng(6)
    s, h, d, r = 80, 2, 12, 5
    D = h * d
    Q1, _ = np.linalg.qr(rng.standard_normal((s, D)))
    Q2, _ = np.linalg.qr(rng.standard_normal((D, D)))
    sigma = np.sort(rng.uniform(0.1, 10.0, D))[::-1]
    M = (Q1 * sigma) @ Q2.T
    k_pre = M.reshape(1, s, h, d).transpose(0, 2, 1, 3)
    A, B, _ = O.svd_factors(k_pre, r)
    rec = A[0] @ B[0].transpose(1, 0, 2).reshape(r, D)
    err2 = np.linalg.norm(M - rec) ** 2
    assert abs(err2 - np.sum(sigma[r:] ** 2)) < 1e-9 * np.sum(sigma ** 2)


# ------------------------------------------------ subspace similarity (P5)
def test_subspace_similarity_closed_forms():
    rng = np.random.default_rng(7)
    n, r = 20, 4
    Q, _ = np.linalg.qr(rng.standard_normal((n, n)))
    V1 = Q[:, :r]
    assert abs(O.subspace_similarity(V1, V1, r) - 1.0) < 1e-12
    assert abs(O.subspace_similarity(V1, Q[:, r:2 * r], r)) < 1e-12
    # principal angles theta_i between span(V1) and span(V2): D = sum cos^2 / r
    th = np.array([0.1, 0.5, 1.0, 1.4])
    V2 = Q[:, :r] * np.cos(th) + Q[:, r:2 * r] * np.sin(th)
    assert abs(O.subspace_similarity(V1, V2, r) - np.sum(np.cos(th) ** 2) / r) < 1e-12


def test_subspace_similarity_random_expectation():
    rng = np.random.default_rng(8)
    n, r = 64, 10
    vals = []
    for _ in range(200):
        V1, _ = np.linalg.qr(rng.standard_normal((n, r)))
        V2, _ = np.linalg.qr(rng.standard_normal((n, r)))
        vals.append(O.subspace_similarity(V1, V2, r))
    assert abs(np.mean(vals) - r / n) < 0.01          # E[D] = r / n


# ---------------------------------------------- equivalent bandwidth (P6)
def test_equivalent_bandwidth_worked_example():
    g = read_golden("equivalent_bandwidth_example.txt")
    bw = O.equivalent_bandwidth(g["S"], g["C"], g["K"], g["O"], 0.6, g["B_GPU_GBps"],
                                g["B_PCIe_GBps"])
    assert abs(bw / 1000.0 - g["printed_TBps"]) <= g["printed_tolerance"]
    assert abs(bw / g["B_GPU_GBps"] - g["printed_ratio_to_hbm"]) <= g["printed_tolerance"]


def test_equivalent_bandwidth_limits():
    # all hits: the PCIe term vanishes -> 2 S B / (S/C + 2 (K+O) C)
    S, C, K, Oc, B = 131072, 8, 256, 48, 2000.0
    assert abs(O.equivalent_bandwidth(S, C, K, Oc, 1.0, B, 31.5) - 2 * S * B / (S / C + 2 * (K + Oc) * C)) < 1e-9
    # C = 1 and K = S/2 with every chunk a hit: S landmark reads plus 2K
    # token reads equal the 2S reads of dense attention, so B~ = B_GPU
    assert abs(O.equivalent_bandwidth(1000, 1.0, 500, 0, 1.0, B, 31.5) - B) < 1e-9
    # misses only add time: B~ falls as alpha falls
    assert O.equivalent_bandwidth(S, C, K, Oc, 0.2, B, 31.5) < O.equivalent_bandwidth(S, C, K, Oc, 0.6, B, 31.5)


def test_key_parameters_budget():
    g = read_golden("key_parameters.txt")
    from sparse_rank_kv_gb300.synth import CONFIGS
    for name in ("llama_b1_s32k", "llama_b8_s128k", "llama_b48_s60k"):
        cfg = CONFIGS[name]
        assert cfg.c == g["chunk_size"] and cfg.r == g["svd_rank"] and cfg.o == g["outlier_chunks"]
        assert abs(100.0 * cfg.k * cfg.c / cfg.s - g["sparse_budget_percent"]) < 0.01


# ------------------------------------------- decode: dense equivalence (P1)
def _dense_reference(k_pre, v, q_steps, knew, vnew, theta):
    """Textbook GQA decode over every token via torch SDPA in float64."""
    b, h, s, d = k_pre.shape
    pos = np.arange(s)
    K = _complex_rope(k_pre, pos, theta)
    V = np.asarray(v, np.float64)
    outs = []
    for t, q in enumerate(q_steps):
        K = np.concatenate([K, knew[t][:, :, None]], axis=2)
        V = np.concatenate([V, vnew[t][:, :, None]], axis=2)
        G = q.shape[1] // h
        Kt = torch.from_numpy(K).repeat_interleave(G, dim=1)
        Vt = torch.from_numpy(V).repeat_interleave(G, dim=1)
        qt = torch.from_numpy(np.asarray(q, np.float64))[:, :, None, :]
        o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt)
        outs.append(o[:, :, 0].numpy())
    return outs


@pytest.mark.parametrize("reduce", ["max", "sum"])
def test_decode_equals_dense_attention_when_everything_is_kept(reduce):
    rng = np.random.default_rng(9)
    b, h_q, h, d, c, w, o = 2, 4, 2, 16, 4, 8, 3
    n = 10
    s = n * c + w
    r = h * d                                        # full rank
    k_pre = rng.standard_normal((b, h, s, d))
    v = rng.standard_normal((b, h, s, d))
    st = O.prefill(k_pre, v, c=c, r=r, o=o, w=w, theta=1e4)
    dec = O.OracleDecoder(st, h_q=h_q, k=n - o, group_reduce=reduce)
    T = 3
    qs = [rng.standard_normal((b, h_q, d)) * 2 for _ in range(T)]
    kn = [rng.standard_normal((b, h, d)) for _ in range(T)]
    vn = [rng.standard_normal((b, h, d)) for _ in range(T)]
    ref = _dense_reference(k_pre, v, qs, kn, vn, 1e4)
    for t in range(T):
        res = dec.step(qs[t], kn[t], vn[t])
        np.testing.assert_allclose(res.out, ref[t], atol=1e-10)
        # every step keeps every candidate: full hits after step 0
        assert np.all(res.hits == (0 if t == 0 else n - o))


def test_decode_selection_single_head_group_is_topk_of_dot_products():
    # G = 1: S2 = softmax(P) is monotone in q.L, so the selection is the top-k
    # of the raw dot products over the candidates.
    rng = np.random.default_rng(10)
    b, h, d, c, w, o, k = 1, 3, 8, 2, 4, 2, 5
    n = 16
    s = n * c + w
    k_pre = rng.standard_normal((b, h, s, d))
    st = O.prefill(k_pre, rng.standard_normal((b, h, s, d)), c=c, r=4, o=o, w=w, theta=1e4)
    dec = O.OracleDecoder(st, h_q=h, k=k)
    q = rng.standard_normal((b, h, d))
    res = dec.step(q)
    for hi in range(h):
        dots = {j: float(sum(q[0, hi, e] * st.L[0, hi, j, e] for e in range(d)))
                for j in range(n) if j not in st.outlier_ids[0, hi]}
        best = sorted(sorted(dots, key=lambda j: -dots[j])[:k])
        assert res.sel[0, hi].tolist() == best


def test_decode_group_readings_agree_when_queries_coincide():
    rng = np.random.default_rng(11)
    b, h_q, h, d, c, w, o, k = 1, 4, 1, 8, 2, 4, 2, 4
    n = 12
    s = n * c + w
    st = O.prefill(rng.standard_normal((b, h, s, d)), rng.standard_normal((b, h, s, d)),
                   c=c, r=4, o=o, w=w, theta=1e4)
    q1 = rng.standard_normal((b, 1, d))
    q = np.repeat(q1, h_q, axis=1)
    sel_max = O.OracleDecoder(st, h_q=h_q, k=k, group_reduce="max").step(q).sel
    sel_sum = O.OracleDecoder(st, h_q=h_q, k=k, group_reduce="sum").step(q).sel
    sel_one = O.OracleDecoder(st, h_q=1, k=k).step(q1).sel
    assert sel_max.tolist() == sel_sum.tolist() == sel_one.tolist()


def test_hit_count_brute_force():
    rng = np.random.default_rng(12)
    for _ in range(20):
        a = np.sort(rng.choice(50, 10, replace=False))
        bb = np.sort(rng.choice(50, 10, replace=False))
        assert O.hit_count(a, bb) == len(set(a.tolist()) & set(bb.tolist()))


def test_rebuilt_keys_equal_post_rope_keys_at_full_rank():
    rng = np.random.default_rng(13)
    b, h, d, c, w, o, k = 1, 2, 8, 2, 4, 1, 3
    n = 8
    s = n * c + w
    k_pre = rng.standard_normal((b, h, s, d))
    st = O.prefill(k_pre, rng.standard_normal((b, h, s, d)), c=c, r=h * d, o=o, w=w, theta=1e4)
    res = O.OracleDecoder(st, h_q=h, k=k).step(rng.standard_normal((b, h, d)))
    K_rope = _complex_rope(k_pre, np.arange(s), 1e4)
    for hi in range(h):
        rows = (res.sel[0, hi][:, None] * c + np.arange(c)).ravel()
        np.testing.assert_allclose(res.K_sparse[0, hi], K_rope[0, hi, rows], atol=1e-10)


# ------------------------------------------------ attention (Alg. 2 step 4)
def test_attention_equals_library_sdpa():
    # an independent implementation: torch's scaled dot-product attention in
    # float64, each query of the group against the shared keys and values
    rng = np.random.default_rng(14)
    q = rng.standard_normal((3, 4, 16)) * 3
    K = rng.standard_normal((3, 37, 16))
    V = rng.standard_normal((3, 37, 16))
    got = O.attention(q, K, V)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(K), torch.from_numpy(V)).numpy()
    np.testing.assert_allclose(got, ref, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(15)
    q = rng.standard_normal((2, 8))
    V = rng.standard_normal((5, 8))
    # one token: the output is its value, whatever the query
    np.testing.assert_allclose(O.attention(q, rng.standard_normal((1, 8)), V[:1]), np.tile(V[:1], (2, 1)),
                               atol=1e-15)
    # equal keys: uniform weights, the output is the mean value
    K = np.tile(rng.standard_normal((1, 8)), (5, 1))
    np.testing.assert_allclose(O.attention(q, K, V), np.tile(V.mean(0), (2, 1)), atol=1e-14)
    # a key with logit 8 ln 2 above the others (scale 1/sqrt(d)): weight 256 : 1
    qv = np.zeros((1, 4))
    qv[0, 0] = 2.0
    K = np.zeros((3, 4))
    K[1, 0] = 8 * np.log(2.0)
    V = np.eye(3, 4)
    np.testing.assert_allclose(O.attention(qv, K, V)[0, :3], np.array([1, 256, 1]) / 258.0, atol=1e-14)


def test_attention_ignores_token_order():
    rng = np.random.default_rng(16)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((50, 16))
    V = rng.standard_normal((50, 16))
    perm = rng.permutation(50)
    np.testing.assert_allclose(O.attention(q, K, V), O.attention(q, K[perm], V[perm]), atol=1e-13)


# ------------------------------------------- element types (reading R11)
def test_store_bf16_matches_library_conversion_and_rounds_ties_to_even():
    rng = np.random.default_rng(17)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.store(x, "bf16"), ref)
    # bf16 keeps 8 significant bits: 1 + k 2^-7 is exact; halfway cases go to even k
    assert O.store(1.0 + 2.0 ** -7, "bf16") == 1.0 + 2.0 ** -7
    assert O.store(1.0 + 2.0 ** -8, "bf16") == 1.0
    assert O.store(1.0 + 3 * 2.0 ** -8, "bf16") == 1.0 + 2.0 ** -6
    assert O.store(-(1.0 + 3 * 2.0 ** -8), "bf16") == -(1.0 + 2.0 ** -6)
    assert O.store(1.0 + 2.0 ** -30, "f32") == 1.0 and O.store(1.0 + 2.0 ** -30, "f64") == 1.0 + 2.0 ** -30


def test_rebuilt_keys_are_stored_in_the_key_type():
    rng = np.random.default_rng(18)
    b, h, d, c, w, o, k = 1, 2, 8, 2, 4, 1, 3
    n = 8
    s = n * c + w
    st = O.prefill(rng.standard_normal((b, h, s, d)), rng.standard_normal((b, h, s, d)), c=c, r=4, o=o, w=w,
                   theta=1e4)
    q = rng.standard_normal((b, h, d))
    exact = O.OracleDecoder(st, h_q=h, k=k).step(q)
    rounded = O.OracleDecoder(st, h_q=h, k=k, key_dtype="bf16").step(q)
    np.testing.assert_array_equal(rounded.K_sparse, O.store(exact.K_sparse, "bf16"))
    assert np.array_equal(rounded.sel, exact.sel)
    assert np.abs(rounded.out - exact.out).max() < 0.05 * np.abs(exact.out).max()

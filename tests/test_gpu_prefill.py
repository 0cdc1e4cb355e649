"""GPU prefill (Algorithm 1) against the CPU oracle, through the C ABI.

Rows covered: a1 RoPE (through L and the gathered keys), a2 landmarks,
a3 minimum in-chunk cosine, a4 outlier ArgTopK (tie-aware) and the gathered
outlier keys/values, a5 the rank-r factors (exact for an exactly low-rank
matrix, Eckart-Young optimal otherwise), a6 the pinned host copy of V and
the local window.  An end-to-end case checks prefill + decode against dense
attention when nothing is dropped (full rank, every chunk selected).
"""
import numpy as np
import pytest
import torch

from helpers import TOL, check_selection, ey_bound, head_errors, np64
from oracle import shadowkv_oracle as O
from sparse_rank_kv_gb300 import binding, build, synth
from sparse_rank_kv_gb300.synth import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.lib()


SMALL = CONFIGS["llama_b1_s32k"].with_(
    name="small_prefill", b=2, h_q=8, h_kv=2, d=128, s=4000 + 64, c=8, r=48, k=30, o=6, w=64,
    theta=5e5, dtype="bf16", steps=3, rank_true=32, n_spike=4, seed=51)


def gpu_prefill(cfg, inp, v_on_host=False, **kw):
    p = binding.make_params(cfg, **kw)
    v = inp["v"].cpu() if v_on_host else inp["v"]
    return binding.prefill(p, inp["k_pre"], v)


def shapes(cfg):
    return cfg.b, cfg.h_kv, cfg.s, cfg.d, cfg.n


def check_stats_and_gathers(cfg, ctx, inp, ost):
    b, h, s, d, n = shapes(cfg)
    c, o, w = cfg.c, cfg.o, cfg.w
    E = 1e-5 if cfg.dtype == "f32" else 2.0 ** -8
    L = np64(ctx.export("L").view(b, h, n, d))
    assert np.all(np.abs(L - ost.L) <= E * np.abs(ost.L) + 1e-5 * np.abs(ost.L).max()), "landmarks"
    m = ctx.export("MIN_COS").view(b, h, n).numpy().astype(np.float64)
    assert np.abs(m - ost.min_cos).max() <= 2e-5, "min cosine"
    ids = ctx.export("OUTLIER_IDS").view(b, h, o).numpy()
    check_selection(ids, -ost.min_cos, o, what="outliers")
    # gathered rows follow the GPU's own outlier choice
    K_rope = O.rope(np64(inp["k_pre"]), np.arange(s), cfg.theta)
    V = np64(inp["v"])
    rows = (ids[..., None].astype(np.int64) * c + np.arange(c)).reshape(b, h, o * c)
    kout = np64(ctx.export("K_OUT").view(b, h, o * c, d))
    vout = np64(ctx.export("V_OUT").view(b, h, o * c, d))
    kref = np.take_along_axis(K_rope, rows[..., None], axis=2)
    vref = np.take_along_axis(V, rows[..., None], axis=2)
    assert np.all(np.abs(kout - kref) <= E * np.abs(kref) + 1e-6 * np.abs(kref).max()), "outlier keys"
    assert np.array_equal(vout, vref), "outlier values"
    cap = w + cfg.max_new
    kloc = np64(ctx.export("K_LOC").view(b, h, cap, d))[:, :, :w]
    vloc = np64(ctx.export("V_LOC").view(b, h, cap, d))[:, :, :w]
    kr = K_rope[:, :, n * c:]
    assert np.all(np.abs(kloc - kr) <= E * np.abs(kr) + 1e-6 * np.abs(kr).max()), "local keys"
    assert np.array_equal(vloc, V[:, :, n * c:]), "local values"
    vcpu = np64(ctx.export("V_CPU").view(b, h, s, d))
    assert np.array_equal(vcpu, V), "pinned host copy of V"


def factor_errors(cfg, ctx, inp):
    """Per sequence: (err_basis^2, err_stored^2, opt^2, |M|^2, sigma^2) where err_basis is
    |M - M X^T X| for the GPU's fp32 orthonormal basis X (the SVD's own
    quality), err_stored is |M - A B| for the stored factors, and opt^2 is the
    Eckart-Young optimum sum_{i>r} sigma_i^2."""
    b, h, s, d, _ = shapes(cfg)
    r, D = cfg.r, h * d
    A = ctx.export("A").view(b, s, r).to(torch.float64)
    Bt = ctx.export("BT").view(b, h, d, r).to(torch.float64)
    X = ctx.export("SVD_BASIS").view(b, r, D).to(torch.float64)
    out = []
    for bi in range(b):
        M = inp["k_pre"][bi].to("cpu", torch.float64).permute(1, 0, 2).reshape(s, D)
        B = Bt[bi].permute(2, 0, 1).reshape(r, D)
        err_basis = float(((M - (M @ X[bi].T) @ X[bi]) ** 2).sum())
        err_stored = float(((M - A[bi] @ B) ** 2).sum())
        sig = np.linalg.svd(M.numpy(), compute_uv=False)
        out.append((err_basis, err_stored, float(np.sum(sig[r:] ** 2)), float(np.sum(sig ** 2)), sig ** 2))
    return out


def check_factors(cfg, ctx, inp, bound=None):
    """Eckart-Young on the fp32 basis; the stored factors may add at most the
    rounding of A and B to the storage type: |M - A B| <= |M - M X^T X| + 3u|M|
    (u = 2^-8 for bf16, 2^-24 for fp32)."""
    u = 2.0 ** -8 if cfg.dtype == "bf16" else 2.0 ** -24
    for eb, es, opt, tot, lam in factor_errors(cfg, ctx, inp):
        bd = ey_bound(cfg, lam) if bound is None else bound
        assert eb <= bd * opt + 1e-9 * tot, ("basis", eb / opt, bd)
        assert np.sqrt(es) <= np.sqrt(eb) + 3 * u * np.sqrt(tot), ("stored", es / opt)


def test_tiny_fp32_prefill_matches_oracle():
    cfg = CONFIGS["tiny_f32_s1k"]
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = gpu_prefill(cfg, inp)
    ost = O.prefill(np64(inp["k_pre"]), np64(inp["v"]), cfg.c, cfg.r, cfg.o, cfg.w, cfg.theta)
    check_stats_and_gathers(cfg, ctx, inp, ost)
    check_factors(cfg, ctx, inp)


def test_bf16_prefill_matches_oracle_and_detects_spikes():
    cfg = SMALL
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = gpu_prefill(cfg, inp)
    ost = O.prefill(np64(inp["k_pre"]), np64(inp["v"]), cfg.c, cfg.r, cfg.o, cfg.w, cfg.theta)
    check_stats_and_gathers(cfg, ctx, inp, ost)
    ids = ctx.export("OUTLIER_IDS").view(cfg.b, cfg.h_kv, cfg.o).numpy()
    for j in inp["spike"].tolist():
        assert np.all((ids == j).any(axis=-1)), f"planted spike chunk {j} not an outlier"
    check_factors(cfg, ctx, inp)


def test_spectral_gap_factors_are_eckart_young_optimal():
    cfg = SMALL.with_(rank_true=48, seed=56)          # true rank = r, noise 0.01
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = gpu_prefill(cfg, inp)
    check_factors(cfg, ctx, inp, bound=1.01)


def test_values_from_host_memory_prefill():
    cfg = SMALL.with_(seed=52)
    inp = synth.make_inputs(cfg, device="cuda")
    a = gpu_prefill(cfg, inp)
    bctx = gpu_prefill(cfg, inp, v_on_host=True)
    for f in ("L", "OUTLIER_IDS", "K_OUT", "V_OUT", "K_LOC", "V_LOC", "V_CPU", "A", "BT"):
        assert torch.equal(a.export(f), bctx.export(f)), f


def test_exact_low_rank_is_reconstructed_to_fp32_roundoff():
    cfg = CONFIGS["tiny_f32_s1k"].with_(r=24, rank_true=24, seed=53)
    inp = synth.make_inputs(cfg, device="cuda", noise=0.0)
    ctx = gpu_prefill(cfg, inp)
    for eb, es, _, tot, _ in factor_errors(cfg, ctx, inp):
        assert np.sqrt(es / tot) <= 1e-5 and np.sqrt(eb / tot) <= 1e-5


def test_basis_is_orthonormal_and_matches_oracle_subspace():
    cfg = SMALL.with_(r=32, rank_true=32, seed=54)
    inp = synth.make_inputs(cfg, device="cuda", noise=0.0)
    ctx = gpu_prefill(cfg, inp)
    b, h, s, d, _ = shapes(cfg)
    D = h * d
    X = ctx.export("SVD_BASIS").view(b, cfg.r, D).numpy().astype(np.float64)
    for bi in range(b):
        assert np.abs(X[bi] @ X[bi].T - np.eye(cfg.r)).max() < 1e-5
        M = np64(inp["k_pre"][bi]).transpose(1, 0, 2).reshape(s, D)
        Vt = np.linalg.svd(M, full_matrices=False)[2][:cfg.r]
        assert O.subspace_similarity(X[bi].T, Vt.T, cfg.r) > 1 - 1e-6


def test_full_rank_prefill_and_decode_equal_dense_attention():
    """Nothing dropped (r = h_kv d, k = n - o): the whole GPU path must equal
    textbook GQA attention over every prompt and appended token."""
    cfg = CONFIGS["tiny_f32_s1k"].with_(r=128, k=124 - 4, seed=55)
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = gpu_prefill(cfg, inp)
    b, h, s, d = cfg.b, cfg.h_kv, cfg.s, cfg.d
    K = torch.from_numpy(O.rope(np64(inp["k_pre"]), np.arange(s), cfg.theta))
    V = torch.from_numpy(np64(inp["v"]))
    G = cfg.h_q // h
    for t in range(cfg.steps):
        q, kn, vn = inp["q"][t], inp["k_new"][t], inp["v_new"][t]
        out = torch.empty(b, cfg.h_q, d, device="cuda")
        ctx.decode_step(q, kn, vn, out)
        K = torch.cat([K, torch.from_numpy(np64(kn))[:, :, None]], dim=2)
        V = torch.cat([V, torch.from_numpy(np64(vn))[:, :, None]], dim=2)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(np64(q))[:, :, None], K.repeat_interleave(G, 1),
            V.repeat_interleave(G, 1))[:, :, 0].numpy()
        torch.cuda.synchronize()
        assert head_errors(np64(out), ref).max() <= TOL["f32"]
    ctx.check()


def test_full_size_32k_prefill_eckart_young_and_stats():
    cfg = CONFIGS["llama_b1_s32k"]
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = gpu_prefill(cfg, inp)
    b, h, s, d, n = shapes(cfg)
    # stats and outliers of the full prefill against the oracle's statistics
    K_rope = O.rope(np64(inp["k_pre"]), np.arange(s), cfg.theta)
    Lref = O.chunk_landmarks(K_rope, cfg.c, n)
    mref = O.chunk_min_cosine(K_rope, Lref, cfg.c)
    L = np64(ctx.export("L").view(b, h, n, d))
    assert np.all(np.abs(L - Lref) <= 2.0 ** -8 * np.abs(Lref) + 1e-5 * np.abs(Lref).max())
    m = ctx.export("MIN_COS").view(b, h, n).numpy().astype(np.float64)
    assert np.abs(m - mref).max() <= 2e-5
    check_selection(ctx.export("OUTLIER_IDS").view(b, h, cfg.o).numpy(), -mref, cfg.o,
                    what="outliers")
    check_factors(cfg, ctx, inp)


@pytest.mark.parametrize("shape", [
    dict(r=256, rank_true=200, seed=57),            # r = h_kv d: Cholesky of the fp64 pass in global memory, 2-stage factor
    dict(d=64, theta=1e4, r=48, seed=58),           # 64-dim heads: one 64-column block per head in the transpose and factor
    dict(r=16, rank_true=12, seed=59),              # the smallest rank the tensor-core path takes
], ids=["r256", "d64", "r16"])
def test_tensor_core_svd_shapes(shape):
    """Shapes at the edges of the tensor-core SVD: landmarks and outliers
    against the oracle, the factors against the Eckart-Young bars."""
    cfg = SMALL.with_(**shape)
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = gpu_prefill(cfg, inp)
    assert ctx.layout()["tc_rebuild"] == (cfg.r % 16 == 0)
    ost = O.prefill(np64(inp["k_pre"]), np64(inp["v"]), cfg.c, cfg.r, cfg.o, cfg.w, cfg.theta)
    check_stats_and_gathers(cfg, ctx, inp, ost)
    check_factors(cfg, ctx, inp)
    ctx.check()

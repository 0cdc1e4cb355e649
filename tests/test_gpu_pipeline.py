"""The whole path as the benchmark runs it, against the CPU oracle.

Algorithm 1 runs on the GPU (shadowkv_prefill on walk-structured keys), the
library's compressed state is exported at storage precision (A, B, L, the
outliers, the local window, the pinned host copy of V) and handed to the
oracle, and then every decode step of the GPU -- bf16, d = 128: K/V records,
tensor-core scores, rebuild and attention, the value fetch inside the
rebuild launch -- is checked against the oracle's Algorithm 2 on that state:
  - the selected chunks by the tie-aware index rule,
  - the cache hits exactly,
  - the output within the bf16 bound (per head, relative to its largest value).
Run this way a decode error cannot hide inside a difference of SVD bases.

The prefill itself is checked on the same runs at the full sizes of the
128K and 256K workloads, one sequence recomputed by the oracle: landmarks and
minimum cosines within storage rounding, outliers by the index rule, and the
rank-r factors against the Eckart-Young optimum (from the Gram matrix, so
the oracle never takes an s x h_kv d SVD).
"""
import numpy as np
import pytest
import torch

from helpers import TOL, check_selection, exported_state, ey_bound, gram_factor_errors, head_errors, np64
from oracle import shadowkv_oracle as O
from sparse_rank_kv_gb300 import binding, build, synth
from sparse_rank_kv_gb300.synth import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.lib()


def decode_against_oracle(cfg, ctx, inp, steps, bsel=None, rows=False, report_exact=False):
    """Decodes `steps` steps of inp on the GPU and checks each against the
    oracle run on the context's exported state (one sequence if bsel), with
    the rebuilt keys in the workload's element type (reading R11).  With
    report_exact, also prints the error against exact (float64) rebuilt keys."""
    b, h, hq, d, k, c = cfg.b, cfg.h_kv, cfg.h_q, cfg.d, cfg.k, cfg.c
    sl = slice(None) if bsel is None else slice(bsel, bsel + 1)
    state = exported_state(ctx, cfg, bsel)
    dec = O.OracleDecoder(state, h_q=hq, k=k, key_dtype=cfg.dtype)
    exact = O.OracleDecoder(state, h_q=hq, k=k) if report_exact else None
    dt = synth.torch_dtype(cfg.dtype)
    worst, alpha = 0.0, []
    for t in range(steps):
        q, kn, vn = (inp[x][t].contiguous() for x in ("q", "k_new", "v_new"))
        out = torch.empty(b, hq, d, dtype=dt, device="cuda")
        ctx.decode_step(q, kn, vn, out)
        torch.cuda.synchronize()
        sel = ctx.export("SEL").view(b, h, k).numpy()[sl]
        qn = np64(q[sl])
        _, S2, _ = dec.scores(qn)
        check_selection(sel, S2, k, what=f"step {t} selection")
        res = dec.step(qn, np64(kn[sl]), np64(vn[sl]), force_sel=sel)
        err = head_errors(np64(out[sl]), res.out)
        worst = max(worst, float(err.max()))
        assert err.max() <= TOL[cfg.dtype], f"step {t}: output error {err.max():.3g}"
        if exact is not None:
            ex = exact.step(qn, np64(kn[sl]), np64(vn[sl]), force_sel=sel)
            print(f"step {t}: output error {err.max():.4f} (rebuilt keys in {cfg.dtype}), "
                  f"{head_errors(np64(out[sl]), ex.out).max():.4f} against exact rebuilt keys")
        hits = ctx.export("HITS").view(b, h).numpy()[sl]
        assert np.array_equal(hits, res.hits), f"step {t}: hits {hits} vs {res.hits}"
        if t:
            alpha.append(hits.mean() / k)
        if rows:
            ks = np64(ctx.export("K_SPARSE").view(b, h, k * c, d)[sl])
            assert np.abs(ks - res.K_sparse).max() <= 8e-3 * np.abs(res.K_sparse).max(), f"step {t}: rebuilt keys"
            lg = ctx.export("LOGITS").view(b, hq, -1).numpy()[sl].astype(np.float64)
            m = ~np.isnan(res.P)
            lerr = np.abs(lg[m] - res.P[m]).max() / np.abs(res.P[m]).max()
            if report_exact:
                print(f"step {t}: logits error {lerr:.2e} of the largest logit")
            # 128 exact bf16 products summed in fp32 in the tensor cores' order:
            # worst case d * 2^-24 = 7.6e-6 of sum |q_i L_i|; 1.5-2.3e-7 measured.
            assert lerr <= 1e-5, f"step {t}: logits {lerr:.3g}"
    ctx.check()
    return worst, (float(np.mean(alpha)) if alpha else None)


def check_prefill_sequence(cfg, ctx, inp, bi):
    """Algorithm 1 on sequence bi against the oracle: L and the minimum cosine
    within storage rounding, outliers by the index rule, the factors against
    the Eckart-Young optimum.  Returns (err_basis^2/opt^2, err_stored^2/opt^2, X)."""
    b, h, s, d, n, r = cfg.b, cfg.h_kv, cfg.s, cfg.d, cfg.n, cfg.r
    D = h * d
    K_rope = O.rope(np64(inp["k_pre"][bi]), np.arange(s), cfg.theta)           # (h, s, d)
    Lref = O.chunk_landmarks(K_rope, cfg.c, n)
    mref = O.chunk_min_cosine(K_rope, Lref, cfg.c)
    del K_rope
    L = np64(ctx.export("L").view(b, h, n, d)[bi])
    assert np.all(np.abs(L - Lref) <= 2.0 ** -8 * np.abs(Lref) + 1e-5 * np.abs(Lref).max()), "landmarks"
    m = ctx.export("MIN_COS").view(b, h, n)[bi].numpy().astype(np.float64)
    assert np.abs(m - mref).max() <= 2e-5, f"min cosine {np.abs(m - mref).max():.3g}"
    check_selection(ctx.export("OUTLIER_IDS").view(b, h, cfg.o)[bi].numpy(), -mref, cfg.o, what="outliers")
    M = inp["k_pre"][bi].to("cpu", torch.float64).permute(1, 0, 2).reshape(s, D)
    X = ctx.export("SVD_BASIS").view(b, r, D)[bi].to(torch.float64)
    A = ctx.export("A").view(b, s, r)[bi].to(torch.float64)
    B = ctx.export("BT").view(b, h, d, r)[bi].to(torch.float64).permute(2, 0, 1).reshape(r, D)
    eb, es, opt, tot, lam = gram_factor_errors(M, X, A, B, r)
    bound = ey_bound(cfg, lam)
    u = 2.0 ** -8
    assert eb <= bound * opt + 1e-9 * tot, ("basis", eb / opt, bound)
    assert np.sqrt(es) <= np.sqrt(eb) + 3 * u * np.sqrt(tot), ("stored", es / opt)
    return eb / opt, es / opt, X


def test_prefill_then_decode_32k():
    cfg = CONFIGS["llama_b1_s32k"]
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = binding.prefill(binding.make_params(cfg), inp["k_pre"], inp["v"])
    worst, alpha = decode_against_oracle(cfg, ctx, inp, cfg.steps, rows=True, report_exact=True)
    assert worst <= TOL["bf16"] and alpha is not None


def test_prefill_then_decode_128k_batch8_sampled_sequence():
    """The benchmark's workload (batch 8, 128K) in its launch configuration:
    the GPU prefills and decodes all 8 sequences; the oracle recomputes
    sequence 5 of the prefill and of 6 decode steps."""
    cfg = CONFIGS["llama_b8_s128k"].with_(steps=6)
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = binding.prefill(binding.make_params(cfg), inp["k_pre"], inp["v"])
    check_prefill_sequence(cfg, ctx, inp, 5)
    decode_against_oracle(cfg, ctx, inp, cfg.steps, bsel=5)


def test_prefill_256k_rank_above_true_rank_then_decode():
    """Algorithm 1 end to end at 256K, batch 2, rank 160 over keys of true
    rank 128 plus noise (32 of the kept directions lie in the noise floor),
    then decode steps with k = 512 on the exported state.  Also prints the
    subspace similarity <H1, H2> / r of the two sequences' bases."""
    cfg = CONFIGS["llama_b2_s256k"].with_(steps=5)
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = binding.prefill(binding.make_params(cfg), inp["k_pre"], inp["v"])
    rb, rs, X1 = check_prefill_sequence(cfg, ctx, inp, 1)
    X0 = ctx.export("SVD_BASIS").view(cfg.b, cfg.r, cfg.h_kv * cfg.d)[0].to(torch.float64)
    D12 = O.subspace_similarity(X0.T.numpy(), X1.T.numpy(), cfg.r)
    print(f"256K: err^2/opt^2 basis {rb:.5f} stored {rs:.5f}; <H1,H2>/r = {D12:.4f}")
    assert 0.0 <= D12 <= 1.0
    decode_against_oracle(cfg, ctx, inp, cfg.steps, bsel=0)


@pytest.mark.parametrize("c,k", [(32, 16), (16, 30)])
def test_prefill_then_decode_other_chunk_sizes(c, k):
    """Chunks of 32 and 16 tokens (K/V records of 4 and 2 groups per chunk),
    every sequence of a batch of 2 recomputed by the oracle."""
    cfg = CONFIGS["llama_b1_s32k"].with_(name=f"c{c}", b=2, s=16384 + 64, c=c, k=k, o=6, steps=6,
                                         seed=80 + c)
    inp = synth.make_inputs(cfg, device="cuda")
    ctx = binding.prefill(binding.make_params(cfg), inp["k_pre"], inp["v"])
    for bi in range(cfg.b):
        check_prefill_sequence(cfg, ctx, inp, bi)
    decode_against_oracle(cfg, ctx, inp, cfg.steps, rows=True)

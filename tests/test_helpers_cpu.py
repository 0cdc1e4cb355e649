"""CPU checks of the test helpers that the GPU parity tests rely on."""
import numpy as np
import torch

from helpers import check_selection, gram_factor_errors


def test_gram_factor_errors_equal_direct_computation():
    rng = np.random.default_rng(21)
    s, D, r = 300, 24, 5
    M = torch.from_numpy(rng.standard_normal((s, 8)) @ rng.standard_normal((8, D))
                         + 0.05 * rng.standard_normal((s, D)))
    X = torch.from_numpy(np.linalg.qr(rng.standard_normal((D, r)))[0].T.copy())
    X = X + 1e-3 * torch.from_numpy(rng.standard_normal((r, D)))     # not quite orthonormal
    A = M @ X.T + 1e-3 * torch.from_numpy(rng.standard_normal((s, r)))
    B = X.clone()
    eb, es, opt, tot, lam = gram_factor_errors(M, X, A, B, r)
    sig = np.linalg.svd(M.numpy(), compute_uv=False)
    assert abs(eb - float(((M - M @ X.T @ X) ** 2).sum())) < 1e-9 * tot
    assert abs(es - float(((M - A @ B) ** 2).sum())) < 1e-9 * tot
    assert abs(opt - float(np.sum(sig[r:] ** 2))) < 1e-9 * tot
    assert abs(tot - float((M ** 2).sum())) < 1e-9 * tot


def test_check_selection_accepts_ties_and_rejects_wrong_sets():
    sc = np.array([5.0, 3.0, 3.0, 1.0, np.nan, 4.0])
    check_selection(np.array([0, 1, 5]), sc, 3)
    check_selection(np.array([0, 2, 5]), sc, 3)          # equal scores: either copy
    for bad in ([0, 3, 5], [0, 4, 5]):
        try:
            check_selection(np.array(bad), sc, 3)
        except AssertionError:
            continue
        raise AssertionError(f"{bad} accepted")


def test_ey_bound_is_the_random_noise_direction_error():
    """Noise floor: keeping the signal and m uniformly random noise directions
    has expected error sum(noise) - m mean(noise); the bound is that over opt."""
    from types import SimpleNamespace
    rng = np.random.default_rng(22)
    lam = np.concatenate([rng.uniform(1e4, 1e5, 6), rng.uniform(1.0, 2.0, 40)])
    cfg = SimpleNamespace(r=10, rank_true=6)
    from helpers import ey_bound
    noise = np.sort(lam)[:40]
    opt = np.sort(lam)[:36].sum()
    assert abs(ey_bound(cfg, lam) - (noise.sum() - 4 * noise.mean()) / opt * (1 + 1e-6)) < 1e-12
    # Monte Carlo: random 4-dimensional subspaces of the 40-dim noise space
    errs = []
    for _ in range(400):
        Q, _ = np.linalg.qr(rng.standard_normal((40, 4)))
        errs.append(noise.sum() - float(np.sum(Q ** 2 * noise[:, None])))
    assert abs(np.mean(errs) / opt - ey_bound(cfg, lam)) < 2e-3
    assert ey_bound(SimpleNamespace(r=6, rank_true=8), lam) == 1.01

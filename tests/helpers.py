"""Shared helpers of the GPU parity tests: conversions, the tie-aware index
rule and the per-head output error."""
from __future__ import annotations

import numpy as np
import torch

from oracle import shadowkv_oracle as O

# Output tolerances: max |gpu - oracle| over a query head's d outputs,
# divided by max |oracle| of that head.
TOL = {"f32": 1e-4, "bf16": 2e-2}
# Index rule: selections may differ from the oracle's only among entries whose
# score lies within this relative distance of the k-th score.
TIE_REL = 1e-3


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


def check_selection(sel, scores, k: int, rel: float = TIE_REL, what: str = "selection"):
    """sel: (..., k) ascending indices from the GPU; scores: (..., n) oracle scores
    with NaN at excluded entries.  Raises AssertionError when the GPU's set
    differs from the oracle's top-k outside the near-tie band."""
    sel = np.asarray(sel).reshape(-1, k)
    sc = np.asarray(scores, np.float64).reshape(sel.shape[0], -1)
    for i in range(sel.shape[0]):
        g = sel[i]
        assert np.all(np.diff(g) > 0), f"{what} row {i}: not strictly ascending: {g}"
        assert g.min() >= 0 and g.max() < sc.shape[1], f"{what} row {i}: index out of range"
        assert not np.any(np.isnan(sc[i, g])), f"{what} row {i}: picked an excluded entry"
        valid = ~np.isnan(sc[i])
        ref = O.argtopk(np.where(valid, sc[i], -np.inf), k, valid=valid)
        if set(g.tolist()) == set(ref.tolist()):
            continue
        vals = np.sort(sc[i][valid])[::-1]
        sk = vals[k - 1]
        band = rel * abs(sk)
        diff = set(g.tolist()) ^ set(ref.tolist())
        bad = [j for j in diff if abs(sc[i, j] - sk) > band]
        assert not bad, (f"{what} row {i}: chunks {bad} differ from the oracle outside the tie band "
                         f"(k-th score {sk:.6g}, band {band:.3g})")


def head_errors(out_gpu: np.ndarray, out_ref: np.ndarray) -> np.ndarray:
    """Per (b, head) max|delta| / max|ref| over the last axis."""
    num = np.abs(out_gpu - out_ref).max(axis=-1)
    den = np.abs(out_ref).max(axis=-1)
    return num / np.maximum(den, 1e-30)


def oracle_state(st: dict, cfg, bsel=None) -> O.OracleState:
    """OracleState from synth.make_state tensors (optionally one batch slice)."""
    sl = slice(None) if bsel is None else slice(bsel, bsel + 1)
    f = lambda key: np32(st[key][sl])
    return O.OracleState(
        c=cfg.c, theta=cfg.theta, A=f("A"), B=f("B"), L=f("L"),
        outlier_ids=st["outlier_ids"][sl].cpu().numpy().astype(np.int64),
        K_out=f("K_out"), V_out=f("V_out"), K_loc=f("K_loc"), V_loc=f("V_loc"), V_cpu=f("v"))


def exported_state(ctx, cfg, bsel=None) -> O.OracleState:
    """OracleState from the library's own exported state (storage precision):
    A, B (from B^T), L, outlier ids, outlier K/V, the w prompt rows of the
    local window and the pinned host copy of V; optionally one sequence."""
    b, h, s, d, n, r, c, o, w = cfg.b, cfg.h_kv, cfg.s, cfg.d, cfg.n, cfg.r, cfg.c, cfg.o, cfg.w
    cap = w + cfg.max_new
    sl = slice(None) if bsel is None else slice(bsel, bsel + 1)
    f = lambda name, *shape: np32(ctx.export(name).view(*shape)[sl])
    Bt = f("BT", b, h, d, r)
    return O.OracleState(
        c=c, theta=cfg.theta, A=f("A", b, s, r), B=np.ascontiguousarray(Bt.transpose(0, 1, 3, 2)),
        L=f("L", b, h, n, d),
        outlier_ids=ctx.export("OUTLIER_IDS").view(b, h, o)[sl].numpy().astype(np.int64),
        K_out=f("K_OUT", b, h, o * c, d), V_out=f("V_OUT", b, h, o * c, d),
        K_loc=f("K_LOC", b, h, cap, d)[:, :, :w], V_loc=f("V_LOC", b, h, cap, d)[:, :, :w],
        V_cpu=f("V_CPU", b, h, s, d))


def gram_factor_errors(M: torch.Tensor, X: torch.Tensor, A: torch.Tensor, B: torch.Tensor, r: int):
    """Squared errors of a rank-r factorisation of M (s x D), from the Gram
    matrix G = M^T M in float64 (no s x D SVD):
      err_basis^2  = |M - M X^T X|^2 = tr G - 2 tr(X G X^T) + tr(X X^T X G X^T)
      err_stored^2 = |M - A B|^2     = tr G - 2 <A^T M, B> + <A^T A, B B^T>
      opt^2        = sum_{i>r} sigma_i^2 = the sum of the D - r smallest eigenvalues of G
    X (r x D) is the basis, A (s x r) and B (r x D) the stored factors; all
    float64.  Returns (err_basis^2, err_stored^2, opt^2, |M|^2, eigenvalues of G)."""
    G = M.T @ M
    tot = float(torch.trace(G))
    lam = torch.linalg.eigvalsh(G)
    opt = float(lam[:-r].sum())
    XG = X @ G
    Q = XG @ X.T
    P = X @ X.T
    eb = tot - 2.0 * float(torch.trace(Q)) + float((P * Q.T).sum())
    AtM = A.T @ M
    es = tot - 2.0 * float((AtM * B).sum()) + float(((A.T @ A) * (B @ B.T)).sum())
    return eb, es, opt, tot, lam.numpy()


def ey_bound(cfg, lam):
    """Allowed err^2 / opt^2 of the rank-r factors, from lam, the squared
    singular values of M (any order).

    Gap case (true rank R >= r): the top-r subspace is well separated and the
    factors must be Eckart-Young optimal to 1%.  Noise floor (R < r): the
    signal subspace must be captured and the other m = r - R kept directions
    may be any directions of the noise subspace; the factors must do no worse
    than the expected error of m directions drawn uniformly from it,
    sum(noise) - m mean(noise), where noise holds the D - R smallest lam.
    (The noise is not isotropic -- bf16 rounding of M scales with |M| -- so
    no closed form of its spectrum is assumed.)
    """
    m = cfg.r - cfg.rank_true
    if m <= 0:
        return 1.01
    lam = np.sort(np.asarray(lam, np.float64))
    opt = lam[: lam.size - cfg.r].sum()
    if opt <= 0.0:
        return 1.01          # r covers every direction: exact up to roundoff
    noise = lam[: lam.size - cfg.rank_true]
    return (noise.sum() - m * noise.mean()) / opt * (1.0 + 1e-6)

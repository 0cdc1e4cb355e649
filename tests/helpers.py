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

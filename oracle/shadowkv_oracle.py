"""CPU oracle for ShadowKV prefill (Algorithm 1) and decode (Algorithm 2).

TEST INFRASTRUCTURE ONLY. This module is the plain, slow, float64 statement of
what the method computes. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import it; the library never does.

Source: "ShadowKV: KV Cache in Shadows for High-Throughput Long-Context LLM
Inference" (xllm-io paper review page), sections 核心公式 (formulas),
算法细节 (Algorithm 1: Pre-filling, Algorithm 2: Decoding) and 关键参数 (key
parameters); the Telegram explainer of ShadowKV for the set-difference cache.

Readings where the page is silent or garbled (each one is listed, with its
reason, in the design notes of the repository):

  R1  RoPE is the rotate-half variant: dimension i pairs with i + d/2 and
      turns by pos * theta**(-2i/d); positions are 0-based token indices.
  R2  The chunked region is tokens [0, s - w); the last w prompt tokens and
      every appended token form the exact local window (the third, bare K of
      the concatenation in Algorithm 2 step 4).  n = (s - w) / c chunks.
  R3  Cosine similarity divides by max(|x| |L|, 1e-8).
  R4  Outliers are chosen per (batch, KV head); decode candidates are all
      chunks of that head except its outliers.
  R5  S2 (undefined on the page) is the maximum over the query heads of a KV
      group of softmax_j(P / sqrt(d)) over the candidates; group_reduce="sum"
      gives the alternative reading (sum over the group).
  R6  ArgTopK breaks ties toward the lower index and returns the indices in
      ascending order.
  R7  Attention is softmax(q K^T / sqrt(d)) V over [outliers; RoPE(rebuilt);
      local], with consecutive query heads sharing a KV head (g // G).
  R8  A = U_r S_r and B = V_r^T split per KV head; only the product A B is
      unique, so checks compare products and projections, never factors.
  R9  Cache: capacity k chunks per (batch, KV head), holding the previous
      step's selection; hits_t = |I_t  intersect  I_{t-1}|; step 0 has none.
  R10 The equivalent-bandwidth example leaves the hit rate unprinted;
      alpha = 0.6 (the page's "about 60%") reproduces 7.2 TB/s.
  R11 K_sparse (Algorithm 2 step 3) is a tensor of the workload's element
      type, like A, B, L, the outliers, the local window and V: its exact
      value RoPE(Gather(A, I) B) is rounded to that type (round to nearest,
      ties to even) before the attention.  key_dtype="f64" keeps it exact.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "rope", "n_chunks", "chunk_landmarks", "chunk_min_cosine", "argtopk",
    "svd_factors", "prefill", "attention", "OracleState", "OracleDecoder",
    "equivalent_bandwidth", "subspace_similarity", "hit_count", "store",
]


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------
# RoPE (reading R1).  Algorithm 1 takes K_RoPE as input; Algorithm 2 step 4
# applies RoPE to the rebuilt keys.
# --------------------------------------------------------------------------
def rope(x, pos, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of x (..., d) at integer positions pos (...)."""
    x = _f64(x)
    d = x.shape[-1]
    half = d // 2
    inv_freq = float(theta) ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = _f64(pos)[..., None] * inv_freq
    cos, sin = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def n_chunks(s: int, c: int, w: int) -> int:
    """Number of chunks of the compressed region (reading R2)."""
    return (s - w) // c


# --------------------------------------------------------------------------
# Algorithm 1 step 2: C = Reduce(K_RoPE), the per-chunk mean (landmarks L).
# --------------------------------------------------------------------------
def chunk_landmarks(k_rope, c: int, n: int) -> np.ndarray:
    """k_rope (..., s, d) -> landmarks (..., n, d): mean of each chunk of c tokens."""
    k = _f64(k_rope)
    chunks = k[..., : n * c, :].reshape(*k.shape[:-2], n, c, k.shape[-1])
    return chunks.sum(axis=-2) / c


# --------------------------------------------------------------------------
# Algorithm 1 steps 3-4: S = CosineSimilarity(C, K_RoPE); Min over the chunk.
# --------------------------------------------------------------------------
def chunk_min_cosine(k_rope, landmarks, c: int) -> np.ndarray:
    """Minimum over the c tokens of a chunk of cos(token, chunk mean) (reading R3)."""
    k = _f64(k_rope)
    L = _f64(landmarks)
    n = L.shape[-2]
    chunks = k[..., : n * c, :].reshape(*k.shape[:-2], n, c, k.shape[-1])
    dots = np.einsum("...ud,...d->...u", chunks, L)
    norms = np.linalg.norm(chunks, axis=-1) * np.linalg.norm(L, axis=-1)[..., None]
    cos = dots / np.maximum(norms, 1e-8)
    return cos.min(axis=-1)


def argtopk(scores, k: int, valid=None) -> np.ndarray:
    """ArgTopK along the last axis (reading R6): the k largest scores, ties to
    the lower index, returned in ascending index order.  Entries where
    ``valid`` is False are never chosen."""
    scores = _f64(scores)
    out = np.empty(scores.shape[:-1] + (k,), dtype=np.int64)
    flat_s = scores.reshape(-1, scores.shape[-1])
    flat_v = None if valid is None else np.asarray(valid, bool).reshape(-1, scores.shape[-1])
    flat_o = out.reshape(-1, k)
    for i in range(flat_s.shape[0]):
        idx = np.arange(flat_s.shape[1])
        sc = flat_s[i]
        if flat_v is not None:
            idx = idx[flat_v[i]]
            sc = sc[flat_v[i]]
        if k > idx.size:
            raise ValueError("k exceeds the number of valid entries")
        # primary key: score descending; secondary: index ascending
        order = np.lexsort((idx, -sc))
        flat_o[i] = np.sort(idx[order[:k]])
    return out


# --------------------------------------------------------------------------
# Algorithm 1 step 1: A in R^{b x s x r}, B in R^{b x h_kv x r x d} <- SVD(K)
# over the pre-RoPE keys of all s tokens (reading R8).
# --------------------------------------------------------------------------
def svd_factors(k_pre, r: int):
    """k_pre (b, h_kv, s, d) -> (A (b, s, r), B (b, h_kv, r, d), sigma (b, min(s, h_kv d)))."""
    k = _f64(k_pre)
    b, h, s, d = k.shape
    A = np.empty((b, s, r))
    B = np.empty((b, h, r, d))
    sig = []
    for bi in range(b):
        M = k[bi].transpose(1, 0, 2).reshape(s, h * d)   # M[t, h*d + e] = K[h, t, e]
        U, S, Vt = np.linalg.svd(M, full_matrices=False)
        A[bi] = U[:, :r] * S[:r]
        B[bi] = Vt[:r].reshape(r, h, d).transpose(1, 0, 2)
        sig.append(S)
    return A, B, np.stack(sig)


@dataclass
class OracleState:
    """Compressed per-layer state after Algorithm 1 (the inputs of Algorithm 2).

    Arrays may be float32 or float64; every use converts to float64.
      A (b, s, r)   B (b, h_kv, r, d)   L (b, h_kv, n, d)
      outlier_ids (b, h_kv, o) ascending    K_out, V_out (b, h_kv, o*c, d)
      K_loc, V_loc (b, h_kv, w, d)          V_cpu (b, h_kv, s, d)
    """
    c: int
    theta: float
    A: np.ndarray
    B: np.ndarray
    L: np.ndarray
    outlier_ids: np.ndarray
    K_out: np.ndarray
    V_out: np.ndarray
    K_loc: np.ndarray
    V_loc: np.ndarray
    V_cpu: np.ndarray
    min_cos: Optional[np.ndarray] = None

    @property
    def shape(self):
        b, h, n, d = self.L.shape
        return b, h, n, d


def prefill(k_pre, v, c: int, r: int, o: int, w: int, theta: float) -> OracleState:
    """Algorithm 1 on pre-RoPE keys k_pre and values v, both (b, h_kv, s, d)."""
    k_pre = _f64(k_pre)
    b, h, s, d = k_pre.shape
    n = n_chunks(s, c, w)
    pos = np.arange(s)
    k_rope = rope(k_pre, pos, theta)                      # K_RoPE
    L = chunk_landmarks(k_rope, c, n)                     # step 2
    m = chunk_min_cosine(k_rope, L, c)                    # step 3 + Min
    out_ids = argtopk(-m, o)                              # step 4
    A, B, _ = svd_factors(k_pre, r)                       # step 1
    rows = (out_ids[..., None] * c + np.arange(c)).reshape(b, h, o * c)
    take = lambda x: np.take_along_axis(x, rows[..., None], axis=2)
    return OracleState(
        c=c, theta=theta, A=A, B=B, L=L, outlier_ids=out_ids,
        K_out=take(k_rope), V_out=take(_f64(v)),
        K_loc=k_rope[:, :, n * c:], V_loc=_f64(v)[:, :, n * c:],
        V_cpu=np.asarray(v), min_cos=m)


# --------------------------------------------------------------------------
# Element types of materialised tensors (reading R11).
# --------------------------------------------------------------------------
def store(x, dtype: str) -> np.ndarray:
    """x rounded to the element type `dtype` ("f64", "f32" or "bf16"), returned
    as float64.  bf16 keeps the upper 16 bits of the float32 value, rounded
    to nearest with ties to even (float64 -> float32 first)."""
    x = _f64(x)
    if dtype == "f64":
        return x
    x32 = np.ascontiguousarray(x.astype(np.float32))
    if dtype == "f32":
        return x32.astype(np.float64)
    if dtype != "bf16":
        raise ValueError(dtype)
    u = x32.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Algorithm 2 step 4: attention over the concatenated keys and values.
# --------------------------------------------------------------------------
def attention(q, K, V) -> np.ndarray:
    """softmax(q K^T / sqrt(d)) V for a group of queries sharing K and V
    (reading R7).  q (..., G, d); K, V (..., T, d) -> (..., G, d)."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    d = q.shape[-1]
    logits = np.einsum("...gd,...td->...gt", q, K) / np.sqrt(d)
    p = np.exp(logits - logits.max(axis=-1, keepdims=True))
    return np.einsum("...gt,...td->...gd", p / p.sum(axis=-1, keepdims=True), V)


@dataclass
class StepResult:
    P: np.ndarray        # (b, h_q, n) q.L / sqrt(d); NaN at outlier chunks
    S2: np.ndarray       # (b, h_kv, n) selection score; NaN at outlier chunks
    sel: np.ndarray      # (b, h_kv, k) chosen chunks, ascending
    out: np.ndarray      # (b, h_q, d)
    hits: np.ndarray     # (b, h_kv)
    K_sparse: np.ndarray  # (b, h_kv, k*c, d) RoPE(Gather(A, I) B)


@dataclass
class OracleDecoder:
    """Algorithm 2, one call per decode step, on an OracleState."""
    state: OracleState
    h_q: int
    k: int
    group_reduce: str = "max"
    key_dtype: str = "f64"          # element type of K_sparse (reading R11)
    t: int = 0
    prev_sel: Optional[np.ndarray] = None
    app_K: list = field(default_factory=list)
    app_V: list = field(default_factory=list)

    def scores(self, q):
        """Steps 1-2: P = MatMul(Q, L^T) and S2 (readings R4, R5)."""
        st = self.state
        b, h, n, d = st.shape
        G = self.h_q // h
        q = _f64(q)
        cand = np.ones((b, h, n), bool)
        for bi in range(b):
            for hi in range(h):
                cand[bi, hi, st.outlier_ids[bi, hi]] = False
        L = _f64(st.L)
        P = np.einsum("bhgd,bhnd->bhgn", q.reshape(b, h, G, d), L) / np.sqrt(d)
        P = np.where(cand[:, :, None, :], P, -np.inf)
        mx = P.max(axis=-1, keepdims=True)
        e = np.exp(P - mx)
        S1 = e / e.sum(axis=-1, keepdims=True)              # softmax over candidates
        if self.group_reduce == "max":
            S2 = S1.max(axis=2)
        elif self.group_reduce == "sum":
            S2 = S1.sum(axis=2)
        else:
            raise ValueError(self.group_reduce)
        P = np.where(cand[:, :, None, :], P, np.nan).reshape(b, self.h_q, n)
        S2 = np.where(cand, S2, np.nan)
        return P, S2, cand

    def step(self, q, k_new=None, v_new=None, force_sel=None) -> StepResult:
        st = self.state
        b, h, n, d = st.shape
        c = st.c
        G = self.h_q // h
        q = _f64(q).reshape(b, self.h_q, d)
        if k_new is not None:
            self.app_K.append(_f64(k_new).reshape(b, h, 1, d))
            self.app_V.append(_f64(v_new).reshape(b, h, 1, d))
        P, S2, cand = self.scores(q)
        sel = argtopk(np.where(cand, S2, -np.inf), self.k, valid=cand)   # step 2
        if force_sel is not None:
            sel = np.asarray(force_sel, np.int64).reshape(b, h, self.k)
        rows = (sel[..., None] * c + np.arange(c)).reshape(b, h, self.k * c)
        A = st.A
        out = np.empty((b, self.h_q, d))
        K_sparse = np.empty((b, h, self.k * c, d))
        hits = np.zeros((b, h), np.int64)
        K_loc = np.concatenate([_f64(st.K_loc)] + self.app_K, axis=2)
        V_loc = np.concatenate([_f64(st.V_loc)] + self.app_V, axis=2)
        for bi in range(b):
            for hi in range(h):
                r_ = rows[bi, hi]
                Ks = _f64(A[bi][r_]) @ _f64(st.B[bi, hi])                 # step 3 (key)
                Ks = store(rope(Ks, r_, st.theta), self.key_dtype)        # step 4 RoPE
                K_sparse[bi, hi] = Ks
                Vs = _f64(st.V_cpu[bi, hi][r_])                           # step 3 (value)
                Katt = np.concatenate([_f64(st.K_out[bi, hi]), Ks, K_loc[bi, hi]])
                Vatt = np.concatenate([_f64(st.V_out[bi, hi]), Vs, V_loc[bi, hi]])
                out[bi, hi * G:(hi + 1) * G] = attention(q[bi, hi * G:(hi + 1) * G], Katt, Vatt)
                if self.prev_sel is not None:
                    hits[bi, hi] = hit_count(self.prev_sel[bi, hi], sel[bi, hi])
        self.prev_sel = sel
        self.t += 1
        return StepResult(P=P, S2=S2, sel=sel, out=out, hits=hits, K_sparse=K_sparse)


def hit_count(prev_sel, sel) -> int:
    """Chunks of this step already resident from the previous step (reading R9)."""
    return int(np.intersect1d(np.asarray(prev_sel), np.asarray(sel)).size)


# --------------------------------------------------------------------------
# 核心公式: equivalent bandwidth and low-rank subspace similarity.
# --------------------------------------------------------------------------
def equivalent_bandwidth(S, C, K, O, alpha, B_gpu, B_pcie):
    """B~ = 2 S B_gpu / (S/C + 2 (K+O) C + (1 - alpha) K C B_gpu / B_pcie)."""
    S, C, K, O = float(S), float(C), float(K), float(O)
    return 2.0 * S * B_gpu / (S / C + 2.0 * (K + O) * C + (1.0 - alpha) * K * C * B_gpu / B_pcie)


def subspace_similarity(V1, V2, r: int) -> float:
    """D(H1, H2) = <H1, H2>_F / r with H = V V^T, V holding r orthonormal columns."""
    V1, V2 = _f64(V1), _f64(V2)
    H1 = V1 @ V1.T
    H2 = V2 @ V2.T
    return float(np.sum(H1 * H2) / r)

"""Seeded synthetic inputs shaped like the ShadowKV review's workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no RoPE, no chunk statistics, no SVD, no attention).
Both the library's tests/benchmark and the CPU oracle consume its output.

Workloads (ShadowKV review page, 关键参数 and 吞吐量评估): Llama-3-8B-style
GQA heads (h_q=32, h_kv=8, d=128, theta=5e5), chunk 8, rank 160, 48 outlier
chunks, a 1.56% sparse budget, 32K-256K contexts, batch 1-48.

Keys (pre-RoPE): K = U W + noise * N(0, 1), with U an (s + T) x R Gaussian
walk along the sequence and W ~ N(0, 1/R) (standard deviation 1/sqrt(R)).
The walk is the stationary form U_t = rho U_{t-1} + sigma e_t with
rho = sqrt(1 - sigma^2) and U_0 ~ N(0, 1), so that every key has unit-scale
entries at every position of a 256K context (a plain cumulative walk would
grow like sqrt(t)).  Planted tokens: token 0 (an attention sink) x8; "heavy"
chunks whose keys are all scaled x8; "spike" chunks where one token is
replaced by its negation, which breaks the chunk's cosine locality.
Values: V ~ N(0, 1).  Queries: q_0 = normalize(N(0, 1)) sqrt(d), then
q_t = normalize(q_{t-1} + sigma_q N(0, 1)) sqrt(d).  Appended keys continue
the same walk past position s and stand in for post-RoPE keys.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

__all__ = ["Config", "CONFIGS", "make_inputs", "make_state", "torch_dtype"]


@dataclass(frozen=True)
class Config:
    name: str
    b: int
    h_q: int
    h_kv: int
    d: int
    s: int
    c: int
    r: int
    k: int
    o: int
    w: int
    theta: float
    dtype: str          # "f32" or "bf16"
    steps: int
    rank_true: int
    q_sigma: float
    seed: int
    n_heavy: int = 2
    n_spike: int = 0
    noise: float = 0.01

    @property
    def n(self) -> int:
        return (self.s - self.w) // self.c

    @property
    def G(self) -> int:
        return self.h_q // self.h_kv

    @property
    def max_new(self) -> int:
        return self.steps

    def with_(self, **kw) -> "Config":
        return replace(self, **kw)


CONFIGS = {
    # tiny single layer, fp32 (parity only)
    "tiny_f32_s1k": Config("tiny_f32_s1k", b=1, h_q=4, h_kv=2, d=64, s=1024, c=8, r=32,
                           k=16, o=4, w=32, theta=1e4, dtype="f32", steps=4,
                           rank_true=24, q_sigma=0.1, seed=0, n_heavy=2, n_spike=0),
    # Llama-3-8B-style layer, 32K context
    "llama_b1_s32k": Config("llama_b1_s32k", b=1, h_q=32, h_kv=8, d=128, s=32768, c=8,
                            r=160, k=64, o=48, w=64, theta=5e5, dtype="bf16", steps=16,
                            rank_true=96, q_sigma=0.1, seed=1, n_spike=8),
    # long context: batch 8 at 128K (the headline decode workload)
    "llama_b8_s128k": Config("llama_b8_s128k", b=8, h_q=32, h_kv=8, d=128, s=131072, c=8,
                             r=160, k=256, o=48, w=64, theta=5e5, dtype="bf16", steps=32,
                             rank_true=96, q_sigma=0.1, seed=2, n_spike=8),
    # large batch at 60K
    "llama_b48_s60k": Config("llama_b48_s60k", b=48, h_q=32, h_kv=8, d=128, s=61440, c=8,
                             r=160, k=120, o=48, w=64, theta=5e5, dtype="bf16", steps=64,
                             rank_true=96, q_sigma=0.1, seed=3, n_spike=8),
    # prefill + decode at 256K
    "llama_b2_s256k": Config("llama_b2_s256k", b=2, h_q=32, h_kv=8, d=128, s=262144, c=8,
                             r=160, k=512, o=48, w=64, theta=5e5, dtype="bf16", steps=64,
                             rank_true=128, q_sigma=0.05, seed=4, n_spike=8),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _walk(e: torch.Tensor, rho: float) -> torch.Tensor:
    """x_t = rho x_{t-1} + e_t along dim 1, by a log-depth doubling scan."""
    x = e.clone()
    step = 1
    n = x.shape[1]
    while step < n:
        x[:, step:] = x[:, step:] + (rho ** step) * x[:, :-step].clone()
        step *= 2
    return x


def _keys(cfg: Config, g: torch.Generator, dev, T: int, rank_true: int, noise: float):
    b, s, D = cfg.b, cfg.s, cfg.h_kv * cfg.d
    sigma = 0.1
    rho = math.sqrt(1.0 - sigma * sigma)
    e = torch.randn(b, s + T, rank_true, generator=g, device=dev)
    e[:, 1:] *= sigma
    U = _walk(e, rho)
    W = torch.randn(b, rank_true, D, generator=g, device=dev) / math.sqrt(rank_true)
    K = torch.bmm(U, W)
    if noise > 0:
        K += noise * torch.randn(b, s + T, D, generator=g, device=dev)
    return K.view(b, s + T, cfg.h_kv, cfg.d).permute(0, 2, 1, 3).contiguous()


def make_inputs(cfg: Config, device="cpu", seed: Optional[int] = None,
                noise: Optional[float] = None, rank_true: Optional[int] = None,
                plant: bool = True):
    """Prefill inputs plus the decode-step stream of cfg.

    Returns a dict of tensors on `device`, in the config's dtype:
      k_pre, v   (b, h_kv, s, d)   pre-RoPE keys and values of the prompt
      q          (T, b, h_q, d)    post-RoPE queries, one per decode step
      k_new, v_new (T, b, h_kv, d) keys/values appended at each step
      heavy, spike (long)          planted chunk indices (for inspection)
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(cfg.seed if seed is None else seed)
    T = cfg.steps
    noise = cfg.noise if noise is None else noise
    rank_true = cfg.rank_true if rank_true is None else rank_true
    K = _keys(cfg, g, dev, T, rank_true, noise)             # (b, h, s+T, d)
    n = cfg.n
    heavy = torch.randperm(n, generator=g, device=dev)[: cfg.n_heavy] if plant else None
    spike = torch.randperm(n, generator=g, device=dev)[: cfg.n_spike] if plant else None
    if plant:
        K[:, :, 0] *= 8.0                                     # attention sink
        for j in heavy.tolist():
            K[:, :, j * cfg.c:(j + 1) * cfg.c] *= 8.0
        for j in spike.tolist():
            u = 1 + (j % (cfg.c - 1))
            K[:, :, j * cfg.c + u] *= -1.0
    k_pre = K[:, :, : cfg.s].contiguous()
    k_new = K[:, :, cfg.s:].permute(2, 0, 1, 3).contiguous()   # (T, b, h, d)
    v = torch.randn(cfg.b, cfg.h_kv, cfg.s, cfg.d, generator=g, device=dev)
    v_new = torch.randn(T, cfg.b, cfg.h_kv, cfg.d, generator=g, device=dev)
    q = _queries(cfg, g, dev, T)
    dt = torch_dtype(cfg.dtype)
    return dict(k_pre=k_pre.to(dt), v=v.to(dt), q=q.to(dt), k_new=k_new.to(dt),
                v_new=v_new.to(dt), heavy=heavy, spike=spike)


def _queries(cfg: Config, g, dev, T: int):
    d = cfg.d
    qs = []
    q = torch.randn(cfg.b, cfg.h_q, d, generator=g, device=dev)
    q = q / q.norm(dim=-1, keepdim=True) * math.sqrt(d)
    for _ in range(T):
        qs.append(q)
        q = q + cfg.q_sigma * torch.randn(cfg.b, cfg.h_q, d, generator=g, device=dev)
        q = q / q.norm(dim=-1, keepdim=True) * math.sqrt(d)
    return torch.stack(qs)


def make_state(cfg: Config, device="cpu", seed: Optional[int] = None, n_hot: int = 8):
    """A random compressed state with the shapes of Algorithm 2's inputs.

    Used to test decode in isolation: both the library (through its state
    import) and the oracle consume the same arrays.  Entries are random; the
    state is not the prefill of any key cache.  `n_hot` landmarks per head
    are scaled x3 so the selection has clear winners.
    Returns tensors in the config's dtype (outlier_ids int32, ascending):
      A (b, s, r)  B (b, h_kv, r, d)  L (b, h_kv, n, d)  outlier_ids (b, h_kv, o)
      K_out, V_out (b, h_kv, o*c, d)  K_loc, V_loc (b, h_kv, w, d)  v (b, h_kv, s, d)
    plus the decode stream q, k_new, v_new as in make_inputs.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed((cfg.seed if seed is None else seed) + 1000)
    b, h, s, d, c, r, o, w, n = cfg.b, cfg.h_kv, cfg.s, cfg.d, cfg.c, cfg.r, cfg.o, cfg.w, cfg.n
    T = cfg.steps
    A = torch.randn(b, s, r, generator=g, device=dev)
    B = torch.randn(b, h, r, d, generator=g, device=dev) / math.sqrt(r)
    L = 0.5 * torch.randn(b, h, n, d, generator=g, device=dev)
    hot = torch.randint(0, n, (b, h, n_hot), generator=g, device=dev)
    L.scatter_(2, hot[..., None].expand(b, h, n_hot, d),
               3.0 * torch.gather(L, 2, hot[..., None].expand(b, h, n_hot, d)))
    keys = torch.rand(b, h, n, generator=g, device=dev)
    ids = torch.sort(torch.topk(keys, o, dim=-1).indices, dim=-1).values.to(torch.int32)
    K_out = torch.randn(b, h, o * c, d, generator=g, device=dev)
    V_out = torch.randn(b, h, o * c, d, generator=g, device=dev)
    K_loc = torch.randn(b, h, w, d, generator=g, device=dev)
    V_loc = torch.randn(b, h, w, d, generator=g, device=dev)
    v = torch.randn(b, h, s, d, generator=g, device=dev)
    q = _queries(cfg, g, dev, T)
    k_new = torch.randn(T, b, h, d, generator=g, device=dev)
    v_new = torch.randn(T, b, h, d, generator=g, device=dev)
    dt = torch_dtype(cfg.dtype)
    out = dict(A=A, B=B, L=L, K_out=K_out, V_out=V_out, K_loc=K_loc, V_loc=V_loc, v=v,
               q=q, k_new=k_new, v_new=v_new)
    out = {key: val.to(dt) for key, val in out.items()}
    out["outlier_ids"] = ids
    return out

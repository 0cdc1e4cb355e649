"""The attention entry point that allocates nothing (shadowkv_attention_noalloc).

Callers that cannot allocate device memory -- an engine that gives all of it
to its own pool at start-up, or a decode loop recorded into a CUDA graph --
run the split-KV attention on keys and values they already hold; the
library's scratch for the split partials and tickets is a static device
array.  This file is collected last on purpose, so that a failure here does
not hide the other GPU tests; it must also pass alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import TOL, head_errors, np64
from oracle import shadowkv_oracle as O
from sparse_rank_kv_gb300 import binding, build, synth
from sparse_rank_kv_gb300.synth import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.lib()


CFG = CONFIGS["llama_b1_s32k"].with_(
    name="noalloc", b=2, h_q=8, h_kv=2, d=128, s=8000 + 64, c=8, r=64, k=37, o=6, w=64,
    theta=5e5, dtype="bf16", steps=4, seed=71)


def _step_inputs(ctx, cfg, n_loc):
    """The keys and values the decode step just attended over, as dense
    b x h_kv x n x d arrays: outliers, rebuilt chunks (values from their cache
    slots), local window."""
    b, h, d, k, c, o = cfg.b, cfg.h_kv, cfg.d, cfg.k, cfg.c, cfg.o
    cap = cfg.w + cfg.max_new
    Kout = ctx.export("K_OUT").view(b, h, o * c, d)
    Vout = ctx.export("V_OUT").view(b, h, o * c, d)
    Ks = ctx.export("K_SPARSE").view(b, h, k * c, d)
    slots = ctx.export("SEL_SLOT").view(b, h, k).long()
    slotV = ctx.export("SLOT_V").view(b, h, k, c, d)
    Vs = torch.gather(slotV, 2, slots[..., None, None].expand(b, h, k, c, d)).reshape(b, h, k * c, d)
    Kl = ctx.export("K_LOC").view(b, h, cap, d)[:, :, :n_loc]
    Vl = ctx.export("V_LOC").view(b, h, cap, d)[:, :, :n_loc]
    K = torch.cat([Kout, Ks, Kl], dim=2).cuda().contiguous()
    V = torch.cat([Vout, Vs, Vl], dim=2).cuda().contiguous()
    return K, V


def test_noalloc_attention_matches_decode_step_and_oracle_twice():
    """Two calls in a row (they share the static scratch and its tickets):
    each output matches the decode step's attention over the same keys and
    values, and the oracle's softmax(q K^T / sqrt(d)) V on them."""
    cfg = CFG
    st = synth.make_state(cfg, device="cuda")
    p = binding.make_params(cfg)
    ctx = binding.load_state(p, st)
    G = cfg.h_q // cfg.h_kv
    for t in range(2):
        q = st["q"][t].contiguous()
        ref = torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=torch.bfloat16, device="cuda")
        ctx.decode_step(q, st["k_new"][t], st["v_new"][t], ref)
        torch.cuda.synchronize()
        K, V = _step_inputs(ctx, cfg, cfg.w + t + 1)
        got = torch.empty_like(ref)
        binding.attention_noalloc(p, q, K, V, got)
        torch.cuda.synchronize()
        err = head_errors(np64(got), np64(ref))
        assert err.max() <= TOL["bf16"], f"call {t}: {err.max():.3g} against the decode step"
        orc = O.attention(np64(q).reshape(cfg.b, cfg.h_kv, G, cfg.d), np64(K), np64(V))
        err = head_errors(np64(got), orc.reshape(cfg.b, cfg.h_q, cfg.d))
        assert err.max() <= TOL["bf16"], f"call {t}: {err.max():.3g} against the oracle"
    ctx.check()


def test_noalloc_rejects_oversized_problems():
    p = binding.make_params(CFG.with_(b=64, h_q=64, h_kv=8))
    q = torch.empty(1, device="cuda")
    ptr = ctypes.c_void_p(q.data_ptr())
    rc = binding.lib().shadowkv_attention_noalloc(ctypes.byref(p), ptr, ptr, ptr, 1 << 20, ptr, None)
    with pytest.raises(binding.ShadowKVError) as ei:
        binding._check(rc)
    assert ei.value.code == 7 and "static scratch" in str(ei.value)


def test_noalloc_rejects_misaligned_keys_before_any_work():
    """K and V are copied 16 bytes at a time: an offset view is refused on
    the host.  n_tokens = 0 would be refused too, after the alignment check,
    so no kernel can run here whichever check answers."""
    p = binding.make_params(CFG)
    buf = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    good = ctypes.c_void_p(buf.data_ptr())
    bad = ctypes.c_void_p(buf.data_ptr() + 2)
    for K, V in ((bad, good), (good, bad)):
        rc = binding.lib().shadowkv_attention_noalloc(ctypes.byref(p), good, K, V, 0, good, None)
        with pytest.raises(binding.ShadowKVError) as ei:
            binding._check(rc)
        assert ei.value.code == 1 and "16-byte aligned" in str(ei.value)
    odd = ctypes.c_void_p(buf.data_ptr() + 1)
    rc = binding.lib().shadowkv_attention_noalloc(ctypes.byref(p), odd, good, good, 0, good, None)
    with pytest.raises(binding.ShadowKVError) as ei:
        binding._check(rc)
    assert ei.value.code == 1 and "element size" in str(ei.value)

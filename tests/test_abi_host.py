"""Host-side checks of the C ABI: the library builds, loads and exports every
symbol include/shadowkv.h declares, and parameter validation, footprint and
kernel naming work without a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest

from sparse_rank_kv_gb300 import binding, build
from sparse_rank_kv_gb300.synth import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "shadowkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(shadowkv_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared_symbols()
    assert len(names) >= 16
    for name in names:
        assert hasattr(lib, name), f"{name} declared in shadowkv.h but not exported"


def test_validate_accepts_every_config(lib):
    for cfg in CONFIGS.values():
        binding.validate_params(binding.make_params(cfg))


@pytest.mark.parametrize("change,code", [
    (dict(h_q=6, h_kv=4), 1),        # h_q not a multiple of h_kv
    (dict(h_q=24, h_kv=8), 7),       # group of 3 unsupported
    (dict(d=96), 7),                 # head dim
    (dict(w=30), 1),                 # (s - w) not a multiple of c
    (dict(k=0), 1),
    (dict(k=4050), 1),               # k > n - o (n = 4088, o = 48)
    (dict(k=2000), 7),               # k > 1024
    (dict(o=-1), 1),
    (dict(r=0), 1),
    (dict(r=5000), 1),               # r > h_kv * d
    (dict(r=300, h_kv=4, d=128), 7), # r > 256
    (dict(dtype=5), 1),
    (dict(group_reduce=2), 1),
    (dict(rope_theta=0.0), 1),
    (dict(reserved=1), 1),
    (dict(max_new=-1), 1),
])
def test_validate_rejects(lib, change, code):
    p = binding.make_params(CONFIGS["llama_b1_s32k"], **change)
    with pytest.raises(binding.ShadowKVError) as ei:
        binding.validate_params(p)
    assert ei.value.code == code
    assert lib.shadowkv_last_error().decode()


def test_too_many_chunks_is_unsupported(lib):
    p = binding.make_params(CONFIGS["llama_b1_s32k"], s=64 * 8 * 1024 + 64)
    with pytest.raises(binding.ShadowKVError) as ei:
        binding.validate_params(p)
    assert ei.value.code == 7


def test_footprint_matches_layout(lib):
    cfg = CONFIGS["llama_b8_s128k"]
    dev, host = binding.footprint(binding.make_params(cfg))
    n = cfg.n
    E = 2
    # host: the pinned copy of V
    assert host == cfg.b * cfg.h_kv * cfg.s * cfg.d * E
    # device: at least A, B, L, the outliers, the slot cache and the rebuilt keys
    floor = (cfg.b * cfg.s * cfg.r + cfg.b * cfg.h_kv * cfg.d * cfg.r + cfg.b * cfg.h_kv * n * cfg.d
             + 2 * cfg.b * cfg.h_kv * cfg.o * cfg.c * cfg.d + 2 * cfg.b * cfg.h_kv * cfg.k * cfg.c * cfg.d) * E
    assert floor <= dev <= floor * 1.3


def test_null_arguments_are_rejected_without_gpu(lib):
    out = ctypes.c_void_p()
    p = binding.make_params(CONFIGS["tiny_f32_s1k"])
    assert lib.shadowkv_prefill(ctypes.byref(p), None, None, 0, None, ctypes.byref(out)) == 1
    assert lib.shadowkv_decode_step(None, None, None, None, None, None) == 1
    assert lib.shadowkv_decode_step_host(None, None, None, None, None, None) == 1
    assert lib.shadowkv_set_option(None, 0, 1) == 1
    lib.shadowkv_free(None)   # NULL-safe


def test_kernel_names(lib):
    names = binding.kernel_names()
    assert names[:5] == ["score", "select", "fetch", "rebuild", "attention"]
    assert len(set(names)) == len(names)


def test_noalloc_alignment_is_checked_on_the_host(lib):
    """The no-alloc attention refuses K/V that are not 16-byte aligned, and q
    or out not aligned to their element size, before any CUDA call (the
    pointers here are never dereferenced: n_tokens = 0 would be refused next)."""
    p = binding.make_params(CONFIGS["llama_b1_s32k"])
    ok, k_bad, q_bad = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008), ctypes.c_void_p(0x10001)
    f = lib.shadowkv_attention_noalloc
    assert f(ctypes.byref(p), ok, k_bad, ok, 0, ok, None) == 1
    assert "16-byte aligned" in lib.shadowkv_last_error().decode()
    assert f(ctypes.byref(p), ok, ok, k_bad, 0, ok, None) == 1
    assert "16-byte aligned" in lib.shadowkv_last_error().decode()
    assert f(ctypes.byref(p), q_bad, ok, ok, 0, ok, None) == 1
    assert "element size" in lib.shadowkv_last_error().decode()
    assert f(ctypes.byref(p), ok, ok, ok, 0, q_bad, None) == 1
    assert "element size" in lib.shadowkv_last_error().decode()
    assert f(ctypes.byref(p), ok, ok, ok, 0, ok, None) == 1
    assert "n_tokens" in lib.shadowkv_last_error().decode()

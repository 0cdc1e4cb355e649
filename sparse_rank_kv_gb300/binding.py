"""ctypes binding of libshadowkv.so (include/shadowkv.h).

Argument marshalling only: tensors become raw pointers, streams become
cudaStream_t handles, status codes become exceptions.  Every computation runs
in the library's CUDA kernels; there is no Python or CPU fallback, and the
binding raises if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libshadowkv.so")

DTYPE_F32, DTYPE_BF16 = 0, 1
GROUP_MAX, GROUP_SUM = 0, 1
OPT_CACHE, OPT_TIMING, OPT_SPLIT_TOKENS, OPT_CUDA_CORES, OPT_REBUILD_IN_ATTENTION = 0, 1, 2, 3, 4

FIELDS = {
    "A": 0, "BT": 1, "L": 2, "MIN_COS": 3, "OUTLIER_IDS": 4, "K_OUT": 5, "V_OUT": 6,
    "K_LOC": 7, "V_LOC": 8, "SEL": 9, "SEL_SLOT": 10, "HITS": 11, "LOGITS": 12,
    "K_SPARSE": 13, "SLOT_CHUNK": 14, "SLOT_V": 15, "V_CPU": 16, "SVD_BASIS": 17,
}
_INT_FIELDS = {"OUTLIER_IDS", "SEL", "SEL_SLOT", "HITS", "SLOT_CHUNK"}
_F32_FIELDS = {"MIN_COS", "LOGITS", "SVD_BASIS"}

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "OOM", 3: "CUDA", 4: "DEVICE_CHECK", 5: "TIMEOUT",
          6: "STATE", 7: "UNSUPPORTED"}


class ShadowKVError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS.get(code, code)}: {msg}")
        self.code = code


class Params(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int), ("h_q", ctypes.c_int), ("h_kv", ctypes.c_int),
                ("d", ctypes.c_int), ("s", ctypes.c_int), ("c", ctypes.c_int),
                ("r", ctypes.c_int), ("k", ctypes.c_int), ("o", ctypes.c_int),
                ("w", ctypes.c_int), ("max_new", ctypes.c_int), ("rope_theta", ctypes.c_float),
                ("dtype", ctypes.c_int), ("group_reduce", ctypes.c_int),
                ("svd_iters", ctypes.c_int), ("reserved", ctypes.c_int),
                ("seed", ctypes.c_ulonglong)]


class StateIn(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("L", ctypes.c_void_p),
                ("outlier_ids", ctypes.c_void_p), ("K_out", ctypes.c_void_p),
                ("V_out", ctypes.c_void_p), ("K_loc", ctypes.c_void_p),
                ("V_loc", ctypes.c_void_p), ("V", ctypes.c_void_p), ("v_on_host", ctypes.c_int)]


class Layout(ctypes.Structure):
    _fields_ = [("kv_records", ctypes.c_int), ("a_tiled", ctypes.c_int), ("tc_score", ctypes.c_int),
                ("tc_rebuild", ctypes.c_int), ("tc_attention", ctypes.c_int),
                ("fetch_in_rebuild", ctypes.c_int), ("fetch_in_attention", ctypes.c_int),
                ("rebuild_in_attention", ctypes.c_int)]


class Stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_longlong), ("hits", ctypes.c_longlong),
                ("misses", ctypes.c_longlong), ("link_bytes", ctypes.c_longlong),
                ("launches", ctypes.c_longlong)]


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libshadowkv.so (built in-tree by sparse_rank_kv_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m sparse_rank_kv_gb300.build` "
                "(the ShadowKV path has no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, V, I, S = ctypes.POINTER, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sig = {
            "shadowkv_validate_params": (I, [P(Params)]),
            "shadowkv_footprint": (I, [P(Params), P(S), P(S)]),
            "shadowkv_prefill": (I, [P(Params), V, V, I, V, P(V)]),
            "shadowkv_load_state": (I, [P(Params), P(StateIn), V, P(V)]),
            "shadowkv_decode_step": (I, [V, V, V, V, V, V]),
            "shadowkv_decode_step_host": (I, [V, V, V, V, V, V]),
            "shadowkv_free": (None, [V]),
            "shadowkv_rewind": (I, [V, V]),
            "shadowkv_last_error": (ctypes.c_char_p, []),
            "shadowkv_set_option": (I, [V, I, ctypes.c_longlong]),
            "shadowkv_get_stats": (I, [V, P(Stats)]),
            "shadowkv_check": (I, [V]),
            "shadowkv_get_layout": (I, [V, P(Layout)]),
            "shadowkv_num_kernels": (I, []),
            "shadowkv_kernel_name": (ctypes.c_char_p, [I]),
            "shadowkv_kernel_times": (I, [V, P(ctypes.c_double), P(ctypes.c_longlong), I]),
            "shadowkv_reset_timers": (I, [V]),
            "shadowkv_field_bytes": (I, [V, I, P(S)]),
            "shadowkv_export": (I, [V, I, V, S]),
            "shadowkv_attention_noalloc": (I, [P(Params), V, V, V, I, V, V]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(code: int):
    if code != 0:
        raise ShadowKVError(code, lib().shadowkv_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_params(cfg=None, **kw) -> Params:
    """Params from a synth.Config (or keyword fields)."""
    if cfg is not None:
        base = dict(b=cfg.b, h_q=cfg.h_q, h_kv=cfg.h_kv, d=cfg.d, s=cfg.s, c=cfg.c, r=cfg.r,
                    k=cfg.k, o=cfg.o, w=cfg.w, max_new=cfg.max_new, rope_theta=cfg.theta,
                    dtype=DTYPE_BF16 if cfg.dtype == "bf16" else DTYPE_F32)
        base.update(kw)
        kw = base
    p = Params()
    for name, _ in Params._fields_:
        setattr(p, name, kw.get(name, 0))
    return p


def validate_params(p: Params) -> None:
    _check(lib().shadowkv_validate_params(ctypes.byref(p)))


def footprint(p: Params):
    dev, host = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().shadowkv_footprint(ctypes.byref(p), ctypes.byref(dev), ctypes.byref(host)))
    return dev.value, host.value


def num_kernels() -> int:
    return lib().shadowkv_num_kernels()


def kernel_names():
    return [lib().shadowkv_kernel_name(i).decode() for i in range(num_kernels())]


class Context:
    """Owns a shadowkv_ctx (freed by close() or garbage collection)."""

    def __init__(self, handle: ctypes.c_void_p, params: Params):
        self._h = handle
        self.params = params

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            lib().shadowkv_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def decode_step(self, q, k_new, v_new, out, stream=None):
        _check(lib().shadowkv_decode_step(self._h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                          _stream(stream)))

    def decode_step_host(self, q, k_new, v_new, out, stream=None):
        """decode_step on host tensors (pinned for asynchronous copies)."""
        _check(lib().shadowkv_decode_step_host(self._h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out),
                                               _stream(stream)))

    def prepared_step(self, q, k_new, v_new, out, stream=None, host=False):
        """A callable that makes the decode_step call (decode_step_host with
        host=True) on these fixed buffers, with the arguments marshalled once
        (a decode loop that reuses its buffers saves that work on every step)."""
        fn = lib().shadowkv_decode_step_host if host else lib().shadowkv_decode_step
        args = (self._h, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(out), _stream(stream))

        def step():
            rc = fn(*args)
            if rc:
                _check(rc)
        return step

    def rewind(self, stream=None):
        _check(lib().shadowkv_rewind(self._h, _stream(stream)))

    def set_option(self, option: int, value: int):
        _check(lib().shadowkv_set_option(self._h, option, value))

    def stats(self) -> Stats:
        st = Stats()
        _check(lib().shadowkv_get_stats(self._h, ctypes.byref(st)))
        return st

    def check(self):
        _check(lib().shadowkv_check(self._h))

    def layout(self) -> dict:
        lay = Layout()
        _check(lib().shadowkv_get_layout(self._h, ctypes.byref(lay)))
        return {name: bool(getattr(lay, name)) for name, _ in Layout._fields_}

    def kernel_times(self):
        n = num_kernels()
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_longlong * n)()
        _check(lib().shadowkv_kernel_times(self._h, ms, cnt, n))
        return {name: (ms[i], cnt[i]) for i, name in enumerate(kernel_names())}

    def reset_timers(self):
        _check(lib().shadowkv_reset_timers(self._h))

    def field_bytes(self, field: str) -> int:
        nb = ctypes.c_size_t()
        _check(lib().shadowkv_field_bytes(self._h, FIELDS[field], ctypes.byref(nb)))
        return nb.value

    def export(self, field: str) -> torch.Tensor:
        """A field copied to a flat CPU tensor (int32, float32, or the context dtype)."""
        nb = self.field_bytes(field)
        if field in _INT_FIELDS:
            dt = torch.int32
        elif field in _F32_FIELDS or self.params.dtype == DTYPE_F32:
            dt = torch.float32
        else:
            dt = torch.bfloat16
        out = torch.empty(nb // torch.tensor([], dtype=dt).element_size(), dtype=dt)
        _check(lib().shadowkv_export(self._h, FIELDS[field], ctypes.c_void_p(out.data_ptr()), nb))
        return out


def prefill(p: Params, k_pre: torch.Tensor, v: torch.Tensor, stream=None) -> Context:
    """Algorithm 1 on device keys k_pre and values v (device or host tensor)."""
    h = ctypes.c_void_p()
    _check(lib().shadowkv_prefill(ctypes.byref(p), _ptr(k_pre), _ptr(v), int(not v.is_cuda),
                                  _stream(stream), ctypes.byref(h)))
    return Context(h, p)


def attention_noalloc(p: Params, q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, out: torch.Tensor,
                      stream=None) -> None:
    """softmax(q K^T / sqrt(d)) V over K, V (b, h_kv, n_tokens, d) on the device,
    with the library's static scratch instead of any allocation."""
    _check(lib().shadowkv_attention_noalloc(ctypes.byref(p), _ptr(q), _ptr(K), _ptr(V),
                                            int(K.shape[2]), _ptr(out), _stream(stream)))


def load_state(p: Params, st: dict, stream=None) -> Context:
    """A context from a given compressed state (keys as in synth.make_state)."""
    s = StateIn(A=_ptr(st["A"]), B=_ptr(st["B"]), L=_ptr(st["L"]),
                outlier_ids=_ptr(st["outlier_ids"]), K_out=_ptr(st["K_out"]),
                V_out=_ptr(st["V_out"]), K_loc=_ptr(st["K_loc"]), V_loc=_ptr(st["V_loc"]),
                V=_ptr(st["v"]), v_on_host=int(not st["v"].is_cuda))
    h = ctypes.c_void_p()
    _check(lib().shadowkv_load_state(ctypes.byref(p), ctypes.byref(s), _stream(stream),
                                     ctypes.byref(h)))
    return Context(h, p)

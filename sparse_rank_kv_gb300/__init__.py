"""ShadowKV decode-time sparse attention for GB300 (sm_103a).

The compute lives in a C-ABI shared library (include/shadowkv.h) built from
the CUDA sources under csrc/; `binding` marshals arguments to it through
ctypes.  Importing this package loads nothing: the library is loaded on first
use of `binding`, and fails loudly if it has not been built.
"""

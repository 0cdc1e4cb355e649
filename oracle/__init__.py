"""CPU oracle (float64) for ShadowKV prefill and decode.

Test infrastructure: imported only by the tests, the smoke check and the
benchmark's CPU-baseline leg.  The library never imports it.
"""
from .shadowkv_oracle import *  # noqa: F401,F403

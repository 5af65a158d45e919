"""RocketKV hot path on GB300: SnapKV++ eviction and hybrid sparse decode (librkv.so).

`rkv` is the ctypes binding of the C ABI in include/rkv.h; `synthetic` draws the seeded inputs.
"""
from . import synthetic  # noqa: F401

__all__ = ["rkv", "synthetic"]

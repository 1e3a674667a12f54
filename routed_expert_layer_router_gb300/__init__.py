"""Routed MoE layer with a per-layer HBM hot-expert cache, for one GB300.

The compute lives in ``libmoe.so`` (hand-written sm_103a CUDA kernels behind
the C ABI in ``include/moe.h``); :mod:`.moe` is a thin ctypes binding with the
same call names, and :mod:`.layer` wires torch-allocated device memory into a
layer object.  Build with :func:`build`.
"""
from .build import build  # noqa: F401
from . import moe  # noqa: F401

"""host_streamed_paged_gb300: host-streamed, block-paged Q8_0-K / Q4_0-V attention on GB300.

The product is the C-ABI CUDA library built from ``csrc/`` (declared in
``include/kvs.h``); :mod:`.kvs` is its ctypes binding.
"""
from . import build  # noqa: F401
from .kvs import *  # noqa: F401,F403
from .kvs import KVStream, KVSError, load  # noqa: F401

"""kv_cache_token_gb300 -- per-decode-step KV-cache eviction engine for GB300.

The compute path is the CUDA library ``libkvevict.so`` (C ABI in
``include/kvevict.h``); this package only marshals torch tensors into it.
There is no CPU fallback: every call fails loudly if the library is absent.
"""
from .binding import (  # noqa: F401
    BF16, F32, H2O, SNAPKV, DROPKV, KEY_F32, KEY_F64, Engine, KvevictError, config_from, lib,
    STAT_NAMES,
)

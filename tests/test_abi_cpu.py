"""The C-ABI library builds, loads without a GPU, exports every symbol the
header declares, and refuses the configurations the pages refuse."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvevict.h")


@pytest.fixture(scope="module")
def lib():
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("nvcc not available")
    from kv_cache_token_gb300 import build as b
    b.build()
    from kv_cache_token_gb300 import binding
    return binding.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvevict_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for required in ("kvevict_decode_step", "kvevict_score", "kvevict_select", "kvevict_compact",
                     "kvevict_create", "kvevict_destroy", "kvevict_workspace_size", "kvevict_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _cfg(**kw):
    from kv_cache_token_gb300 import binding
    base = dict(policy=binding.SNAPKV, num_layers=1, batch=4, num_q_heads=32, num_kv_heads=8,
                head_dim=128, kv_dtype=binding.BF16, blocks_per_pool=1024, max_tokens=4400,
                budget=1024, recent_window=256, obs_window=32, pool_kernel=7)
    base.update(kw)
    return binding.config_from(**base)


def test_refusals(lib):
    from kv_cache_token_gb300 import binding
    v = binding.validate
    assert v(_cfg()) == 0
    assert v(_cfg(pool_kernel=6)) == 2            # even poolKernel
    assert v(_cfg(pool_kernel=0)) == 2
    assert v(_cfg(recent_window=1024)) == 3       # recentWindow >= budget
    assert v(_cfg(recent_window=2000)) == 3
    assert v(_cfg(obs_window=0)) == 4             # obsWindow 0
    assert v(_cfg(block_size=32)) == 1
    assert v(_cfg(num_q_heads=30)) == 1
    assert v(_cfg(head_dim=96)) == 6
    assert v(_cfg(kv_dtype=7)) == 6
    assert v(_cfg(recent_window=0)) == 1
    assert v(_cfg(policy=binding.H2O, obs_window=0)) == 0   # obsWindow only matters for SnapKV
    assert v(_cfg(pool_kernel=1)) == 0


def test_sizes(lib):
    from kv_cache_token_gb300 import binding
    c = _cfg()
    lanes, C, P = 32, 4400, 1024
    sz = lambda w: lib.kvevict_buffer_size(ctypes.byref(c), w)
    assert sz(binding.BUF_K_POOL) == P * 16 * 128 * 2
    assert sz(binding.BUF_POSITIONS) == lanes * C * 4
    assert sz(binding.BUF_RING) == P * 16 * 32 * 4      # a history row per slot
    assert sz(binding.BUF_STATS) == binding.NSTATS * 8
    assert sz(binding.BUF_WORKSPACE) == lib.kvevict_workspace_size(ctypes.byref(c)) > 0
    assert sz(binding.BUF_RING) > 0
    assert lib.kvevict_buffer_size(ctypes.byref(_cfg(policy=binding.H2O)), binding.BUF_RING) == 0
    assert lib.kvevict_buffer_size(ctypes.byref(_cfg(pool_kernel=4)), binding.BUF_K_POOL) == 0


def test_create_rejects_bad_config_before_touching_cuda(lib):
    from kv_cache_token_gb300 import binding
    h = ctypes.c_void_p()
    bufs = binding.Buffers()
    assert lib.kvevict_create(ctypes.byref(_cfg(pool_kernel=2)), ctypes.byref(bufs), ctypes.byref(h)) == 2
    assert not h.value
    assert lib.kvevict_create(ctypes.byref(_cfg()), ctypes.byref(bufs), ctypes.byref(h)) == 1   # NULL buffers
    assert not h.value

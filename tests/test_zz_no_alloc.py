"""kvevict_attend_static: attention for callers that cannot allocate.

Some callers cannot give the library device memory for scratch -- code that
runs while a CUDA graph is being captured (cudaMalloc cannot be captured),
hosts whose own allocator owns all device memory, serving loops that forbid
allocation on the hot path because cudaMalloc synchronises the device.  For
them kvevict_attend_static keeps its scratch in an array compiled into the
library.  These tests call it through the C ABI and check that it returns
the attention output and log-sum-exp that kvevict_decode_step returns for
the same engine state, on two calls in a row, and that a layer too large for
the built-in array is refused before any work is queued.  The file name
makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

from kv_cache_token_gb300 import Engine, KvevictError, config_from
from tests.gpu_helpers import assert_rows_close
from workloads import Workload, scaled

pytestmark = pytest.mark.gpu


def test_attend_static_matches_decode_step_twice():
    shp = scaled("h2o_70b", num_layers=1, batch=2, num_kv_heads=2, num_q_heads=16, ctx=700, steps=4,
                 budget=200, recent_window=64)
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    eng.reset()
    K, V = wl.context(0)
    eng.prefill(0, K.cuda(), V.cuda())
    for t in range(2):
        q, kn, vn, pos = wl.step(0, t)
        q, kn, vn = q.cuda(), kn.cuda(), vn.cuda()
        out_s, lse_s = eng.attend_static(0, q, kn, vn)
        torch.cuda.synchronize()
        out_s, lse_s = out_s.cpu().numpy(), lse_s.cpu().numpy()
        out, lse, _, _ = eng.decode_step(0, q, kn, vn, pos)
        torch.cuda.synchronize()
        assert_rows_close(out_s, out.cpu().numpy(), "call %d output" % t)
        assert_rows_close(lse_s[..., None], lse.cpu().numpy()[..., None], "call %d lse" % t)
    code, msg = eng.last_error()
    assert code == 0, msg


def test_attend_static_refuses_a_layer_beyond_the_array():
    # 64 lanes of group 8 need 64 * 64 * 8 * 130 * 4 B = 17 MB of split-K partials
    shp = scaled("h2o_70b", num_layers=1, batch=8, num_kv_heads=8, num_q_heads=64, ctx=64, steps=1,
                 budget=32, recent_window=8)
    eng = Engine(config_from(shp))
    eng.reset()
    q = torch.zeros((8, 64, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((8, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(KvevictError) as err:
        eng.attend_static(0, q, kv, kv)
    assert err.value.code == 10

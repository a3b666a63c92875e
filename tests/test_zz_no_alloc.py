"""kvevict_attend_static: attention for callers that cannot allocate.

Some callers cannot give the library device memory for scratch -- code that
runs while a CUDA graph is being captured (cudaMalloc cannot be captured),
hosts whose own allocator owns all device memory, serving loops that forbid
allocation on the hot path because cudaMalloc synchronises the device.  For
them kvevict_attend_static keeps its scratch in an array compiled into the
library.  These tests call it through the C ABI and check, on two calls in a
row, that it returns the attention output and log-sum-exp of the oracle's
decode attention and of kvevict_decode_step for the same engine state: on
the bf16 tensor-core path (group 8, d=128) and on the fp32 path of the H2O
toy workload (d=64, several 128-token chunks per lane); and that a layer too
large for the built-in array is refused before any work is queued.  The file
name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

from kv_cache_token_gb300 import Engine, KvevictError, config_from
from oracle.attention import decode_attention
from tests.gpu_helpers import assert_rows_close
from workloads import Workload, scaled

pytestmark = pytest.mark.gpu


def oracle_attention(eng, shp, q, kn, vn):
    """The oracle's decode attention of every lane over the engine's kept
    tokens (read back from the engine's tables) and the new token."""
    torch.cuda.synchronize()
    g, d = shp.group, shp.head_dim
    counts = eng.counts[0].cpu().numpy()
    slots = eng.slots[0].cpu().numpy()
    Kp = eng.k_pool[0].double().cpu().numpy().reshape(-1, d)
    Vp = eng.v_pool[0].double().cpu().numpy().reshape(-1, d)
    out = np.zeros((shp.batch, shp.num_q_heads, d))
    lse = np.zeros((shp.batch, shp.num_q_heads))
    for lane in range(eng.lanes):
        b, h = divmod(lane, shp.num_kv_heads)
        s = slots[lane, :int(counts[lane])]
        Ka = np.vstack([Kp[s], kn[b, h].double().numpy()[None]])
        Va = np.vstack([Vp[s], vn[b, h].double().numpy()[None]])
        o, ls, _ = decode_attention(q[b, h * g:(h + 1) * g].double().numpy(), Ka, Va)
        out[b, h * g:(h + 1) * g] = o
        lse[b, h * g:(h + 1) * g] = ls
    return out, lse


def check_two_calls(shp):
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    eng.reset()
    K, V = wl.context(0)
    eng.prefill(0, K.cuda(), V.cuda())
    for t in range(2):
        q, kn, vn, pos = wl.step(0, t)
        ref_out, ref_lse = oracle_attention(eng, shp, q, kn, vn)
        qc, knc, vnc = q.cuda(), kn.cuda(), vn.cuda()
        out_s, lse_s = eng.attend_static(0, qc, knc, vnc)
        torch.cuda.synchronize()
        out_s, lse_s = out_s.cpu().numpy(), lse_s.cpu().numpy()
        assert_rows_close(out_s, ref_out, "call %d output against the oracle" % t)
        assert_rows_close(lse_s[..., None], ref_lse[..., None], "call %d lse against the oracle" % t)
        out, lse, _, _ = eng.decode_step(0, qc, knc, vnc, pos)
        torch.cuda.synchronize()
        assert_rows_close(out_s, out.cpu().numpy(), "call %d output against kvevict_decode_step" % t)
        assert_rows_close(lse_s[..., None], lse.cpu().numpy()[..., None], "call %d lse against decode_step" % t)
    code, msg = eng.last_error()
    assert code == 0, msg


def test_attend_static_bf16_group8_twice():
    check_two_calls(scaled("h2o_70b", num_layers=1, batch=2, num_kv_heads=2, num_q_heads=16, ctx=700, steps=4,
                           budget=200, recent_window=64))


def test_attend_static_fp32_toy_twice():
    """The fp32 path (one chunk of 128 tokens per CTA, chunk 0 writing the
    segment count) on the H2O toy workload's shape: d=64, one head per lane,
    here three lanes of a 512-token prompt."""
    check_two_calls(scaled("h2o_toy", batch=3, steps=4, budget=600, recent_window=64))


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

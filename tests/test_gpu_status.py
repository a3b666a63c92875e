"""Device-side failure reporting, exercised without faulting anything: the
status word that kernels set instead of trapping, read and cleared by
kvevict_last_error, and the context staying usable afterwards.

* a bounded wait whose barrier nothing completes gives up and reports a
  timeout (the path every producer/consumer wait of the library takes);
* a decode step whose new position does not follow the lane's last one is
  refused on the device and changes no state;
* an admission that finds no free block drops that token and reports the
  exhausted pool."""
import numpy as np
import pytest
import torch

from kv_cache_token_gb300 import Engine, config_from
from tests.gpu_helpers import (assert_rows_close, compare_states, gpu_state, make_pair, oracle_state,
                               prefill_both, victim_lists)
from workloads import Workload, scaled

pytestmark = pytest.mark.gpu

E_TIMEOUT, E_DEVICE = 8, 9


def small_h2o():
    return scaled("h2o_70b", num_layers=1, batch=1, num_kv_heads=2, num_q_heads=16, ctx=300, steps=6,
                  budget=120, recent_window=40)


def test_bounded_wait_timeout_is_reported_and_cleared():
    shp = small_h2o()
    wl = Workload(shp)
    eng, orc = make_pair(shp)
    prefill_both(eng, orc, wl, 0)
    eng.check_wait_timeout(1000)
    code, msg = eng.last_error()
    assert code == E_TIMEOUT and "bounded wait" in msg, (code, msg)
    assert eng.last_error()[0] == 0          # read clears it
    q, kn, vn, pos = wl.step(0, 0)
    out, lse, vic, nv = eng.decode_step(0, q.cuda(), kn.cuda(), vn.cuda(), pos)
    ref = orc.decode_step(0, q.double().numpy(), kn.double().numpy(), vn.double().numpy(), pos)
    torch.cuda.synchronize()
    assert_rows_close(out.cpu().numpy(), ref["out"], "out after the timeout")
    compare_states(gpu_state(eng, 0), oracle_state(orc, 0), shp.policy, "after the timeout")
    assert eng.last_error()[0] == 0


def test_non_increasing_position_is_refused_on_the_device():
    shp = small_h2o()
    wl = Workload(shp)
    eng, orc = make_pair(shp)
    prefill_both(eng, orc, wl, 0)
    for t in range(2):
        q, kn, vn, pos = wl.step(0, t)
        eng.decode_step(0, q.cuda(), kn.cuda(), vn.cuda(), pos)
        orc.decode_step(0, q.double().numpy(), kn.double().numpy(), vn.double().numpy(), pos)
    before = gpu_state(eng, 0)
    q, kn, vn, pos = wl.step(0, 2)
    _, _, vic, nv = eng.decode_step(0, q.cuda(), kn.cuda(), vn.cuda(), pos - 1)   # repeats the last position
    torch.cuda.synchronize()
    assert int(nv.sum()) == 0
    code, msg = eng.last_error()
    assert code == E_DEVICE and "position" in msg, (code, msg)
    compare_states(gpu_state(eng, 0), oracle_state(orc, 0), shp.policy, "after the refused step")
    for a, b in zip(before["lanes"], gpu_state(eng, 0)["lanes"]):
        np.testing.assert_array_equal(a["score"], b["score"])
    # the proper step still runs
    out, lse, vic, nv = eng.decode_step(0, q.cuda(), kn.cuda(), vn.cuda(), pos)
    ref = orc.decode_step(0, q.double().numpy(), kn.double().numpy(), vn.double().numpy(), pos)
    torch.cuda.synchronize()
    assert_rows_close(out.cpu().numpy(), ref["out"], "out")
    for l, v in enumerate(victim_lists(nv, vic)):
        np.testing.assert_array_equal(v, ref["victims"][l])
    compare_states(gpu_state(eng, 0), oracle_state(orc, 0), shp.policy, "after the proper step")
    assert eng.last_error()[0] == 0


def test_exhausted_pool_drops_the_admission_and_reports_it():
    """Two lanes of 64 prompt tokens fill an 8-block pool exactly; the next
    token of each lane needs a fresh block (the budget is not reached, so
    nothing is evicted) and there is none."""
    shp = scaled("h2o_70b", num_layers=1, batch=1, num_kv_heads=2, num_q_heads=16, ctx=64, steps=4,
                 budget=200, recent_window=40)
    eng = Engine(config_from(shp, blocks_per_pool=8))
    eng.reset()
    wl = Workload(shp)
    K, V = wl.context(0)
    eng.prefill(0, K.cuda(), V.cuda())
    torch.cuda.synchronize()
    assert eng.last_error()[0] == 0
    pool_k = eng.k_pool[0].clone()
    q, kn, vn, pos = wl.step(0, 0)
    eng.decode_step(0, q.cuda(), kn.cuda(), vn.cuda(), pos)
    torch.cuda.synchronize()
    code, msg = eng.last_error()
    assert code == E_DEVICE and "pool exhausted" in msg, (code, msg)
    st = gpu_state(eng, 0)
    np.testing.assert_array_equal(st["counts"], [64, 64])     # the new tokens were not stored
    for lane in st["lanes"]:
        np.testing.assert_array_equal(lane["pos"], np.arange(64))
    assert torch.equal(pool_k, eng.k_pool[0])
    assert (st["owner"] >= 0).all()

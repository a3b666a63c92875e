"""SnapKV window sums taken exactly as the page fixes them: float64 sums of
the float32 history in slot order 0 upward (SnapKV, "How it works" and
"Complexity").  Both sides are given the same float32 history rows; a null
query step then evicts on those rows alone, so the victims must agree
exactly, ties of the last bit included."""
import numpy as np
import pytest
import torch

from tests.gpu_helpers import compare_states, gpu_state, make_pair, oracle_state, prefill_both, victim_lists
from workloads import Workload, scaled

pytestmark = pytest.mark.gpu

TINY = np.float32(2.0 ** -53)


def crafted_rows(rng, n, W):
    """History rows of several kinds: narrow exponent spread (summed exactly
    by integers on the GPU), wide spread (float64 rounding depends on the
    order), subnormals, zeros, and infinities."""
    kinds = rng.integers(0, 6, size=n)
    hist = np.zeros((n, W), np.float32)
    for i, kd in enumerate(kinds):
        if kd == 0:
            hist[i] = rng.uniform(1e-3, 1.0, W).astype(np.float32)
        elif kd == 1:      # one large weight and many below its last bit
            hist[i] = TINY
            hist[i, rng.integers(0, W)] = 1.0
        elif kd == 2:
            hist[i] = (2.0 ** rng.uniform(-60, 0, W)).astype(np.float32)
        elif kd == 3:
            hist[i] = np.float32(1e-40) * rng.integers(1, 100, W).astype(np.float32)
        elif kd == 4:
            pass           # an empty history
        else:
            hist[i] = rng.uniform(0.0, 2.0, W).astype(np.float32)
            if rng.random() < 0.2:
                hist[i, rng.integers(0, W)] = np.inf
    return hist


def set_history(eng, orc, layer, make):
    """Give every lane's kept tokens the same float32 rows on both sides."""
    PL = orc.layers[layer]
    for lane, L in enumerate(PL.lanes):
        n = L.pos.size
        hist = make(lane, n)
        L.hist[:] = hist
        slots = eng.slots[layer][lane, :n].long()
        eng.ring[layer][slots] = torch.from_numpy(hist).cuda()
    torch.cuda.synchronize()


def null_step(eng, orc, wl, layer, t):
    q, kn, vn, pos = wl.step(layer, t)
    _, _, vic, nv = eng.decode_step(layer, None, kn.cuda(), vn.cuda(), pos)
    ref = orc.decode_step(layer, None, kn.double().numpy(), vn.double().numpy(), pos)
    got = victim_lists(nv, vic)
    for lane in range(eng.lanes):
        np.testing.assert_array_equal(got[lane], ref["victims"][lane], err_msg="step %d lane %d" % (t, lane))
    compare_states(gpu_state(eng, layer), oracle_state(orc, layer), 1, "step %d" % t)


@pytest.mark.parametrize("pool_kernel", [1, 3])
def test_window_sums_in_slot_order(pool_kernel):
    shp = scaled("snapkv_decode", batch=1, num_kv_heads=2, num_q_heads=8, ctx=300, steps=4,
                 budget=200, recent_window=20, obs_window=32, pool_kernel=pool_kernel)
    wl = Workload(shp)
    eng, orc = make_pair(shp, layers=[0])
    prefill_both(eng, orc, wl, 0)
    rng = np.random.default_rng(11 + pool_kernel)
    W = shp.obs_window

    # step 0: 101 victims among rows of every kind
    set_history(eng, orc, 0, lambda lane, n: crafted_rows(rng, n, W))
    null_step(eng, orc, wl, 0, 0)

    # step 1: one victim decided in the last bit.  A = [1, tiny x 31] sums to
    # 1 in slot order (each tiny add rounds away); B holds the same values
    # with the 1 last and sums to 1 + 31 tiny, rounded up.  Exact or
    # reordered sums would tie them and evict B, the lower position.
    def last_bit(lane, n):
        hist = np.full((n, W), 2.0, np.float32)
        b, a = 10 + lane, 50 + lane
        hist[b] = TINY
        hist[b, W - 1] = 1.0
        hist[a] = TINY
        hist[a, 0] = 1.0
        return hist
    set_history(eng, orc, 0, last_bit)
    null_step(eng, orc, wl, 0, 1)
    assert eng.last_error()[0] == 0

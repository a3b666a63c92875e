"""Bottom-k selection on given keys: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

from kv_cache_token_gb300 import Engine, config_from
from oracle.engine import select as oracle_select
from workloads import scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eng():
    shp = scaled("h2o_70b", num_layers=1, batch=1, num_kv_heads=1, num_q_heads=8, ctx=64, steps=0,
                 budget=32, recent_window=8)
    return Engine(config_from(shp))


def _run(eng, keys, pos, counts, budget, R):
    kt = torch.tensor(keys).cuda()
    pt = torch.tensor(pos, dtype=torch.int32).cuda()
    ct = torch.tensor(counts, dtype=torch.int32).cuda()
    v, nv = eng.select(kt, pt, ct, budget, R)
    torch.cuda.synchronize()
    got = [v[l, :int(nv[l])].cpu().numpy() for l in range(len(counts))]
    ref = oracle_select(keys, pos, counts, budget, R)
    for l in range(len(counts)):
        np.testing.assert_array_equal(got[l], ref[l], err_msg="lane %d" % l)


@pytest.mark.parametrize("dtype,lanes,stride", [(np.float32, 37, 3000), (np.float64, 37, 3000),
                                                (np.float32, 8, 70000)])
def test_random_with_ties(eng, dtype, lanes, stride):
    """Ties, NaN, -0 and tiny keys; 70,000-entry tables take the 16-CTA
    cluster path (64K entries and more), the others the 8-CTA one."""
    rng = np.random.default_rng(11)
    keys = np.zeros((lanes, stride), dtype)
    pos = np.zeros((lanes, stride), np.int32)
    counts = rng.integers(0, stride + 1, lanes)
    counts[0], counts[1], counts[2] = 0, 1, stride
    for l in range(lanes):
        kind = l % 4
        if kind == 0:
            keys[l] = rng.standard_normal(stride)
        elif kind == 1:
            keys[l] = rng.integers(0, 5, stride)          # heavy ties
        elif kind == 2:
            keys[l] = rng.random(stride) * 1e-30          # tiny values
        else:
            keys[l] = np.where(rng.random(stride) < 0.1, np.nan, rng.standard_normal(stride))
            keys[l, ::7] = -0.0
            keys[l, 3::7] = 0.0
        pos[l] = np.sort(rng.choice(10 * stride, stride, replace=False))
    for budget, R in [(100, 10), (stride - 1, 1), (500, 50), (10, 3)]:
        _run(eng, keys, pos, counts, budget, R)


def test_large_lane_and_k_one(eng):
    rng = np.random.default_rng(12)
    stride = 131072
    keys = rng.standard_normal((2, stride)).astype(np.float32)
    pos = np.tile(np.arange(stride, dtype=np.int32), (2, 1))
    counts = np.array([stride, stride - 77])
    _run(eng, keys, pos, counts, 6553, 64)
    _run(eng, keys, pos, counts, stride - 1, 64)       # k = 1 (or 0)
    keys[:] = 1.0                                        # all tied: oldest candidates go
    _run(eng, keys, pos, counts, 6553, 64)

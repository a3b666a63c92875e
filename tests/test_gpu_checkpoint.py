"""Checkpoint and resume: every piece of engine state lives in the caller's
buffers (K/V pools, token tables, scores, history ring and its slot, block
owners and masks, lane block lists, counters), so saving those tensors and
copying them into a freshly created engine resumes decoding exactly: the
two engines then produce bit-identical outputs, victims and state."""
import pytest
import torch

from kv_cache_token_gb300 import Engine, config_from
from workloads import Workload, scaled

pytestmark = pytest.mark.gpu

STATE = ("k_pool", "v_pool", "positions", "slots", "counts", "scores", "ring", "ring_slot", "block_owner",
         "block_mask", "lane_blocks", "lane_nblocks", "stats_buf")


def bits(t):
    return t.view({2: torch.int16, 4: torch.int32, 8: torch.int64}[t.element_size()])


@pytest.mark.parametrize("name,kw", [
    ("snapkv_decode", dict(batch=2, num_kv_heads=2, num_q_heads=8, ctx=700, steps=10, budget=200,
                           recent_window=40, obs_window=8, pool_kernel=5)),
    ("h2o_70b", dict(num_layers=2, batch=2, num_kv_heads=2, num_q_heads=16, ctx=900, steps=10, budget=300,
                     recent_window=100)),
])
def test_resume_from_saved_state_buffers(name, kw):
    shp = scaled(name, **kw)
    wl = Workload(shp)
    a = Engine(config_from(shp))
    a.reset()
    layers = range(shp.num_layers)
    for layer in layers:
        K, V = wl.context(layer)
        a.prefill(layer, K.cuda(), V.cuda())

    def step(eng, t, layer):
        q, kn, vn, pos = wl.step(layer, t)
        out, lse, vic, nv = eng.decode_step(layer, q.cuda(), kn.cuda(), vn.cuda(), pos,
                                            victims=torch.zeros_like(eng.victims),
                                            n_victims=torch.zeros_like(eng.n_victims))
        return out, lse, vic, nv

    for t in range(4):                   # mass eviction at step 0, then steady steps
        for layer in layers:
            step(a, t, layer)
    torch.cuda.synchronize()
    saved = {k: getattr(a, k).cpu().clone() for k in STATE if getattr(a, k) is not None}   # the checkpoint
    b = Engine(config_from(shp))
    b.reset()
    for k, v in saved.items():
        getattr(b, k).copy_(v)
    torch.cuda.synchronize()
    for t in range(4, shp.steps):
        for layer in layers:
            ra = step(a, t, layer)
            rb = step(b, t, layer)
            torch.cuda.synchronize()
            assert torch.equal(bits(ra[0]), bits(rb[0])) and torch.equal(bits(ra[1]), bits(rb[1])), (t, layer)
            assert torch.equal(ra[3], rb[3]), (t, layer)
            for l in range(a.lanes):
                n = int(ra[3][l])
                assert torch.equal(ra[2][l, :n], rb[2][l, :n]), (t, layer, l)
    for k in saved:
        # raw bit patterns: never-written pool rows may hold NaN patterns
        assert torch.equal(bits(getattr(a, k)), bits(getattr(b, k))), k
    assert a.last_error()[0] == 0 and b.last_error()[0] == 0

"""Forced compaction: freed block ids, move tuples and the resulting tables
bit-exact against the oracle (vToken invariants I1, I2, I4 hold on both)."""
import numpy as np
import pytest
import torch

from tests.gpu_helpers import compare_states, gpu_state, make_pair, oracle_state, prefill_both
from workloads import Workload, scaled

pytestmark = pytest.mark.gpu


def _victims(orc, layer, frac, rng, lanes, cap, protect):
    vic = np.zeros((lanes, cap), np.int32)
    nv = np.zeros(lanes, np.int32)
    lists = []
    for l in range(lanes):
        pos = orc.layers[layer].lanes[l].pos
        cand = pos[:-protect] if protect else pos
        k = int(frac * cand.size)
        v = np.sort(rng.choice(cand, k, replace=False)) if k else np.zeros(0, np.int64)
        vic[l, :k] = v
        nv[l] = k
        lists.append(v)
    return vic, nv, lists


@pytest.mark.parametrize("frac", [0.95, 0.5, 0.0])
def test_compact_matches_oracle(frac):
    rng = np.random.default_rng(21)
    shp = scaled("paged_128k", ctx=3000, num_kv_heads=3, num_q_heads=12, budget=150, recent_window=16)
    wl = Workload(shp)
    eng, orc = make_pair(shp)
    prefill_both(eng, orc, wl, 0)
    vic, nv, lists = _victims(orc, 0, frac, rng, eng.lanes, shp.max_tokens, 16)
    freed, n_freed, moves, n_moves = eng.compact(0, torch.tensor(vic).cuda(), torch.tensor(nv).cuda())
    ref = orc.compact(0, lists)
    torch.cuda.synchronize()
    nf, nm = int(n_freed.item()), int(n_moves.item())
    np.testing.assert_array_equal(freed[:nf].cpu().numpy(), np.array(ref["freed"], np.int32))
    got_moves = [tuple(r) for r in moves[:nm].cpu().numpy().tolist()]
    assert got_moves == [tuple(int(x) for x in m) for m in ref["moves"]]
    compare_states(gpu_state(eng, 0), oracle_state(orc, 0), shp.policy, "after compaction")
    st = eng.stats(0).cpu().numpy()
    N, live, F, half = orc.layers[0].stats()
    assert (st[9], st[10], st[11]) == (N, live, half)
    assert eng.last_error()[0] == 0


def test_compact_defers_when_pool_is_short():
    """With no headroom the relocation plans are deferred, dead blocks still
    return to the pool, and the call reports no moves."""
    rng = np.random.default_rng(22)
    shp = scaled("paged_128k", ctx=800, num_kv_heads=2, num_q_heads=8, budget=40, recent_window=8)
    import dataclasses
    shp = dataclasses.replace(shp)
    wl = Workload(shp)
    from kv_cache_token_gb300 import Engine, config_from
    from oracle.engine import Engine as Oracle
    blocks = 2 * 50            # exactly the prompt: no free block left for destinations
    cfg = config_from(shp, blocks_per_pool=blocks)
    eng = Engine(cfg)
    eng.reset()

    class S:
        pass
    oc = S()
    for k in ("policy", "num_layers", "batch", "num_q_heads", "num_kv_heads", "head_dim", "budget",
              "recent_window", "obs_window", "pool_kernel", "theta_f"):
        setattr(oc, k, getattr(shp, k))
    oc.blocks_per_pool = blocks
    orc = Oracle(oc)
    prefill_both(eng, orc, wl, 0)
    vic, nv, lists = _victims(orc, 0, 0.3, rng, eng.lanes, shp.max_tokens, 8)
    freed, n_freed, moves, n_moves = eng.compact(0, torch.tensor(vic).cuda(), torch.tensor(nv).cuda())
    ref = orc.compact(0, lists)
    torch.cuda.synchronize()
    assert ref["deferred"]
    assert int(n_moves.item()) == 0
    np.testing.assert_array_equal(freed[:int(n_freed.item())].cpu().numpy(), np.array(ref["freed"], np.int32))
    compare_states(gpu_state(eng, 0), oracle_state(orc, 0), shp.policy, "deferred")
    assert int(eng.stats(0)[7].item()) == 1

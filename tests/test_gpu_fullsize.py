"""Parity at the workloads' full sizes, in the launch configuration the bench
uses, on outputs the oracle can compute one by one: sampled lanes of the
70B-shaped H2O layer and of the SnapKV workload (each sampled lane runs in a
one-lane oracle; block ids differ there, everything per lane must match),
sampled tokens of the 32K and 128K DropKV window scores, and the full 128K
compaction with seeded victim lists (bit-exact)."""
import dataclasses
import types

import numpy as np
import pytest
import torch

from kv_cache_token_gb300 import Engine, config_from
from oracle.engine import Engine as Oracle
from tests.gpu_helpers import (assert_rows_close, assert_scores_close, compare_states, count_tie_swaps,
                               gpu_state, near_tie, oracle_state, victim_lists)
from workloads import Workload, shape

pytestmark = pytest.mark.gpu


def lane_oracle(shp, K, V):
    """A one-lane oracle engine holding the given lane's prompt."""
    per_lane = -(-shp.max_tokens // 16) + -(-shp.budget // 16) + 2
    cfg = types.SimpleNamespace(policy=shp.policy, num_layers=1, batch=1, num_q_heads=shp.group,
                                num_kv_heads=1, head_dim=shp.head_dim, blocks_per_pool=per_lane,
                                budget=shp.budget, recent_window=shp.recent_window,
                                obs_window=shp.obs_window, pool_kernel=shp.pool_kernel,
                                theta_f=float(np.float32(shp.theta_f)))
    o = Oracle(cfg)
    o.prefill(0, K[None, None], V[None, None])
    return o


def run_sampled_decode(shp, lanes, steps):
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    eng.reset()
    K, V = wl.context(0, device="cuda")
    eng.prefill(0, K, V)
    g = shp.group
    orcs = {}
    for lane in lanes:
        b, h = divmod(lane, shp.num_kv_heads)
        orcs[lane] = lane_oracle(shp, K[b, h].double().cpu().numpy(), V[b, h].double().cpu().numpy())
    del K, V
    live = set(lanes)
    swaps = 0
    for t in range(steps):
        q, kn, vn, pos = wl.step(0, t, device="cuda")
        out, lse, vic, nv = eng.decode_step(0, q, kn, vn, pos)
        torch.cuda.synchronize()
        got_v = victim_lists(nv, vic)
        o_np, l_np = out.cpu().numpy(), lse.cpu().numpy()
        for lane in sorted(live):
            b, h = divmod(lane, shp.num_kv_heads)
            r = orcs[lane].decode_step(0, q[b:b + 1, h * g:(h + 1) * g].double().cpu().numpy(),
                                       kn[b:b + 1, h:h + 1].double().cpu().numpy(),
                                       vn[b:b + 1, h:h + 1].double().cpu().numpy(), pos)
            assert_rows_close(o_np[b, h * g:(h + 1) * g], r["out"][0], "step %d lane %d out" % (t, lane))
            assert_rows_close(l_np[b, h * g:(h + 1) * g, None], r["lse"][0][:, None], "step %d lane %d lse" % (t, lane))
            if not np.array_equal(got_v[lane], r["victims"][0]):
                assert near_tie(r["keys"][0], r["pos"][0], got_v[lane], r["victims"][0]), \
                    "step %d lane %d victims differ beyond a tie" % (t, lane)
                swaps += 1
                live.discard(lane)          # the trajectories part here; stop following this lane
                continue
            L = orcs[lane].layers[0].lanes[0]
            n = int(eng.counts[0, lane].item())
            np.testing.assert_array_equal(eng.positions[0, lane, :n].cpu().numpy(), L.pos,
                                          err_msg="step %d lane %d kept positions" % (t, lane))
            if shp.policy == 0:
                assert_scores_close(eng.scores[0, lane, :n].cpu().numpy(), L.score, "step %d lane %d scores" % (t, lane))
            else:
                slots = eng.slots[0, lane, :n].long()
                assert_scores_close(eng.ring[0][slots].cpu().numpy().ravel(), L.hist.ravel(),
                                    "step %d lane %d history" % (t, lane))
    assert eng.last_error()[0] == 0
    print("NEAR-TIE swaps, %s: %d of %d sampled lanes over %d steps" % (shp.name, swaps, len(lanes), steps))
    assert swaps <= 1, "near-tie swaps: %d" % swaps
    return swaps


def test_h2o_70b_layer_full_size():
    """One layer of the 70B-shaped workload: 16 x 8 lanes, 16384-token
    prompts, group 8, budget 3276; mass eviction then steady state."""
    shp = dataclasses.replace(shape("h2o_70b"), num_layers=1)
    run_sampled_decode(shp, [0, 41, 86, 127], 5)


def test_snapkv_decode_full_size():
    """The SnapKV workload as specified (32 lanes, 4096-token prompts,
    obsWindow 32, poolKernel 7, budget 1024, recent 256), 64 of its 256 steps
    on sampled lanes."""
    run_sampled_decode(shape("snapkv_decode"), [0, 13, 31], 64)


@pytest.mark.parametrize("name", ["dropkv_prefill", "paged_128k"])
def test_window_scores_full_size(name):
    shp = shape(name)
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    eng.reset()
    K, V = wl.context(0, device="cuda")
    eng.prefill(0, K, V)
    q, qp = wl.window(0, device="cuda")
    lse, a, sc = eng.score(0, q, qp)
    torch.cuda.synchronize()
    rng = np.random.default_rng(31)
    g, n = shp.group, shp.ctx
    for lane in (0, 5):
        b, h = divmod(lane, shp.num_kv_heads)
        tok = np.unique(np.concatenate([rng.choice(n, 400, replace=False), np.arange(n - 80, n), [0, 1]]))
        o = lane_oracle(dataclasses.replace(shp, budget=shp.budget), K[b, h].double().cpu().numpy(),
                        V[b, h].double().cpu().numpy())
        qs = q[b:b + 1, h * g:(h + 1) * g].double().cpu().numpy()
        r = o.score(0, qs, qp.cpu().numpy(), token_idx=tok)
        assert_rows_close(lse[b, h * g:(h + 1) * g].cpu().numpy()[..., None], r["lse"][0][..., None], "lse")
        assert_rows_close(a[b, h * g:(h + 1) * g].cpu().numpy(), r["a"][0], "window outputs")
        assert_scores_close(sc[lane, tok].cpu().numpy(), r["scores"][0], "lane %d sampled scores" % lane)
    assert eng.last_error()[0] == 0


def test_paged_128k_compaction_full_size():
    """128K prompts in 8192 blocks per lane, keep floor(5%) = 6553 (the last
    64 protected), forced compaction: freed ids, moves and tables bit-exact;
    token-level against block-granular reclamation reported."""
    shp = shape("paged_128k")
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    eng.reset()
    K, V = wl.context(0, device="cuda")
    eng.prefill(0, K, V)
    Kh, Vh = K.float().cpu().numpy(), V.float().cpu().numpy()
    del K, V
    orc = Oracle(shp)
    orc.prefill(0, Kh, Vh)
    blockwise = Oracle(shp, store_kv=False)       # block-granular counterfactual
    blockwise.prefill(0, Kh, Vh)
    del Kh, Vh
    rng = np.random.default_rng(32)
    n, keep, R = shp.ctx, shp.budget, shp.recent_window
    vic = np.zeros((eng.lanes, shp.max_tokens), np.int32)
    nv = np.zeros(eng.lanes, np.int32)
    lists = []
    for lane in range(eng.lanes):
        kept = rng.choice(n - R, keep - R, replace=False)
        v = np.setdiff1d(np.arange(n - R), kept)
        vic[lane, :v.size] = v
        nv[lane] = v.size
        lists.append(v)
    freed_block_gran = sum(len(blockwise.layers[0].evict(l, lists[l])) for l in range(eng.lanes))
    Nb, live_b, Fb, half_b = blockwise.layers[0].stats()
    freed, n_freed, moves, n_moves = eng.compact(0, torch.tensor(vic).cuda(), torch.tensor(nv).cuda())
    ref = orc.compact(0, lists)
    torch.cuda.synchronize()
    nf, nm = int(n_freed.item()), int(n_moves.item())
    np.testing.assert_array_equal(freed[:nf].cpu().numpy(), np.array(ref["freed"], np.int32))
    got_moves = moves[:nm].cpu().numpy()
    np.testing.assert_array_equal(got_moves, np.array(ref["moves"], np.int32).reshape(-1, 6))
    compare_states(gpu_state(eng, 0), oracle_state(orc, 0), shp.policy, "after compaction")
    st = eng.stats(0).cpu().numpy()
    N, live, F, half = orc.layers[0].stats()
    assert (st[9], st[10], st[11]) == (N, live, half)
    # token-level reclamation frees far more blocks than block-granular eviction
    assert nf > freed_block_gran and F < Fb
    print("128K: freed token-level %d vs block-granular %d; F %.3f vs %.3f; blocks <=50%% %d vs %d"
          % (nf, freed_block_gran, F, Fb, half, half_b))
    assert eng.last_error()[0] == 0


@pytest.mark.parametrize("name", ["dropkv_prefill", "paged_128k"])
def test_victims_from_gpu_scores_full_lane(name):
    """Configurations 3 and 5 end to end on one full lane: the GPU's window
    scores of all 8 lanes, the GPU's selection to the budget on them, and
    lane 0's victim set against the oracle's selection on its float64 scores
    of the whole lane (swaps only between near-equal keys; counted)."""
    shp = shape(name)
    wl = Workload(shp)
    eng = Engine(config_from(shp))
    eng.reset()
    K, V = wl.context(0, device="cuda")
    eng.prefill(0, K, V)
    q, qp = wl.window(0, device="cuda")
    lse, a, sc = eng.score(0, q, qp)
    v, nv = eng.select(sc, eng.positions[0].contiguous(), eng.counts[0].contiguous(), shp.budget,
                       shp.recent_window)
    torch.cuda.synchronize()
    g, lane = shp.group, 0
    o = lane_oracle(shp, K[0, 0].double().cpu().numpy(), V[0, 0].double().cpu().numpy())
    del K, V
    r = o.score(0, q[0:1, 0:g].double().cpu().numpy(), qp.cpu().numpy())
    from oracle.select import select_lane
    L = o.layers[0].lanes[0]
    ref_v = select_lane(np.asarray(r["scores"][0], np.float64), L.pos, shp.budget, shp.recent_window)
    got = v[lane, :int(nv[lane])].cpu().numpy()
    assert got.size == ref_v.size == shp.ctx - shp.budget
    swaps = count_tie_swaps(r["scores"][0], L.pos, got, ref_v, "%s lane 0" % name)
    print("NEAR-TIE swaps, %s lane 0 (%d victims of %d tokens): %d" % (name, ref_v.size, shp.ctx, swaps))
    assert swaps <= 4
    assert eng.last_error()[0] == 0

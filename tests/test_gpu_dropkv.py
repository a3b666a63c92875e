"""DropKV prefill-window scoring: LSE, window outputs and per-token scores
against the oracle (causal window, ragged chunk tails, heavy-tailed keys),
then the budgeted selection and compaction on those scores."""
import numpy as np
import pytest
import torch

from tests.gpu_helpers import (assert_rows_close, assert_scores_close, compare_states, gpu_state,
                               make_pair, oracle_state, prefill_both)
from workloads import Workload, scaled

pytestmark = pytest.mark.gpu


def run_score(shp):
    wl = Workload(shp)
    eng, orc = make_pair(shp)
    prefill_both(eng, orc, wl, 0)
    q, qp = wl.window(0)
    lse, a, sc = eng.score(0, q.cuda(), qp.cuda())
    ref = orc.score(0, q.double().numpy(), qp.numpy())
    torch.cuda.synchronize()
    assert_rows_close(lse.cpu().numpy()[..., None], ref["lse"][..., None], "lse")
    assert_rows_close(a.cpu().numpy(), ref["a"], "window outputs")
    for l in range(eng.lanes):
        n = shp.ctx
        assert_scores_close(sc[l, :n].cpu().numpy(), ref["scores"][l], "lane %d scores" % l)
    return eng, orc, sc, ref


def test_window_scores_scaled():
    shp = scaled("dropkv_prefill", ctx=3000, num_kv_heads=2, num_q_heads=8)
    run_score(shp)


def test_window_scores_many_rows():
    """384 window rows per lane (group 8 x 48 positions): more rows than the
    two 128-row tensor-memory tiles, so the general kernel scores them."""
    shp = scaled("dropkv_prefill", ctx=1500, num_kv_heads=2, num_q_heads=16, window=48, budget=80,
                 recent_window=48)
    run_score(shp)


def test_window_scores_single_partial_tile():
    """A lane shorter than one 64-key tile, with window rows before every key."""
    shp = scaled("dropkv_prefill", ctx=40, num_kv_heads=1, num_q_heads=4, window=16, budget=20,
                 recent_window=16)
    run_score(shp)


def test_window_scores_short_window_group8():
    shp = scaled("dropkv_prefill", ctx=2100, num_kv_heads=1, num_q_heads=8, window=20, budget=105,
                 recent_window=20)
    run_score(shp)


def test_null_window_is_inert():
    shp = scaled("dropkv_prefill", ctx=300, num_kv_heads=1, num_q_heads=4, window=8, budget=30,
                 recent_window=8)
    wl = Workload(shp)
    eng, orc = make_pair(shp)
    prefill_both(eng, orc, wl, 0)
    before = eng.scores.clone()
    assert eng.score(0, None, None) is None
    torch.cuda.synchronize()
    assert torch.equal(before, eng.scores)


def test_score_select_compact_pipeline():
    """The paged-128K flow at small size: score, keep 5%, compact."""
    shp = scaled("paged_128k", ctx=4000, num_kv_heads=2, num_q_heads=8, budget=200, recent_window=64)
    eng, orc, sc, ref = run_score(shp)
    C = shp.max_tokens
    pos = eng.positions[0].contiguous()
    keys = torch.tensor(np.stack([ref["scores"][l] for l in range(eng.lanes)]).astype(np.float32))
    kfull = torch.zeros((eng.lanes, C), dtype=torch.float32)
    kfull[:, :shp.ctx] = keys
    v, nv = eng.select(kfull.cuda(), pos, eng.counts[0].contiguous(), shp.budget, shp.recent_window)
    torch.cuda.synchronize()
    from oracle.select import select_lane
    lists = []
    for l in range(eng.lanes):
        L = orc.layers[0].lanes[l]
        r = select_lane(kfull[l, :shp.ctx].double().numpy(), L.pos, shp.budget, shp.recent_window)
        np.testing.assert_array_equal(v[l, :int(nv[l])].cpu().numpy(), r)
        lists.append(r)
    freed, n_freed, moves, n_moves = eng.compact(0, v, nv)
    cref = orc.compact(0, lists)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(freed[:int(n_freed.item())].cpu().numpy(), np.array(cref["freed"], np.int32))
    assert int(n_moves.item()) == len(cref["moves"])
    compare_states(gpu_state(eng, 0), oracle_state(orc, 0), shp.policy, "after compaction")

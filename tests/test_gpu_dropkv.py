"""DropKV prefill-window scoring: LSE, window outputs and per-token scores
against the oracle (causal window, ragged chunk tails, heavy-tailed keys),
then the budgeted selection and compaction on those scores."""
import numpy as np
import pytest
import torch

from tests.gpu_helpers import (assert_rows_close, assert_scores_close, compare_states, count_tie_swaps,
                               gpu_state, make_pair, oracle_state, prefill_both)
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


def test_window_scores_one_row_tile():
    """128 window rows (group 4 x 32 positions): one row tile, so pass 2
    writes each key's sum itself (no second tile adds into it); the context
    spans several chunks and ends in a ragged tile."""
    shp = scaled("dropkv_prefill", ctx=5001, num_kv_heads=2, num_q_heads=8, window=32, budget=250,
                 recent_window=32)
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


def test_window_scores_scattered_slots():
    """The scores depend on each kept token's position and K/V rows, not on
    where the rows sit in the pool.  After a prefill, each lane's slots are
    permuted among themselves (K/V rows moved along): the first 128 tokens
    keep consecutive slots (whole-tile copies), the next 256 keep in-order
    16-token blocks in shuffled block order (16-row copies), the rest are
    scattered token by token (four-row gathers), with ragged ends.  The
    scores must equal the oracle's on the unpermuted tokens."""
    shp = scaled("dropkv_prefill", ctx=3000, num_kv_heads=2, num_q_heads=8)
    wl = Workload(shp)
    eng, orc = make_pair(shp)
    prefill_both(eng, orc, wl, 0)
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    n = shp.ctx
    slots = eng.slots[0].cpu().numpy()
    kp = eng.k_pool[0].reshape(-1, shp.head_dim).clone()
    vp = eng.v_pool[0].reshape(-1, shp.head_dim).clone()
    for l in range(eng.lanes):
        old = slots[l, :n].copy()
        order = np.arange(n)
        blocks = np.arange(128, 384).reshape(16, 16)
        order[128:384] = blocks[rng.permutation(16)].reshape(-1)
        order[384:] = 384 + rng.permutation(n - 384)
        new = old[order]                  # token i now lives where token order[i] lived
        src = torch.as_tensor(old, dtype=torch.long, device="cuda")
        dst = torch.as_tensor(new, dtype=torch.long, device="cuda")
        kp[dst] = eng.k_pool[0].reshape(-1, shp.head_dim)[src]
        vp[dst] = eng.v_pool[0].reshape(-1, shp.head_dim)[src]
        slots[l, :n] = new
    eng.k_pool[0].copy_(kp.reshape(eng.k_pool[0].shape))
    eng.v_pool[0].copy_(vp.reshape(eng.v_pool[0].shape))
    eng.slots[0].copy_(torch.as_tensor(slots))
    torch.cuda.synchronize()
    q, qp = wl.window(0)
    lse, a, sc = eng.score(0, q.cuda(), qp.cuda())
    ref = orc.score(0, q.double().numpy(), qp.numpy())
    torch.cuda.synchronize()
    assert_rows_close(lse.cpu().numpy()[..., None], ref["lse"][..., None], "lse")
    assert_rows_close(a.cpu().numpy(), ref["a"], "window outputs")
    for l in range(eng.lanes):
        assert_scores_close(sc[l, :n].cpu().numpy(), ref["scores"][l], "lane %d scores" % l)
    code, msg = eng.last_error()
    assert code == 0, msg


def test_victims_from_gpu_scores_end_to_end():
    """The whole chain on the GPU (window scores, then the budgeted selection
    on those scores) against the oracle's selection on its own float64
    scores: the victim sets are equal except for swaps between tokens whose
    oracle keys are within the score tolerance of the threshold (DropKV
    explainer: drop the k lowest-scoring tokens); the swap count is printed
    and bounded."""
    shp = scaled("dropkv_prefill", ctx=6000, num_kv_heads=2, num_q_heads=8, budget=300, recent_window=64)
    eng, orc, sc, ref = run_score(shp)
    v, nv = eng.select(sc, eng.positions[0].contiguous(), eng.counts[0].contiguous(), shp.budget,
                       shp.recent_window)
    torch.cuda.synchronize()
    from oracle.select import select_lane
    swaps = 0
    for l in range(eng.lanes):
        L = orc.layers[0].lanes[l]
        r = select_lane(np.asarray(ref["scores"][l], np.float64), L.pos, shp.budget, shp.recent_window)
        got = v[l, :int(nv[l])].cpu().numpy()
        swaps += count_tie_swaps(ref["scores"][l], L.pos, got, r, "lane %d" % l)
    print("NEAR-TIE swaps, DropKV window scoring + selection (6000 tokens x %d lanes): %d" % (eng.lanes, swaps))
    assert swaps <= 2

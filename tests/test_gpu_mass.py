"""Prefill-window attention mass (kvevict_score_mass) against the oracle:
SnapKV's one-shot prefill keys (causal window sums, pooled over kept
neighbours) and H2O's causal-prefill scores (rows strictly after each token),
on the tensor-memory path (<= 256 rows per lane) and the general path (more
rows), with ragged tails; then the SnapKV prefill selection and compaction."""
import dataclasses

import numpy as np
import pytest
import torch

from tests.gpu_helpers import (assert_rows_close, assert_scores_close, compare_states, gpu_state,
                               make_pair, oracle_state, prefill_both)
from workloads import Workload, scaled

pytestmark = pytest.mark.gpu

SNAP, H2O_KIND = 0, 1          # kvevict_mass_kind
ORACLE_KIND = {SNAP: 1, H2O_KIND: 0}   # the oracle names the kinds by policy


def run_mass(shp, kind, lanes=None):
    wl = Workload(shp)
    eng, orc = make_pair(shp)
    prefill_both(eng, orc, wl, 0)
    q, qp = wl.window(0)
    lse, sc = eng.score_mass(0, q.cuda(), qp.cuda(), kind)
    ref = orc.score_mass(0, q.double().numpy(), qp.numpy(), ORACLE_KIND[kind], lanes=lanes)
    torch.cuda.synchronize()
    check = range(eng.lanes) if lanes is None else lanes
    for l in check:
        b, h = divmod(l, shp.num_kv_heads)
        g = shp.group
        assert_rows_close(lse[b, h * g:(h + 1) * g].cpu().numpy()[..., None],
                          ref["lse"][b, h * g:(h + 1) * g][..., None], "lse lane %d" % l)
        assert_scores_close(sc[l, :shp.ctx].cpu().numpy(), ref["scores"][l], "lane %d mass" % l)
    code, msg = eng.last_error()
    assert code == 0, msg
    return eng, orc, sc, ref


def test_snapkv_prefill_keys_tensor_memory_path():
    """128 rows per lane (group 4 x window 32), poolKernel 7, ragged tail."""
    run_mass(scaled("snapkv_prefill", ctx=3000, num_kv_heads=2, num_q_heads=8, budget=200), SNAP)


def test_snapkv_prefill_keys_general_path():
    """384 rows per lane (group 8 x window 48): the warp-level path."""
    run_mass(scaled("snapkv_prefill", ctx=1500, num_kv_heads=2, num_q_heads=16, window=48, budget=200,
                    recent_window=48), SNAP)


def test_snapkv_prefill_keys_no_pooling_and_wide_pool():
    """poolKernel 1 (the sums themselves) and 31 (the largest the
    configuration accepts), on a lane shorter than one 64-key tile and on one
    whose pooling halo crosses the 1024-entry tiles of the pooling kernel."""
    for ctx, pk in ((40, 1), (40, 31), (2100, 31)):
        shp = scaled("snapkv_prefill", ctx=ctx, num_kv_heads=1, num_q_heads=4, window=16, budget=30,
                     recent_window=16, pool_kernel=pk)
        run_mass(shp, SNAP)


def test_h2o_prefill_scores_window():
    """H2O kind, tensor-memory path: rows strictly after each token."""
    shp = scaled("snapkv_prefill", ctx=2100, num_kv_heads=1, num_q_heads=8, window=20, budget=105,
                 recent_window=20)
    run_mass(dataclasses.replace(shp, policy=0), H2O_KIND)


def test_h2o_prefill_scores_whole_prompt():
    """H2O kind over every prompt position (the score equation's S_j after
    a 512-token prompt, one head): 512 rows, the general path."""
    shp = scaled("snapkv_prefill", ctx=512, num_kv_heads=1, num_q_heads=1, window=512, budget=128,
                 recent_window=64)
    shp = dataclasses.replace(shp, policy=0)
    wl = Workload(shp)
    eng, orc = make_pair(shp)
    prefill_both(eng, orc, wl, 0)
    qfull, _ = wl.window(0)
    qp = torch.arange(0, 512, dtype=torch.int32)
    # the layer's own score table as the output: H2O decoding starts from it
    lse, sc = eng.score_mass(0, qfull.cuda(), qp.cuda(), H2O_KIND, scores=eng.scores[0])
    ref = orc.score_mass(0, qfull.double().numpy(), qp.numpy(), 0)
    torch.cuda.synchronize()
    assert sc.data_ptr() == eng.scores[0].data_ptr()
    assert_scores_close(eng.scores[0][0, :512].cpu().numpy(), ref["scores"][0], "whole-prompt S")
    assert_rows_close(lse[0, 0].cpu().numpy()[:, None], ref["lse"][0, 0][:, None], "lse")
    # the last token has no later row: exactly zero
    assert float(eng.scores[0][0, 511]) == 0.0


def test_mass_null_window_is_inert():
    shp = scaled("snapkv_prefill", ctx=300, num_kv_heads=1, num_q_heads=4, window=8, budget=30,
                 recent_window=8)
    wl = Workload(shp)
    eng, orc = make_pair(shp)
    prefill_both(eng, orc, wl, 0)
    before = eng.scores.clone()
    assert eng.score_mass(0, None, None, SNAP) is None
    assert eng.score_mass(0, None, None, H2O_KIND) is None
    torch.cuda.synchronize()
    assert torch.equal(before, eng.scores)


def test_snapkv_prefill_select_compact_pipeline():
    """SnapKV's one-shot prefill selection at small size: keys, keep the
    budget (window protected), compact; the selection runs on the oracle's
    keys rounded to fp32 on both sides, so it must agree bit for bit."""
    shp = scaled("snapkv_prefill", ctx=4000, num_kv_heads=2, num_q_heads=8, budget=250)
    eng, orc, sc, ref = run_mass(shp, SNAP)
    C = shp.max_tokens
    keys = torch.zeros((eng.lanes, C), dtype=torch.float32)
    for l in range(eng.lanes):
        keys[l, :shp.ctx] = torch.tensor(ref["scores"][l].astype(np.float32))
    v, nv = eng.select(keys.cuda(), eng.positions[0].contiguous(), eng.counts[0].contiguous(), shp.budget,
                       shp.recent_window)
    torch.cuda.synchronize()
    from oracle.select import select_lane
    lists = []
    for l in range(eng.lanes):
        L = orc.layers[0].lanes[l]
        r = select_lane(keys[l, :shp.ctx].double().numpy(), L.pos, shp.budget, shp.recent_window)
        np.testing.assert_array_equal(v[l, :int(nv[l])].cpu().numpy(), r)
        assert r.size == shp.ctx - shp.budget
        lists.append(r)
    freed, n_freed, moves, n_moves = eng.compact(0, v, nv)
    cref = orc.compact(0, lists)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(freed[:int(n_freed.item())].cpu().numpy(), np.array(cref["freed"], np.int32))
    assert int(n_moves.item()) == len(cref["moves"])
    compare_states(gpu_state(eng, 0), oracle_state(orc, 0), shp.policy, "after compaction")


def test_snapkv_prefill_keys_full_32k_sampled_lanes():
    """The 32K SnapKV prefill workload at full size, two lanes checked."""
    run_mass(shape_full("snapkv_prefill"), SNAP, lanes=[0, 5])


def test_snapkv_prefill_keys_full_128k_sampled_lane():
    """The 128K SnapKV prefill workload at full size (the launch the bench
    times), one lane checked."""
    run_mass(shape_full("snapkv_prefill_128k"), SNAP, lanes=[6])


def shape_full(name):
    from workloads import shape
    return shape(name)

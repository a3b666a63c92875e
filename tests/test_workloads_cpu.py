"""The synthetic generators do what their recipes say (checked by statistics
on small scaled copies; the recipes are readings where the configs are
silent, so this pins the construction, not a page)."""
import math

import numpy as np
import torch

from workloads import Workload, scaled


def test_h2o_70b_logits_follow_zipf_ranks():
    """k_j = (-1.1 ln pi_j) u + (part orthogonal to u) and q_h = sqrt(d) u +
    0.1 noise, so q_h . k_j / sqrt(d) is about -1.1 ln(rank_j): a Zipf
    s = 1.1 weight profile."""
    shp = scaled("h2o_70b", num_layers=1, batch=1, num_kv_heads=2, num_q_heads=16, ctx=2048, steps=2)
    wl = Workload(shp)
    K, _ = wl.context(0)
    q, _, _, _ = wl.step(0, 0)
    d = shp.head_dim
    for kvh in range(2):
        k = K[0, kvh].float()
        s = (q[0, kvh * shp.group].float() @ k.T / math.sqrt(d)).numpy()
        # the ranks from the keys' components along the lane's direction u
        u = wl._direction(0, "cpu")[0][0, kvh].float()
        comp = (k @ u).numpy()
        rank_est = np.exp(-comp / 1.1)
        slope, icpt = np.polyfit(-1.1 * np.log(rank_est), s, 1)
        assert abs(slope - 1.0) < 0.05, slope
        assert np.corrcoef(-1.1 * np.log(rank_est), s)[0, 1] > 0.99
        # the ranks are a permutation of 1..ctx (bf16 storage rounds them)
        r = np.sort(rank_est)
        assert abs(r[0] - 1.0) < 0.05 and abs(r[-1] / shp.ctx - 1.0) < 0.05


def test_snapkv_runs_lift_logits_by_about_three():
    """Planted runs get k += 3u with queries q* + N(0, I): a run token's
    logit exceeds the others' by about 3 on average (|q*| ~ sqrt(d)); 40 runs
    of 8-32 tokens per 4096 positions."""
    shp = scaled("snapkv_decode", batch=1, num_kv_heads=2, num_q_heads=8, ctx=4096, steps=2)
    wl = Workload(shp)
    K, _ = wl.context(0)
    q, _, _, _ = wl.step(0, 0)
    runs = wl._runs(0)
    for kvh in range(2):
        assert len(runs[kvh]) == 40
        assert all(8 <= ln <= 32 for _, ln in runs[kvh])
        mask = np.zeros(shp.ctx, bool)
        for st, ln in runs[kvh]:
            assert not mask[st:st + ln].any()        # non-overlapping
            mask[st:st + ln] = True
        s = (q[0, kvh * shp.group].float() @ K[0, kvh].float().T / math.sqrt(shp.head_dim)).numpy()
        lift = s[mask].mean() - s[~mask].mean()
        assert 2.0 < lift < 4.0, lift


def test_dropkv_heavy_tail_is_one_percent_scaled_by_four():
    """1 % of each lane's key positions are scaled x4: their norms sit near
    4 sqrt(d), the rest near sqrt(d)."""
    shp = scaled("dropkv_prefill", ctx=8192, num_kv_heads=2, num_q_heads=8)
    K, _ = Workload(shp).context(0)
    d = shp.head_dim
    norms = K[0].float().norm(dim=-1).numpy() / math.sqrt(d)
    for kvh in range(2):
        heavy = norms[kvh] > 2.5
        assert heavy.sum() == shp.ctx // 100
        assert abs(np.median(norms[kvh][heavy]) - 4.0) < 0.2
        assert abs(np.median(norms[kvh][~heavy]) - 1.0) < 0.05


def test_inputs_are_seeded_and_stored_in_the_workload_dtype():
    shp = scaled("snapkv_decode", batch=1, num_kv_heads=1, num_q_heads=4, ctx=256, steps=2)
    a, b = Workload(shp).context(0), Workload(shp).context(0)
    assert torch.equal(a[0], b[0]) and a[0].dtype == torch.bfloat16
    toy = Workload(scaled("h2o_toy", ctx=64, steps=2)).context(0)[0]
    assert toy.dtype == torch.float32

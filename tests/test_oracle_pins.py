"""Pins for the oracle: checks against what the pages and mathematics fix,
never against the oracle's own formulas retyped.  CPU only."""
import itertools
import json
import math
import os
import types

import numpy as np
import pytest
import torch

from oracle import attention, dropkv, h2o, paged, select, snapkv
from oracle.engine import DROPKV, Engine, H2O, SNAPKV

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def test_decode_attention_matches_library_sdpa():
    """No eviction: the oracle's attention is textbook softmax attention;
    checked against torch's scaled_dot_product_attention in float64."""
    rng = np.random.default_rng(0)
    for g, n, d in [(1, 7, 64), (4, 33, 128), (8, 129, 16)]:
        q = rng.standard_normal((g, d))
        K = rng.standard_normal((n, d))
        V = rng.standard_normal((n, d))
        out, lse, p = attention.decode_attention(q, K, V)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(q)[None, :, None, :], torch.tensor(K)[None, None].expand(1, g, n, d),
            torch.tensor(V)[None, None].expand(1, g, n, d))[0, :, 0].numpy()
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
        # weights of one query sum to one (DropKV jargon, "Attention weight")
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-13)
        # LSE is the log of the softmax denominator
        s = q @ K.T / math.sqrt(d)
        np.testing.assert_allclose(lse, np.log(np.exp(s).sum(axis=1)), rtol=1e-12)


def test_causal_attention_matches_masked_sdpa():
    rng = np.random.default_rng(1)
    r, n, d = 6, 20, 32
    q = rng.standard_normal((r, d))
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    kpos = np.arange(n)
    qpos = np.arange(n - r, n)
    out, lse, p = attention.causal_attention(q, qpos, K, V, kpos)
    mask = torch.tensor(kpos[None, :] <= qpos[:, None])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q)[None], torch.tensor(K)[None], torch.tensor(V)[None], attn_mask=mask)[0].numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.all(p[~mask.numpy()] == 0.0)


# --------------------------------------------------------------------------
# H2O
# --------------------------------------------------------------------------
def test_h2o_uniform_attention_closed_form():
    """All logits equal: the query at step t spreads 1/(t+1) over tokens
    0..t, so S_j = H * sum_{t=j+1}^{T} 1/(t+1) = H (h_{T+1} - h_{j+1}) with
    h_m the m-th harmonic number.  Built with the oracle's incremental
    accumulate (new token's self weight excluded)."""
    H, T = 3, 12
    S = np.zeros(1)            # token 0 exists before step 1
    for t in range(1, T + 1):
        p = np.full((H, t + 1), 1.0 / (t + 1))   # kept tokens 0..t-1, new token t
        S = h2o.accumulate(S, p)
        S = np.append(S, 0.0)                   # the new token enters with score 0
    harm = lambda m: sum(1.0 / i for i in range(1, m + 1))
    ref = np.array([H * (harm(T + 1) - harm(j + 1)) for j in range(T + 1)])
    np.testing.assert_allclose(S, ref, rtol=1e-13, atol=1e-15)
    # and the literal double sum over a full weight tensor agrees
    A = np.zeros((H, T + 1, T + 1))
    for t in range(T + 1):
        A[:, t, : t + 1] = 1.0 / (t + 1)
    np.testing.assert_allclose(h2o.cumulative_scores_from_rows(A), ref, rtol=1e-13, atol=1e-15)


def test_h2o_group_sum_is_gqa_aggregation():
    """GQA FAQ: the score adds the weights of every query head of the group."""
    p = np.array([[0.5, 0.25, 0.25], [0.1, 0.2, 0.7]])
    np.testing.assert_allclose(h2o.accumulate(np.zeros(2), p), [0.6, 0.45])


def _cfg(**kw):
    base = dict(policy=H2O, num_layers=1, batch=1, num_q_heads=4, num_kv_heads=1, head_dim=16,
                blocks_per_pool=64, budget=8, recent_window=4, obs_window=1, pool_kernel=1,
                theta_f=0.25)
    base.update(kw)
    return types.SimpleNamespace(**base)


def test_h2o_boosted_token_survives():
    """H2O Guide's own check, restated: a token that every query attends
    strongly stays in the cache through 16 steps at budget 8 (4 + 4)."""
    rng = np.random.default_rng(2)
    cfg = _cfg()
    d = cfg.head_dim
    E = Engine(cfg)
    anchor = rng.standard_normal(d)
    anchor /= np.linalg.norm(anchor)
    K0 = rng.standard_normal((1, 1, 1, d))
    K0[0, 0, 0] = 6.0 * anchor
    V0 = rng.standard_normal((1, 1, 1, d))
    E.prefill(0, K0, V0)
    for t in range(1, 17):
        q = rng.standard_normal((1, 4, d)) + 6.0 * anchor
        E.decode_step(0, q, rng.standard_normal((1, 1, d)), rng.standard_normal((1, 1, d)), t)
        assert 0 in E.layers[0].lanes[0].pos.tolist()
        assert E.layers[0].lanes[0].pos.size <= cfg.budget
    E.layers[0].check_invariants()


def _equal_key_prompt(n, g, w, d=8):
    """A prompt whose keys are all equal: every query spreads its weight
    evenly over the keys it sees.  Rows are (head, window position) for the
    last w positions of n, every head's query random (the logits stay equal)."""
    rng = np.random.default_rng(7)
    K = np.tile(rng.standard_normal(d), (n, 1))
    q = rng.standard_normal((g * w, d))
    qpos = np.tile(np.arange(n - w, n), g)
    kpos = np.arange(n)
    _, _, p = attention.causal_attention(q, qpos, K, K, kpos)
    return p, qpos, kpos


def test_h2o_prefill_scores_closed_form():
    """Causal-prefill S_j with equal keys: the row at position t gives
    1/(t+1) to each of tokens 0..t, and S_j counts rows t >= j+1 only, so
    S_j = g (h_n - h_{j+1}) over a whole-prompt window (h: harmonic numbers),
    and every row's weight is counted except its own diagonal entry."""
    n, g = 11, 3
    p, qpos, kpos = _equal_key_prompt(n, g, n)
    S = h2o.prefill_scores(p, qpos, kpos)
    harm = lambda m: sum(1.0 / i for i in range(1, m + 1))
    np.testing.assert_allclose(S, [g * (harm(n) - harm(j + 1)) for j in range(n)], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S.sum(), g * n - g * sum(1.0 / (t + 1) for t in range(n)), rtol=1e-13)
    # the same S_j as the decode-time accumulation over the same queries
    # (the H2O Guide's step-by-step rule run over the prompt)
    A = np.zeros((g, n, n))
    for t in range(n):
        A[:, t, : t + 1] = 1.0 / (t + 1)
    np.testing.assert_allclose(S, h2o.cumulative_scores_from_rows(A), rtol=1e-13, atol=1e-15)


def test_h2o_prefill_scores_random_against_sdpa_weights():
    """Random keys: S_j equals the column sums, over rows strictly after j,
    of torch's causal softmax (its own masked softmax, float64)."""
    rng = np.random.default_rng(8)
    n, d, g = 40, 16, 2
    K = rng.standard_normal((n, d))
    q = rng.standard_normal((g, n, d))
    mask = torch.tril(torch.ones(n, n, dtype=torch.bool))
    logits = torch.tensor(q) @ torch.tensor(K).T / math.sqrt(d)
    P = torch.softmax(logits.masked_fill(~mask, float("-inf")), dim=-1).numpy()
    strict = np.tril(np.ones((n, n)), -1)
    ref = (P * strict).sum(axis=(0, 1))
    qpos = np.tile(np.arange(n), g)
    _, _, p = attention.causal_attention(q.reshape(g * n, d), qpos, K, K, np.arange(n))
    np.testing.assert_allclose(h2o.prefill_scores(p, qpos, np.arange(n)), ref, rtol=1e-12, atol=1e-14)


def test_snapkv_prefill_sums_closed_form_and_mass():
    """SnapKV prefill observation with equal keys: sums_j = g * sum over the
    window positions t >= j of 1/(t+1); every row sums to one, so the sums
    add up to the number of rows; poolKernel 1 leaves them unchanged."""
    n, g, w = 30, 4, 6
    p, qpos, kpos = _equal_key_prompt(n, g, w)
    sums = snapkv.prefill_sums(p, qpos, kpos)
    ref = [g * sum(1.0 / (t + 1) for t in range(max(j, n - w), n)) for j in range(n)]
    np.testing.assert_allclose(sums, ref, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(sums.sum(), g * w, rtol=1e-13)
    np.testing.assert_array_equal(snapkv.prefill_keys(p, qpos, kpos, 1), sums)


def test_snapkv_prefill_one_row_is_last_query_softmax():
    """A window of one query of one head: the keys are that query's softmax
    weights (the SnapKV page's TOVA reduction, at prefill), checked against
    torch.softmax; pooled with r = 1 they match a hand-clamped max."""
    rng = np.random.default_rng(9)
    n, d = 25, 16
    K = rng.standard_normal((n, d))
    q = rng.standard_normal((1, d))
    _, _, p = attention.causal_attention(q, np.array([n - 1]), K, K, np.arange(n))
    ref = torch.softmax(torch.tensor(q @ K.T / math.sqrt(d))[0], dim=0).numpy()
    keys1 = snapkv.prefill_keys(p, np.array([n - 1]), np.arange(n), 1)
    np.testing.assert_allclose(keys1, ref, rtol=1e-12)
    keys3 = snapkv.prefill_keys(p, np.array([n - 1]), np.arange(n), 3)
    hand = [max(ref[max(0, j - 1): j + 2]) for j in range(n)]
    np.testing.assert_allclose(keys3, hand, rtol=1e-12)


def test_engine_score_mass_dispatch():
    """Engine.score_mass: SnapKV keys are the pooled window sums of the kept
    tokens, H2O scores count only rows after the token; a null window is
    inert."""
    rng = np.random.default_rng(10)
    cfg = _cfg(policy=SNAPKV, obs_window=4, pool_kernel=3, num_q_heads=2)
    E = Engine(cfg)
    n, d, w = 20, cfg.head_dim, 5
    K = rng.standard_normal((1, 1, n, d)).astype(np.float32).astype(np.float64)   # the table stores fp32
    E.prefill(0, K, rng.standard_normal((1, 1, n, d)))
    qw = rng.standard_normal((1, 2, w, d))
    qp = np.arange(n - w, n)
    rows = qw[0].reshape(2 * w, d)
    _, _, p = attention.causal_attention(rows, np.tile(qp, 2), K[0, 0], K[0, 0], np.arange(n))
    snap = E.score_mass(0, qw, qp, SNAPKV)["scores"][0]
    h2 = E.score_mass(0, qw, qp, H2O)["scores"][0]
    vis = np.arange(n)[None, :] <= np.tile(qp, 2)[:, None]
    later = np.arange(n)[None, :] < np.tile(qp, 2)[:, None]
    sums = (p * vis).sum(axis=0)
    np.testing.assert_allclose(snap, [sums[max(0, j - 1): j + 2].max() for j in range(n)], rtol=1e-13)
    np.testing.assert_allclose(h2, (p * later).sum(axis=0), rtol=1e-13, atol=1e-16)
    assert E.score_mass(0, None, qp, SNAPKV) is None


# --------------------------------------------------------------------------
# SnapKV
# --------------------------------------------------------------------------
def test_snapkv_hand_example_clamped_pool():
    """Hand-computed: sums (1,5,2,0,3,1) with poolKernel 3 (r = 1), ends
    clamped -> (5,5,5,3,3,3); poolKernel 5 (r = 2) -> (5,5,5,5,3,3)."""
    sums = np.array([1.0, 5.0, 2.0, 0.0, 3.0, 1.0])
    np.testing.assert_array_equal(snapkv.max_pool(sums, 3), [5, 5, 5, 3, 3, 3])
    np.testing.assert_array_equal(snapkv.max_pool(sums, 5), [5, 5, 5, 5, 3, 3])
    np.testing.assert_array_equal(snapkv.max_pool(sums, 1), sums)   # poolKernel 1 disables
    with pytest.raises(ValueError):
        snapkv.max_pool(sums, 4)


def test_snapkv_window_sum_slot_order_and_null_inert():
    hist = np.zeros((3, 4), np.float32)
    slot = 0
    for w in ([1, 2, 3], [4, 5, 6], None, [7, 8, 9]):
        slot = snapkv.ring_write(hist, slot, None if w is None else np.array(w, float))
    assert slot == 3                      # the null step did not advance the ring
    np.testing.assert_array_equal(hist[:, 3], 0.0)
    np.testing.assert_array_equal(snapkv.window_sums(hist), [12.0, 15.0, 18.0])
    # the ring wraps: a fifth and sixth observed step overwrite slots 3 and 0
    for w in ([1, 1, 1], [2, 2, 2]):
        slot = snapkv.ring_write(hist, slot, np.array(w, float))
    assert slot == 1
    np.testing.assert_array_equal(hist[:, 0], 2.0)


def test_snapkv_window_sum_is_float64_in_slot_order():
    """SnapKV, "How it works" (sums recomputed afresh, slot 0 upward) and
    "Complexity" (float32 history, the sums are doubles).  Two float32 rows
    whose float64 sum depends on the order, with the slot-order results
    written out as exact binary values:
    row 0 = (1, 2^-53, 2^-53, 2^-53): slot order rounds 1 + 2^-53 to 1 three
    times (ties to even) -> exactly 1.  Pairwise order gives 1 + 2^-52,
    reverse order 1 + 2^-51, the exact sum rounds to 1 + 2^-51.
    row 1 = (1, 2^-24, 2^-24, 0): float64 holds 1 + 2^-23 exactly, while a
    float32 accumulation rounds 1 + 2^-24 back to 1 twice."""
    t53, t24 = 2.0 ** -53, 2.0 ** -24
    hist = np.array([[1.0, t53, t53, t53], [1.0, t24, t24, 0.0]], dtype=np.float32)
    assert np.all(hist.astype(np.float64) == np.array([[1.0, t53, t53, t53], [1.0, t24, t24, 0.0]]))
    sums = snapkv.window_sums(hist)
    assert sums.dtype == np.float64
    assert sums[0] == 1.0
    assert sums[1] == 1.0 + 2.0 ** -23
    # the orders and precisions a mistake would take give other values
    assert (1.0 + t53) + (t53 + t53) == 1.0 + 2.0 ** -52
    assert ((t53 + t53) + t53) + 1.0 == 1.0 + 2.0 ** -51
    assert math.fsum([1.0, t53, t53, t53]) == 1.0 + 2.0 ** -51
    f32 = np.float32(0.0)
    for x in hist[1]:
        f32 = np.float32(f32 + x)
    assert float(f32) == 1.0
    # the eviction keys with pooling off are these sums
    np.testing.assert_array_equal(snapkv.keys(hist, 1), [1.0, 1.0 + 2.0 ** -23])


def test_snapkv_refusals():
    assert snapkv.validate(1024, 256, 32, 6) == "pool_kernel_even"
    assert snapkv.validate(256, 256, 32, 7) == "recent_ge_budget"
    assert snapkv.validate(1024, 256, 0, 7) == "obs_window_zero"
    assert snapkv.validate(1024, 256, 32, 7) is None


def _run_pair(policy_a, kw_a, policy_b, kw_b, steps=24, seed=3):
    rng = np.random.default_rng(seed)
    d = 16
    Ea = Engine(_cfg(policy=policy_a, budget=10, recent_window=3, **kw_a))
    Eb = Engine(_cfg(policy=policy_b, budget=10, recent_window=3, **kw_b))
    K0 = rng.standard_normal((1, 1, 12, d))
    V0 = rng.standard_normal((1, 1, 12, d))
    Ea.prefill(0, K0, V0)
    Eb.prefill(0, K0, V0)
    for t in range(steps):
        q = 2.0 * rng.standard_normal((1, 4, d))
        k = rng.standard_normal((1, 1, d))
        v = rng.standard_normal((1, 1, d))
        ra = Ea.decode_step(0, q, k, v, 12 + t)
        rb = Eb.decode_step(0, q, k, v, 12 + t)
        yield ra, rb, Ea, Eb


def test_snapkv_window_covering_run_reduces_to_h2o():
    """SnapKV page: with the window longer than the run and pooling off, the
    policy becomes H2O."""
    for ra, rb, _, _ in _run_pair(H2O, {}, SNAPKV, dict(obs_window=64, pool_kernel=1)):
        np.testing.assert_array_equal(ra["victims"][0], rb["victims"][0])


def test_snapkv_window_one_ranks_by_latest_weights():
    """obsWindow 1 with pooling off ranks by the latest step's weights
    (the tova reduction on the SnapKV page); compared with a selection made
    directly from the step's group weights."""
    rng = np.random.default_rng(4)
    d = 16
    E = Engine(_cfg(policy=SNAPKV, budget=10, recent_window=3, obs_window=1, pool_kernel=1))
    K0 = rng.standard_normal((1, 1, 12, d))
    V0 = rng.standard_normal((1, 1, 12, d))
    E.prefill(0, K0, V0)
    for t in range(20):
        L = E.layers[0].lanes[0]
        Kk, Vk = E.layers[0].rows(0)
        q = 2.0 * rng.standard_normal((1, 4, d))
        k = rng.standard_normal((1, 1, d))
        v = rng.standard_normal((1, 1, d))
        _, _, p = attention.decode_attention(q[0], np.vstack([Kk, k[0]]), np.vstack([Vk, v[0]]))
        w = p.sum(axis=0)
        w[-1] = 0.0                      # the new token enters with an empty history
        w = w.astype(np.float32).astype(np.float64)
        pos = np.append(L.pos, 12 + t)
        expect = select.select_lane(w, pos, 10, 3)
        r = E.decode_step(0, q, k, v, 12 + t)
        np.testing.assert_array_equal(r["victims"][0], expect)


# --------------------------------------------------------------------------
# selection
# --------------------------------------------------------------------------
def _brute_victims(keys, pos, k, cand):
    """Independent formulation: a candidate is a victim iff fewer than k
    candidates precede it in (key, position) order."""
    out = []
    idx = [i for i in range(len(keys)) if cand[i]]
    for i in idx:
        before = sum(1 for j in idx if (keys[j], pos[j]) < (keys[i], pos[i]))
        if before < k:
            out.append(pos[i])
    return sorted(out)


def test_select_against_brute_force():
    rng = np.random.default_rng(5)
    for trial in range(300):
        n = int(rng.integers(1, 14))
        keys = rng.integers(0, 4, n).astype(float) * 0.25     # many ties
        pos = np.sort(rng.choice(100, n, replace=False))
        k = int(rng.integers(0, n + 1))
        cand = rng.random(n) < 0.8
        got = select.bottom_k(keys, pos, k, cand)
        assert got.tolist() == _brute_victims(keys.tolist(), pos.tolist(), k, cand.tolist())


def test_select_ties_evict_lower_position_and_ascending():
    keys = np.array([3.0, 1.0, 1.0, 1.0, 2.0, 0.5])
    pos = np.array([10, 11, 12, 13, 14, 15])
    got = select.bottom_k(keys, pos, 3, np.ones(6, bool))
    assert got.tolist() == [11, 12, 15]
    # -0.0 and +0.0 are the same key; the tie goes to the lower position
    got = select.bottom_k(np.array([0.0, -0.0, 1.0]), np.array([5, 6, 7]), 1, np.ones(3, bool))
    assert got.tolist() == [5]
    # NaN keys are evicted last
    got = select.bottom_k(np.array([np.nan, 2.0, np.inf]), np.array([1, 2, 3]), 2, np.ones(3, bool))
    assert got.tolist() == [2, 3]


def test_select_lane_recent_window_and_budget():
    pos = np.arange(20)
    keys = np.zeros(20)            # all tied: the oldest go first
    v = select.select_lane(keys, pos, budget=12, recent_window=5)
    assert v.tolist() == list(range(8))
    v = select.select_lane(np.arange(20.0)[::-1], pos, budget=12, recent_window=5)
    assert v.tolist() == list(range(7, 15))      # lowest keys outside the last 5


# --------------------------------------------------------------------------
# DropKV
# --------------------------------------------------------------------------
def test_lemma1_equals_bruteforce_removal():
    rng = np.random.default_rng(6)
    for trial in range(50):
        n = int(rng.integers(2, 12))
        d = int(rng.integers(1, 9))
        p, _ = attention.softmax_rows(rng.standard_normal((1, n)) * 2)
        p = p[0]
        V = rng.standard_normal((n, d))
        for j in range(n):
            np.testing.assert_allclose(dropkv.lemma1_shift(p, V, j),
                                       dropkv.removal_shift(p, V, [j]), rtol=1e-11, atol=1e-13)


def test_worked_example_golden():
    g = json.load(open(os.path.join(GOLDEN, "dropkv_worked_example.json")))
    pr = g["printed"]
    p = np.array(g["weights"])
    V = np.array(g["values"], float)[:, None]
    a = p @ V
    assert a[0] == pytest.approx(pr["output_a"], abs=1e-12)
    np.testing.assert_allclose(np.abs(a - V)[:, 0], pr["residuals_abs"], atol=1e-12)
    s = dropkv.token_scores(p, V)
    np.testing.assert_allclose(s, pr["scores_2dp"], atol=0.005)
    k = pr["evict_k"]
    greedy = dropkv.greedy_set(s, k)
    assert [i + 1 for i in greedy] == pr["dropkv_removes_1based"]
    by_weight = sorted(np.argsort(p)[:k].tolist())
    assert [i + 1 for i in by_weight] == pr["weight_ranking_removes_1based"]
    sw = dropkv.removal_shift(p, V, by_weight)
    assert (a + sw)[0] == pytest.approx(pr["weight_ranking_new_output"], abs=1e-12)
    assert abs(sw[0]) == pytest.approx(pr["weight_ranking_shift"], abs=1e-12)
    sg = dropkv.removal_shift(p, V, greedy)
    assert (a + sg)[0] == pytest.approx(pr["dropkv_new_output_approx"], abs=0.005)
    assert abs(sg[0]) == pytest.approx(pr["dropkv_shift_approx"], abs=0.005)
    best, best_norm = dropkv.best_set_bruteforce(p, V, k)
    assert len(list(itertools.combinations(range(4), k))) == pr["number_of_pairs"]
    assert best == greedy and pr["dropkv_pair_is_best_of_all_pairs"]


def test_window_scores_against_bruteforce_removal():
    """Prefill-window scores = sum over rows of the brute-force single-token
    removal shift length (rows that cannot see the token contribute 0)."""
    rng = np.random.default_rng(7)
    r, n, d = 5, 11, 8
    q = rng.standard_normal((r, d))
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    kpos = np.arange(n)
    qpos = np.arange(n - r, n)
    got, _, _ = dropkv.window_scores(q, qpos, K, V, kpos)
    ref = np.zeros(n)
    for i in range(r):
        vis = kpos <= qpos[i]
        _, _, p = attention.decode_attention(q[i:i + 1], K[vis], V[vis])
        pv = p[0]
        for jj, j in enumerate(np.nonzero(vis)[0]):
            ref[j] += np.linalg.norm(dropkv.removal_shift(pv, V[vis], [jj]))
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-14)
    sub, _, _ = dropkv.window_scores(q, qpos, K, V, kpos, token_idx=[0, 3, 10])
    np.testing.assert_allclose(sub, ref[[0, 3, 10]], rtol=1e-12)


def test_token_score_p_one_is_never_evicted():
    s = dropkv.token_scores(np.array([1.0, 0.0]), np.array([[1.0], [2.0]]))
    assert s[0] == np.inf and s[1] == 0.0


def test_dropkv_decode_scores_equal_a_one_row_window():
    """A decode step's DropKV scores are the window scores of a window that
    holds just the current query of each head (every key visible), on the
    kept tokens; the window scorer is pinned to brute-force removal above."""
    rng = np.random.default_rng(12)
    for g, n, d in ((4, 13, 8), (1, 5, 3), (8, 30, 16)):
        q = 2.0 * rng.standard_normal((g, d))
        K = rng.standard_normal((n + 1, d))
        V = rng.standard_normal((n + 1, d))
        o, _, p = attention.decode_attention(q, K, V)
        got = dropkv.decode_scores(p, o, V, n)
        ref, _, _ = dropkv.window_scores(q, np.full(g, n), K, V, np.arange(n + 1))
        np.testing.assert_allclose(got, ref[:n], rtol=1e-12)


def test_dropkv_decode_step_evicts_least_output_shift():
    """With a one-step history (obsWindow 1, no pooling) a DropKV decode step
    evicts, among the candidates, the tokens whose single removal (weights
    renormalised, computed by brute force) moves the group's outputs least in
    summed norm; the new token enters with an empty history."""
    rng = np.random.default_rng(13)
    d, g = 16, 4
    E = Engine(_cfg(policy=DROPKV, budget=10, recent_window=3, obs_window=1, pool_kernel=1))
    E.prefill(0, rng.standard_normal((1, 1, 12, d)), rng.standard_normal((1, 1, 12, d)))
    for t in range(15):
        L = E.layers[0].lanes[0]
        Kk, Vk = E.layers[0].rows(0)
        q = 2.0 * rng.standard_normal((1, g, d))
        k = rng.standard_normal((1, 1, d))
        v = rng.standard_normal((1, 1, d))
        Ka, Va = np.vstack([Kk, k[0]]), np.vstack([Vk, v[0]])
        _, _, p = attention.decode_attention(q[0], Ka, Va)
        n = Kk.shape[0]
        shift = [sum(np.linalg.norm(dropkv.removal_shift(p[h], Va, [j])) for h in range(g)) for j in range(n)]
        keys = np.append(np.array(shift, np.float32).astype(np.float64), 0.0)
        pos = np.append(L.pos, 12 + t)
        expect = select.select_lane(keys, pos, 10, 3)
        r = E.decode_step(0, q, k, v, 12 + t)
        np.testing.assert_array_equal(r["victims"][0], expect)
    E.layers[0].check_invariants()


def test_dropkv_decode_null_query_is_inert():
    rng = np.random.default_rng(14)
    d = 16
    E = Engine(_cfg(policy=DROPKV, budget=20, recent_window=3, obs_window=3, pool_kernel=1))
    E.prefill(0, rng.standard_normal((1, 1, 12, d)), rng.standard_normal((1, 1, 12, d)))
    E.decode_step(0, rng.standard_normal((1, 4, d)), rng.standard_normal((1, 1, d)),
                  rng.standard_normal((1, 1, d)), 12)
    L = E.layers[0].lanes[0]
    hist, slot = L.hist.copy(), L.ring_slot
    assert slot == 1 and np.all(hist[:12, 0] > 0)
    E.decode_step(0, None, rng.standard_normal((1, 1, d)), rng.standard_normal((1, 1, d)), 13)
    L = E.layers[0].lanes[0]
    assert L.ring_slot == slot
    np.testing.assert_array_equal(L.hist[:13], hist[:13])


def test_bound_constants_by_hand():
    """The reading of the explainer's undefined c and eps, on a 2-D example
    computed by hand.  Weights p = (.5, .1, .2, .2), values v0 = (.8, 1.6),
    v1 = (-2, 0), v2 = (0, -3), v3 = (-1, -1): the output a = sum p v = 0, so
    the candidates' residuals a - v are (2, 0), (0, 3), (1, 1) (token 0 is
    protected).  Their unit directions (1, 0), (0, 1), (1, 1)/sqrt 2 average
    to the direction (1, 1)/sqrt 2, so u = (1, 1)/sqrt 2 and
    c = min(1/sqrt 2, 1/sqrt 2, 1) = 1/sqrt 2 (the unnormalised residuals
    would give sqrt 2, and their mean direction u = (3, 4)/5 would give .6);
    eps = the largest candidate weight = .2 (not token 0's .5); with k = 2
    the bound is 1/(c (1 - .2)(1 - .4)) = sqrt 2 / .48."""
    p = np.array([0.5, 0.1, 0.2, 0.2])
    V = np.array([[0.8, 1.6], [-2.0, 0.0], [0.0, -3.0], [-1.0, -1.0]])
    c, eps, bound = dropkv.bound_constants(p, V, [1, 2, 3], 2)
    assert c == pytest.approx(1.0 / math.sqrt(2.0), abs=1e-12)
    assert eps == 0.2
    assert bound == pytest.approx(math.sqrt(2.0) / 0.48, rel=1e-12)
    # k eps >= 1: the guarantee does not apply
    assert dropkv.bound_constants(p, V, [1, 2, 3], 5) is None
    # residuals (1, 0) and (-1, 0) lie in no common cone: no c > 0
    p2 = np.array([0.5, 0.25, 0.25])
    V2 = np.array([[0.0, 0.0], [-1.0, 0.0], [1.0, 0.0]])
    assert dropkv.bound_constants(p2, V2, [1, 2], 1) is None


def test_greedy_within_bound_when_cone_holds():
    """Exhaustive best-k on <= 12 tokens; whenever the reading's c > 0 and
    k eps < 1 hold, greedy's shift is within 1/(c(1-eps)(1-k eps)) of the best."""
    rng = np.random.default_rng(8)
    checked = 0
    for trial in range(400):
        n = int(rng.integers(5, 12))
        d = 3
        k = int(rng.integers(1, 4))
        logits = rng.standard_normal(n) * 0.5
        logits[0] += 4.0                            # one dominant token, others small
        p, _ = attention.softmax_rows(logits[None])
        p = p[0]
        base = rng.standard_normal(d)
        V = rng.standard_normal((n, d)) * 0.3 - base   # residuals a - v roughly along +base
        cand = list(range(1, n))                     # the dominant token is protected
        scores = dropkv.token_scores(p, V)
        order = sorted(cand, key=lambda j: (scores[j], j))
        greedy = order[:k]
        best_norm = np.inf
        for S in itertools.combinations(cand, k):
            best_norm = min(best_norm, np.linalg.norm(dropkv.removal_shift(p, V, S)))
        consts = dropkv.bound_constants(p, V, cand, k)
        if consts is None or best_norm == 0:
            continue
        c, eps, bound = consts
        g_norm = np.linalg.norm(dropkv.removal_shift(p, V, greedy))
        assert g_norm <= bound * best_norm * (1 + 1e-12)
        checked += 1
    assert checked > 50


# --------------------------------------------------------------------------
# paged token table
# --------------------------------------------------------------------------
def test_waste_ratio_eq1_and_slot_eq2():
    assert paged.waste_ratio([16, 16]) == 0.0
    assert paged.waste_ratio([1, 1]) == pytest.approx(1 - 2 / 32)
    assert paged.waste_ratio([8, 4, 16, 0]) == pytest.approx(1 - 28 / 64)
    assert paged.waste_ratio([]) == 0.0
    assert paged.slot_of(5, 3) == 83


def _hash_live(PL, lane):
    L = PL.lanes[lane]
    Kk, Vk = PL.rows(lane)
    return hash((tuple(L.pos.tolist()), Kk.tobytes(), Vk.tobytes()))


def test_compaction_invariants_and_packing():
    """I1 (token conservation), I2 (unique mapping), I4 (strict decrease),
    destinations filled completely in ascending position, and after a full
    compaction at most one partial block per lane (F <= 15/(16 N))."""
    rng = np.random.default_rng(9)
    d = 4
    lanes, n = 3, 100
    PL = paged.PagedLayer(lanes, 64, d)
    K = [rng.standard_normal((n, d)).astype(np.float32) for _ in range(lanes)]
    V = [rng.standard_normal((n, d)).astype(np.float32) for _ in range(lanes)]
    PL.prefill(K, V)
    assert [sorted(PL.lanes[l].blocks) for l in range(lanes)] == \
        [list(range(0, 7)), list(range(7, 14)), list(range(14, 21))]
    for lane in range(lanes):
        victims = np.sort(rng.choice(n, 70, replace=False))
        PL.evict(lane, victims)
    before = [_hash_live(PL, l) for l in range(lanes)]
    plans = {l: PL.plan(l, True, 0.25) for l in range(lanes)}
    for l, p in plans.items():
        sources, t_live, n_dst = p
        assert len(sources) > n_dst and n_dst == -(-t_live // 16)
    moves, freed, deferred = PL.reclaim(plans)
    assert not deferred
    after = [_hash_live(PL, l) for l in range(lanes)]
    assert before == after
    PL.check_invariants()
    for l in range(lanes):
        lm = [m for m in moves if m[0] == l]
        assert [m[1] for m in lm] == sorted(m[1] for m in lm)       # ascending position
        dst_seq = [(m[4], m[5]) for m in lm]
        blocks = sorted(set(b for b, _ in dst_seq))
        assert dst_seq == [(blocks[q // 16], q % 16) for q in range(len(dst_seq))]
        counts = PL.live_counts(l)
        N = len(counts)
        assert sum(1 for c in counts.values() if c < 16) <= 1
        assert paged.waste_ratio(counts.values()) <= 15 / (16 * N) + 1e-12
    # destinations came from the lowest free ids, lane 0 first
    freed_before = set(range(21, 64))
    dsts0 = sorted(set(m[4] for m in moves if m[0] == 0))
    assert dsts0 == sorted(freed_before)[: len(dsts0)]


def test_plan_rejected_without_strict_decrease():
    PL = paged.PagedLayer(1, 8, 2)
    K = [np.zeros((32, 2), np.float32)]
    PL.prefill(K, K)
    PL.evict(0, [0])          # blocks: 15 + 16 live -> one source, one destination
    assert PL.plan(0, True, 0.25) is None


def test_admission_reuses_lowest_evicted_slot():
    PL = paged.PagedLayer(1, 8, 2)
    K = [np.zeros((40, 2), np.float32)]
    PL.prefill(K, K)          # blocks 0,1,2 ; block 2 holds 8
    PL.evict(0, [3, 20])
    assert PL.admit(0, 40, np.ones(2), np.ones(2))
    assert PL.lanes[0].slot[-1] == 3
    assert PL.admit(0, 41, np.ones(2), np.ones(2))
    assert PL.lanes[0].slot[-1] == 20
    assert PL.admit(0, 42, np.ones(2), np.ones(2))
    assert PL.lanes[0].slot[-1] == 2 * 16 + 8    # then the tail block
    PL.check_invariants()


def test_new_blocks_go_to_waiting_lanes_lowest_id_first():
    """Reading of the vToken review, Sec. 3.2-3.3 (the pages leave the order
    open): new blocks are the lowest free ids, handed to the lanes whose new
    token found no free slot in ascending lane order, the token at offset 0.
    Hand-built pool of 8 blocks: lane 1 holds block 0, lane 3 holds blocks 2
    and 5, so the free ids are 1, 3, 4, 6, 7; lanes 0, 2 and 3 wait."""
    d = 2
    PL = paged.PagedLayer(4, 8, d)
    for blk, lane in ((0, 1), (2, 3), (5, 3)):
        PL.assign(blk, lane)
        PL.live[blk, :] = True
    np.testing.assert_array_equal(PL.free_blocks(), [1, 3, 4, 6, 7])
    rows = {}
    for lane in (0, 2, 3):
        PL.lanes[lane].append(100 + lane, -1)           # admitted, waiting for a block
        rows[lane] = (np.full(d, 10.0 + lane), np.full(d, 20.0 + lane))
    PL.allocate_admissions([0, 2, 3], rows)
    expect = {0: 1, 2: 3, 3: 4}                         # lane -> block, by hand
    for lane, blk in expect.items():
        assert PL.owner[blk] == lane
        assert blk in PL.lanes[lane].blocks
        assert PL.lanes[lane].slot[-1] == blk * 16      # offset 0 (Eq. (2))
        np.testing.assert_array_equal(PL.live[blk], [True] + [False] * 15)
        np.testing.assert_array_equal(PL.K[blk, 0], rows[lane][0])
        np.testing.assert_array_equal(PL.V[blk, 0], rows[lane][1])
    np.testing.assert_array_equal(PL.free_blocks(), [6, 7])
    # a pool with fewer free blocks than waiting lanes refuses the admission
    for lane in (0, 1):
        PL.lanes[lane].append(200 + lane, -1)
    PL.assign(7, 2)
    with pytest.raises(paged.NoBlocks):
        PL.allocate_admissions([0, 1], {0: rows[0], 1: rows[0]})


def test_stats_counts_half_full_blocks_by_hand():
    """vToken review, Sec. 2 (Fig. 1: blocks at 50% utilisation or less) and
    Eq. (1).  Owned blocks with live counts 8, 9, 16, 1 and one free block:
    N = 4, live = 34, F = 1 - 34/64, and the blocks at <= 50% are the ones
    with 8 and 1 live tokens (8/16 is exactly one half; 9/16 is above)."""
    PL = paged.PagedLayer(2, 5, 2)
    for blk, lane, n_live in ((0, 0, 8), (1, 0, 9), (2, 1, 16), (4, 1, 1)):
        PL.assign(blk, lane)
        PL.live[blk, :n_live] = True
    N, live, F, half = PL.stats()
    assert (N, live, half) == (4, 34, 2)
    assert F == 1.0 - 34.0 / 64.0


def test_kv_bytes_formula():
    """H2O Guide's memory formula 2 x 2 x L x Hkv x d x len x B (bytes)."""
    from workloads.generators import Shape
    s = Shape("x", 0, 80, 16, 64, 8, 128, "bf16", 64000, 0, 1, 0, 1, 1, seed=0)
    assert s.kv_bytes / 1e9 == pytest.approx(335.5, abs=0.05)
    from workloads import shape
    assert shape("h2o_70b").kv_bytes / 1e9 == pytest.approx(85.9, abs=0.05)


def test_per_layer_budget_equals_uniform_engine_per_layer():
    """H2O Guide, "Asymmetric Layer Allocation": a layer given its own budget
    behaves exactly like an engine configured with that budget everywhere;
    the other layers keep the configured one.  Kept counts stop at each
    layer's budget, and the layer's recent window survives every step."""
    rng = np.random.default_rng(12)
    d, n0, steps = 16, 30, 25
    base = _cfg(num_layers=2, num_q_heads=2, budget=20, recent_window=5)
    E = Engine(base)
    E.set_layer_budget(1, 12, 8)
    ref0 = Engine(_cfg(num_layers=1, num_q_heads=2, budget=20, recent_window=5))
    ref1 = Engine(_cfg(num_layers=1, num_q_heads=2, budget=12, recent_window=8))
    with pytest.raises(ValueError):
        E.set_layer_budget(0, 8, 8)
    K = rng.standard_normal((2, 1, 1, n0, d))
    V = rng.standard_normal((2, 1, 1, n0, d))
    for layer in (0, 1):
        E.prefill(layer, K[layer], V[layer])
    ref0.prefill(0, K[0], V[0])
    ref1.prefill(0, K[1], V[1])
    for t in range(steps):
        pos = n0 + t
        for layer, R in ((0, ref0), (1, ref1)):
            q = rng.standard_normal((1, 2, d))
            kn = rng.standard_normal((1, 1, d))
            vn = rng.standard_normal((1, 1, d))
            a = E.decode_step(layer, q, kn, vn, pos)
            b = R.decode_step(0, q, kn, vn, pos)
            np.testing.assert_array_equal(a["victims"][0], b["victims"][0])
            kept = E.layers[layer].lanes[0].pos
            budget, recent = (20, 5) if layer == 0 else (12, 8)
            assert kept.size == min(n0 + t + 1, budget)
            assert set(range(pos - recent + 1, pos + 1)) <= set(kept.tolist())


def test_deferred_relocation_equals_in_step_relocation():
    """vToken review, Sec. 3.3 Stage 4: moving the relocation copy to after
    the step (its own stream) changes no outcome.  A step with relocation
    deferred, then relocate(), leaves the same tables, blocks, K/V rows and
    move list as the step that relocates inline; without relocate() the
    deferred step moves nothing."""
    rng = np.random.default_rng(13)
    d, n0 = 16, 200
    cfg = _cfg(num_q_heads=2, budget=40, recent_window=8, blocks_per_pool=64)
    A, B = Engine(cfg), Engine(cfg)
    B.defer_reloc = True
    K = rng.standard_normal((1, 1, n0, d))
    V = rng.standard_normal((1, 1, n0, d))
    A.prefill(0, K, V)
    B.prefill(0, K, V)
    fired = 0
    for t in range(6):
        q = rng.standard_normal((1, 2, d))
        kn = rng.standard_normal((1, 1, d))
        vn = rng.standard_normal((1, 1, d))
        ra = A.decode_step(0, q, kn, vn, n0 + t)
        rb = B.decode_step(0, q, kn, vn, n0 + t)
        assert rb["moves"] == []
        rr = B.relocate(0)
        assert ra["moves"] == rr["moves"]
        fired += len(ra["moves"]) > 0
        la, lb = A.layers[0], B.layers[0]
        np.testing.assert_array_equal(la.lanes[0].pos, lb.lanes[0].pos)
        np.testing.assert_array_equal(la.lanes[0].slot, lb.lanes[0].slot)
        np.testing.assert_array_equal(la.live, lb.live)
        np.testing.assert_array_equal(la.owner, lb.owner)
        np.testing.assert_array_equal(la.K, lb.K)
        la.check_invariants()
    assert fired >= 1

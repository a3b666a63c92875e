"""Helpers shared by the GPU parity tests: run the CUDA engine (through the
C ABI) and the oracle on the same seeded inputs and compare them."""
import numpy as np
import torch

from kv_cache_token_gb300 import Engine, config_from
from oracle.engine import Engine as Oracle
from workloads import Workload

# Tolerances.  Floating outputs: the task's 2e-3 relative bound, plus an
# absolute floor for entries that cancel towards zero: 1e-4 of the largest
# magnitude in the same row (fp32 accumulation over <= 2^17 terms of bf16
# products leaves ~1e-6 of the row scale; 1e-4 keeps two orders of margin).
RTOL = 2e-3
ROW_FLOOR = 1e-4
# Scores: 2e-3 relative plus 1e-6 of the lane's largest score (expansion
# cancellation and fp32 underflow of tiny weights).
SCORE_FLOOR = 1e-6


def assert_rows_close(got, ref, what, rtol=RTOL, floor=ROW_FLOOR):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.max(np.abs(ref), axis=-1, keepdims=True)
    bad = np.abs(got - ref) > rtol * np.abs(ref) + floor * scale
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d mismatches, first at %s got %r ref %r" %
                             (what, int(bad.sum()), tuple(i), got[tuple(i)], ref[tuple(i)]))


def assert_scores_close(got, ref, what, rtol=RTOL, floor=SCORE_FLOOR):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf = np.isinf(ref)
    assert np.array_equal(inf, np.isinf(got)) or not inf.any(), what + ": inf pattern"
    fin = ~inf
    if not fin.any():
        return
    scale = np.max(np.abs(ref[fin]))
    bad = np.abs(got[fin] - ref[fin]) > rtol * np.abs(ref[fin]) + floor * scale
    if bad.any():
        i = np.nonzero(bad)[0][0]
        raise AssertionError("%s: %d mismatches, first %r vs %r" % (what, int(bad.sum()), got[fin][i], ref[fin][i]))


def make_pair(shp, layers=None):
    eng = Engine(config_from(shp))
    orc = Oracle(shp, layers=layers)
    eng.reset()
    return eng, orc


def prefill_both(eng, orc, wl, layer):
    K, V = wl.context(layer)
    eng.prefill(layer, K.cuda().contiguous(), V.cuda().contiguous())
    orc.prefill(layer, K.double().numpy(), V.double().numpy())


def gpu_state(eng, layer):
    """Token tables, pool metadata and kept K/V rows of one layer (numpy)."""
    torch.cuda.synchronize()
    counts = eng.counts[layer].cpu().numpy()
    pos = eng.positions[layer].cpu().numpy()
    slots = eng.slots[layer].cpu().numpy()
    scores = eng.scores[layer].cpu().numpy()
    ring = eng.ring[layer].cpu().numpy() if eng.ring is not None else None
    nb = eng.lane_nblocks[layer].cpu().numpy()
    lb = eng.lane_blocks[layer].cpu().numpy()
    st = dict(counts=counts, owner=eng.block_owner[layer].cpu().numpy(),
              mask=eng.block_mask[layer].cpu().numpy() & 0xFFFF,
              ring_slot=eng.ring_slot[layer].cpu().numpy(), lanes=[])
    K = eng.k_pool[layer].float().cpu().numpy().reshape(-1, eng.cfg.head_dim)
    V = eng.v_pool[layer].float().cpu().numpy().reshape(-1, eng.cfg.head_dim)
    for l in range(eng.lanes):
        n = int(counts[l])
        s = slots[l, :n]
        st["lanes"].append(dict(pos=pos[l, :n], slot=s, score=scores[l, :n],
                                hist=None if ring is None else ring[s],
                                blocks=set(lb[l, :nb[l]].tolist()), K=K[s], V=V[s]))
    return st


def oracle_state(orc, layer):
    PL = orc.layers[layer]
    bits = (1 << np.arange(16))
    st = dict(counts=np.array([L.pos.size for L in PL.lanes]), owner=PL.owner.copy(),
              mask=(PL.live * bits).sum(axis=1), ring_slot=np.array([L.ring_slot for L in PL.lanes]),
              lanes=[])
    for lane, L in enumerate(PL.lanes):
        s = L.slot
        st["lanes"].append(dict(pos=L.pos, slot=s, score=L.score, hist=L.hist, blocks=set(L.blocks),
                                K=PL.K[s // 16, s % 16], V=PL.V[s // 16, s % 16]))
    return st


def compare_states(g, o, policy, what=""):
    np.testing.assert_array_equal(g["counts"], o["counts"], err_msg=what + " counts")
    np.testing.assert_array_equal(g["owner"], o["owner"], err_msg=what + " owners")
    np.testing.assert_array_equal(g["mask"], o["mask"], err_msg=what + " masks")
    for l, (a, b) in enumerate(zip(g["lanes"], o["lanes"])):
        np.testing.assert_array_equal(a["pos"], b["pos"], err_msg="%s lane %d positions" % (what, l))
        np.testing.assert_array_equal(a["slot"], b["slot"], err_msg="%s lane %d slots" % (what, l))
        assert a["blocks"] == b["blocks"], "%s lane %d block list" % (what, l)
        np.testing.assert_array_equal(a["K"], b["K"], err_msg="%s lane %d K rows" % (what, l))
        np.testing.assert_array_equal(a["V"], b["V"], err_msg="%s lane %d V rows" % (what, l))
        if policy == 0:
            assert_scores_close(a["score"], b["score"], "%s lane %d H2O scores" % (what, l))
        if policy in (1, 2) and a["hist"] is not None:
            np.testing.assert_array_equal(g["ring_slot"], o["ring_slot"], err_msg=what + " ring slot")
            assert_scores_close(a["hist"].ravel(), b["hist"].ravel(), "%s lane %d history" % (what, l))


def victim_lists(n_victims, victims):
    nv = n_victims.cpu().numpy()
    v = victims.cpu().numpy()
    return [v[l, :int(nv[l])] for l in range(len(nv))]


def near_tie(ref_keys, ref_pos, got_v, ref_v, rtol=RTOL):
    """True if two victim sets differ only by swaps between tokens whose
    oracle keys lie within the tolerance of the selection threshold."""
    a, b = set(got_v.tolist()), set(ref_v.tolist())
    if a == b:
        return True
    diff = a ^ b
    key_of = dict(zip(ref_pos.tolist(), ref_keys.tolist()))
    chosen = [key_of[p] for p in b]
    thr = max(chosen) if chosen else 0.0
    return all(abs(key_of[p] - thr) <= rtol * abs(thr) + 1e-12 for p in diff)


def count_tie_swaps(ref_keys, ref_pos, got_v, ref_v, what, rtol=RTOL, floor=SCORE_FLOOR):
    """Number of victims the GPU chose that the oracle did not (as many the
    other way round), after checking that every such token's oracle key lies
    within the score tolerance of the oracle's selection threshold (the
    largest key the oracle evicted): a swap between near-equal keys, which
    fp32 against fp64 scoring may order differently.  Raises otherwise."""
    a, b = set(np.asarray(got_v).tolist()), set(np.asarray(ref_v).tolist())
    assert len(a) == len(b), "%s: %d victims against %d" % (what, len(a), len(b))
    if a == b:
        return 0
    keys = np.asarray(ref_keys, dtype=np.float64)
    key_of = dict(zip(np.asarray(ref_pos).tolist(), keys.tolist()))
    thr = max(key_of[p] for p in b)
    fin = keys[np.isfinite(keys)]
    scale = float(np.max(np.abs(fin))) if fin.size else 0.0
    for p in a ^ b:
        k = key_of[p]
        assert abs(k - thr) <= rtol * abs(thr) + floor * scale, \
            "%s: position %d (oracle key %r) differs from the threshold %r beyond the tolerance" % (what, p, k, thr)
    return len(a - b)

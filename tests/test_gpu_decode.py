"""Decode-step parity: the CUDA engine (attention, scoring, selection,
eviction, admission, relocation) against the oracle, step by step, on the
full H2O toy workload and on scaled copies of the SnapKV and 70B-shaped
workloads (several tiles per lane, ragged tails, mass eviction at step 1)."""
import numpy as np
import pytest
import torch

from tests.gpu_helpers import (assert_rows_close, compare_states, gpu_state, make_pair, near_tie,
                               oracle_state, prefill_both, victim_lists)
from workloads import Workload, scaled, shape

pytestmark = pytest.mark.gpu


def run_decode(shp, steps, layers=(0,), check_state_every=1, null_steps=(), layer_budgets=None):
    wl = Workload(shp)
    eng, orc = make_pair(shp, layers=list(layers))
    for layer, (budget, recent) in (layer_budgets or {}).items():
        eng.set_layer_budget(layer, budget, recent)
        orc.set_layer_budget(layer, budget, recent)
    for layer in layers:
        prefill_both(eng, orc, wl, layer)
        compare_states(gpu_state(eng, layer), oracle_state(orc, layer), shp.policy, "prefill")
    for t in range(steps):
        for layer in layers:
            q, kn, vn, pos = wl.step(layer, t)
            null = t in null_steps
            qg = None if null else q.cuda()
            out, lse, vic, nv = eng.decode_step(layer, qg, kn.cuda(), vn.cuda(), pos)
            ref = orc.decode_step(layer, None if null else q.double().numpy(), kn.double().numpy(),
                                  vn.double().numpy(), pos)
            torch.cuda.synchronize()
            if not null:
                assert_rows_close(out.cpu().numpy(), ref["out"], "step %d out" % t)
                assert_rows_close(lse.cpu().numpy()[..., None], ref["lse"][..., None], "step %d lse" % t)
            got = victim_lists(nv, vic)
            for l in range(eng.lanes):
                if not np.array_equal(got[l], ref["victims"][l]):
                    assert near_tie(ref["keys"][l], ref["pos"][l], got[l], ref["victims"][l]), \
                        "step %d lane %d victims differ beyond a tie" % (t, l)
                    pytest.fail("step %d lane %d: near-tie swap (trajectories would diverge)" % (t, l))
            if t % check_state_every == 0 or t == steps - 1:
                compare_states(gpu_state(eng, layer), oracle_state(orc, layer), shp.policy,
                               "step %d layer %d" % (t, layer))
    code, msg = eng.last_error()
    assert code == 0, msg
    return eng, orc


def test_h2o_toy_full():
    """The H2O toy workload as specified: fp32, d=64, 512 + 32 steps, budget 128."""
    run_decode(shape("h2o_toy"), 32)


def test_snapkv_scaled():
    shp = scaled("snapkv_decode", batch=2, num_kv_heads=4, num_q_heads=16, ctx=700, steps=12,
                 budget=200, recent_window=40, obs_window=8, pool_kernel=5)
    run_decode(shp, 12)


def test_snapkv_window_and_pool_as_specified_short_context():
    """obsWindow 32 and poolKernel 7 as in the SnapKV workload, on a short prompt."""
    shp = scaled("snapkv_decode", batch=1, ctx=1500, steps=40, budget=1024, recent_window=256)
    run_decode(shp, 40, check_state_every=8)


def test_h2o_group8_scaled():
    shp = scaled("h2o_70b", num_layers=2, batch=2, num_kv_heads=2, num_q_heads=16, ctx=1000, steps=6,
                 budget=200, recent_window=100)
    run_decode(shp, 6, layers=(0, 1))


def test_h2o_group8_below_budget_growth():
    """Lanes below the budget grow: admissions append, fill the tail block,
    then take new blocks; no eviction happens until the budget is reached."""
    shp = scaled("h2o_70b", num_layers=1, batch=1, num_kv_heads=3, num_q_heads=24, ctx=100, steps=40,
                 budget=120, recent_window=30)
    run_decode(shp, 40)


def test_dropkv_decode_variant():
    """DropKV decode variant: each step's residual-output scores (sum over the
    group of p / (1 - p) ||a_h - v_j||) go through a history ring of 4 steps;
    keys are the window sums (no pooling); heavy-tailed keys."""
    shp = scaled("dropkv_prefill", ctx=600, num_kv_heads=2, num_q_heads=8, steps=12, budget=200,
                 recent_window=40, obs_window=4, pool_kernel=1, kind="decode")
    run_decode(shp, 12)


def test_dropkv_decode_variant_pooled_with_null_steps_fp32():
    shp = scaled("dropkv_prefill", ctx=400, num_kv_heads=2, num_q_heads=8, steps=10, budget=150,
                 recent_window=20, obs_window=3, pool_kernel=3, kind="decode")
    run_decode(shp, 10, null_steps=(2, 5))
    shp = scaled("h2o_toy", policy=2, ctx=300, steps=12, budget=100, recent_window=20, obs_window=2,
                 pool_kernel=1)
    run_decode(shp, 12)


def test_null_query_is_inert():
    shp = scaled("snapkv_decode", batch=1, num_kv_heads=2, num_q_heads=8, ctx=300, steps=6,
                 budget=200, recent_window=20, obs_window=4, pool_kernel=3)
    run_decode(shp, 6, null_steps=(1, 4))
    shp = scaled("h2o_70b", num_layers=1, batch=1, num_kv_heads=2, num_q_heads=16, ctx=300, steps=4,
                 budget=200, recent_window=20)
    run_decode(shp, 4, null_steps=(0, 2))


@pytest.mark.parametrize("order", [(0, 0, 0, 0, 0, 0), (0, 2, 0, 2, 2, 0, 1, 1, 2), (1, 0, 2, 2, 1, 0, 0)])
def test_steps_enqueued_without_host_sync(order):
    """Decode steps enqueued back to back with no host synchronisation, in
    orders that revisit a layer or its scratch parity immediately (the
    second step's kernels must not start on tables or scratch the first is
    still writing).  Step 1 of every layer is a mass eviction followed by
    relocation, so the apply kernel has work.  Every call's outputs and the
    final tables match the oracle run in the same order."""
    shp = scaled("h2o_70b", num_layers=3, batch=2, num_kv_heads=2, num_q_heads=16, ctx=1000, steps=12,
                 budget=200, recent_window=100)
    wl = Workload(shp)
    layers = sorted(set(order))
    eng, orc = make_pair(shp, layers=layers)
    for layer in layers:
        prefill_both(eng, orc, wl, layer)
    torch.cuda.synchronize()
    t_of = {l: 0 for l in layers}
    calls = []
    for layer in order:
        t = t_of[layer]
        t_of[layer] += 1
        q, kn, vn, pos = wl.step(layer, t)
        vic = torch.zeros((eng.lanes, shp.max_tokens), dtype=torch.int32, device="cuda")
        nv = torch.zeros((eng.lanes,), dtype=torch.int32, device="cuda")
        out, lse, _, _ = eng.decode_step(layer, q.cuda(), kn.cuda(), vn.cuda(), pos, victims=vic, n_victims=nv)
        calls.append((layer, t, q, kn, vn, pos, out, lse, vic, nv))
    torch.cuda.synchronize()
    for layer, t, q, kn, vn, pos, out, lse, vic, nv in calls:
        ref = orc.decode_step(layer, q.double().numpy(), kn.double().numpy(), vn.double().numpy(), pos)
        what = "layer %d step %d" % (layer, t)
        assert_rows_close(out.cpu().numpy(), ref["out"], what + " out")
        assert_rows_close(lse.cpu().numpy()[..., None], ref["lse"][..., None], what + " lse")
        got = victim_lists(nv, vic)
        for l in range(eng.lanes):
            np.testing.assert_array_equal(got[l], ref["victims"][l], err_msg=what + " lane %d victims" % l)
    for layer in layers:
        compare_states(gpu_state(eng, layer), oracle_state(orc, layer), shp.policy, "final layer %d" % layer)
    code, msg = eng.last_error()
    assert code == 0, msg


def test_decode_steps_captured_in_a_cuda_graph():
    """The library never allocates or synchronises inside a step, so decode
    steps can be captured into a CUDA graph (programmatic-dependent launches
    included) and replayed.  Four steps over two layers are captured once and
    replayed once; every captured call's outputs, victims and the final
    tables match the oracle run in the same order."""
    shp = scaled("h2o_70b", num_layers=2, batch=2, num_kv_heads=2, num_q_heads=16, ctx=900, steps=6,
                 budget=200, recent_window=100)
    wl = Workload(shp)
    layers = [0, 1]
    eng, orc = make_pair(shp, layers=layers)
    for layer in layers:
        prefill_both(eng, orc, wl, layer)
    # one eager step per layer first (mass eviction and relocation)
    for layer in layers:
        q, kn, vn, pos = wl.step(layer, 0)
        eng.decode_step(layer, q.cuda(), kn.cuda(), vn.cuda(), pos)
        orc.decode_step(layer, q.double().numpy(), kn.double().numpy(), vn.double().numpy(), pos)
    torch.cuda.synchronize()
    calls = []
    for t in (1, 2):
        for layer in layers:
            q, kn, vn, pos = wl.step(layer, t)
            calls.append(dict(layer=layer, t=t, q=q, kn=kn, vn=vn, pos=pos, qg=q.cuda(), kg=kn.cuda(),
                              vg=vn.cuda(),
                              out=torch.empty((shp.batch, shp.num_q_heads, shp.head_dim), dtype=torch.float32,
                                              device="cuda"),
                              lse=torch.empty((shp.batch, shp.num_q_heads), dtype=torch.float32, device="cuda"),
                              vic=torch.zeros((eng.lanes, shp.max_tokens), dtype=torch.int32, device="cuda"),
                              nv=torch.zeros((eng.lanes,), dtype=torch.int32, device="cuda")))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for c in calls:
            eng.decode_step(c["layer"], c["qg"], c["kg"], c["vg"], c["pos"], c["out"], c["lse"], c["vic"], c["nv"])
    graph.replay()
    torch.cuda.synchronize()
    for c in calls:
        ref = orc.decode_step(c["layer"], c["q"].double().numpy(), c["kn"].double().numpy(),
                              c["vn"].double().numpy(), c["pos"])
        what = "layer %d step %d (graph)" % (c["layer"], c["t"])
        assert_rows_close(c["out"].cpu().numpy(), ref["out"], what + " out")
        assert_rows_close(c["lse"].cpu().numpy()[..., None], ref["lse"][..., None], what + " lse")
        got = victim_lists(c["nv"], c["vic"])
        for l in range(eng.lanes):
            np.testing.assert_array_equal(got[l], ref["victims"][l], err_msg=what + " lane %d victims" % l)
    for layer in layers:
        compare_states(gpu_state(eng, layer), oracle_state(orc, layer), shp.policy, "final layer %d" % layer)
    code, msg = eng.last_error()
    assert code == 0, msg


def test_per_layer_budgets_h2o_and_snapkv():
    """Per-layer budgets (H2O Guide, "Asymmetric Layer Allocation"): three
    H2O layers with their own budgets and recent windows (one of them a
    one-victim steady state, one still mass-evicting, one below its budget
    and growing), then two SnapKV layers; every step against the oracle."""
    shp = scaled("h2o_70b", num_layers=3, batch=2, num_kv_heads=2, num_q_heads=16, ctx=600, steps=8,
                 budget=400, recent_window=100)
    run_decode(shp, 8, layers=(0, 1, 2), layer_budgets={0: (599, 300), 1: (150, 20), 2: (640, 64)})
    shp = scaled("snapkv_decode", num_layers=2, batch=1, num_kv_heads=2, num_q_heads=8, ctx=700, steps=6,
                 budget=200, recent_window=40, obs_window=8, pool_kernel=5)
    run_decode(shp, 6, layers=(0, 1), layer_budgets={1: (300, 100)})
    eng, _ = make_pair(shp)
    from kv_cache_token_gb300.binding import KvevictError
    with pytest.raises(KvevictError):
        eng.set_layer_budget(0, 50, 50)
    with pytest.raises(KvevictError):
        eng.set_layer_budget(2, 100, 10)


def test_deferred_relocation_on_side_stream():
    """vToken review, Sec. 3.3 Stage 4: decode steps with relocation deferred,
    each layer's kvevict_relocate on a second stream after an event on the
    step's stream, and the layer's next step waiting on an event after it;
    the next layer's step runs meanwhile.  Tables, blocks, K/V rows, freed
    blocks and move lists against the oracle doing the same (mass eviction
    at step 1 makes relocation fire)."""
    shp = scaled("h2o_70b", num_layers=2, batch=2, num_kv_heads=2, num_q_heads=16, ctx=900, steps=5,
                 budget=120, recent_window=40)
    wl = Workload(shp)
    layers = (0, 1)
    eng, orc = make_pair(shp, layers=list(layers))
    eng.defer_relocation(True)
    orc.defer_reloc = True
    for layer in layers:
        prefill_both(eng, orc, wl, layer)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    done = {layer: None for layer in layers}
    outs = []
    moved = 0
    for t in range(shp.steps):
        for layer in layers:
            if done[layer] is not None:
                main.wait_event(done[layer])
            q, kn, vn, pos = wl.step(layer, t)
            out, lse, vic, nv = eng.decode_step(layer, q.cuda(), kn.cuda(), vn.cuda(), pos,
                                                victims=torch.empty_like(eng.victims),
                                                n_victims=torch.empty_like(eng.n_victims))
            ref = orc.decode_step(layer, q.double().numpy(), kn.double().numpy(), vn.double().numpy(), pos)
            stepped = torch.cuda.Event()
            stepped.record(main)
            side.wait_event(stepped)
            res = eng.relocate(layer, stream=side)
            done[layer] = torch.cuda.Event()
            done[layer].record(side)
            rref = orc.relocate(layer)
            outs.append((t, layer, out, lse, vic, nv, res, ref, rref))
    torch.cuda.synchronize()
    for t, layer, out, lse, vic, nv, res, ref, rref in outs:
        assert_rows_close(out.cpu().numpy(), ref["out"], "step %d layer %d out" % (t, layer))
        for l, v in enumerate(victim_lists(nv, vic)):
            np.testing.assert_array_equal(v, ref["victims"][l])
        freed, n_freed, moves, n_moves = res
        np.testing.assert_array_equal(freed[:int(n_freed.item())].cpu().numpy(),
                                      np.array(rref["freed"], np.int32))
        m = int(n_moves.item())
        assert m == len(rref["moves"]), (t, layer)
        if m:
            np.testing.assert_array_equal(moves[:m].cpu().numpy(), np.array(rref["moves"], np.int32))
        moved += m
    for layer in layers:
        compare_states(gpu_state(eng, layer), oracle_state(orc, layer), shp.policy, "layer %d" % layer)
    assert moved > 0
    code, msg = eng.last_error()
    assert code == 0, msg


def test_more_lanes_than_resident_epilogue_ctas():
    """160 lanes: more than the epilogue CTAs the device holds at once (one
    per SM), so admissions and relocations go through the separate apply
    kernel instead of the epilogue; every step against the oracle, with
    mass eviction and relocation at step 1."""
    shp = scaled("h2o_70b", num_layers=1, batch=20, num_kv_heads=8, num_q_heads=64, ctx=200, steps=4,
                 budget=64, recent_window=16)
    run_decode(shp, 4)


def test_decode_steps_while_another_stream_holds_the_sms():
    """The epilogue applies admissions into fresh blocks and relocations
    itself, lane by lane, claimed by its CTAs once the layer allocator has
    published its result; a CTA that gave up waiting leaves its lane to the
    others.  Here a second stream keeps every SM busy with long matrix
    products while the decode steps run (the first step is a mass eviction
    with a relocation in every lane, the later ones the steady state): every
    step's outputs, victims and tables still match the oracle."""
    shp = scaled("h2o_70b", num_layers=2, batch=4, num_kv_heads=8, num_q_heads=64, ctx=1200, steps=6,
                 budget=300, recent_window=100)
    wl = Workload(shp)
    eng, orc = make_pair(shp, layers=[0, 1])
    for layer in (0, 1):
        prefill_both(eng, orc, wl, layer)
    side = torch.cuda.Stream()
    a = torch.randn((8192, 8192), dtype=torch.bfloat16, device="cuda")
    bmat = torch.randn((8192, 8192), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    for t in range(shp.steps):
        with torch.cuda.stream(side):
            for _ in range(4):
                torch.matmul(a, bmat)          # ~ms of work on every SM, concurrent with the step
        for layer in (0, 1):
            q, kn, vn, pos = wl.step(layer, t)
            out, lse, vic, nv = eng.decode_step(layer, q.cuda(), kn.cuda(), vn.cuda(), pos)
            ref = orc.decode_step(layer, q.double().numpy(), kn.double().numpy(), vn.double().numpy(), pos)
            torch.cuda.synchronize()
            assert_rows_close(out.cpu().numpy(), ref["out"], "step %d layer %d out" % (t, layer))
            got = victim_lists(nv, vic)
            for l in range(eng.lanes):
                assert np.array_equal(got[l], ref["victims"][l]) or \
                    near_tie(ref["keys"][l], ref["pos"][l], got[l], ref["victims"][l]), \
                    "step %d layer %d lane %d victims" % (t, layer, l)
            compare_states(gpu_state(eng, layer), oracle_state(orc, layer), shp.policy,
                           "step %d layer %d" % (t, layer))
    st = eng.stats(0).cpu().numpy()
    assert st[5] > 0, "the first step relocated tokens"
    code, msg = eng.last_error()
    assert code == 0, msg

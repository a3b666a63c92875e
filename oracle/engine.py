"""Oracle: the eviction engine's calls, step by step (test infrastructure only).

Per decode step of one layer, for every lane (sequence b, KV head h), in
this order (H2O Guide, "Step-by-Step Eviction Lifecycle"; vToken review,
Algorithm 1, whose only policy-specific line is SelectVictims):

1. attend: the g query heads of the group attend the kept tokens and the new
   token (the new token's K/V come with the call);
2. score: H2O adds the group's weights to the kept tokens' cumulative
   scores; SnapKV writes them into the history ring and advances it; DropKV
   (decode variant) writes each kept token's residual-output score of this
   step into the same kind of ring; a null query is inert (SnapKV, "How it
   works");
3. keys: H2O uses the scores, SnapKV and DropKV the pooled window sums, over
   the kept tokens plus the new token (score 0, zero history);
4. select: k = max(0, n + 1 - budget) victims among tokens older than the
   recent window, smallest (key, position) first, ascending output;
5. evict: victims leave the token table, their slots die, empty blocks go
   back to the pool;
6. admit: the new token takes the lowest free slot of its lane's blocks
   (an evicted slot is overwritten in place), else waits for a new block;
then, for the whole layer: new blocks for waiting admissions, then
relocation of lanes whose waste ratio exceeds theta_F.

The window scorer (DropKV prefill), the standalone selection and the forced
compaction are the other calls.
"""
import numpy as np

from . import h2o, snapkv
from .attention import causal_attention, decode_attention
from .dropkv import decode_scores, window_scores
from .paged import PagedLayer
from .select import select_lane

H2O, SNAPKV, DROPKV = 0, 1, 2


class Engine:
    """cfg needs: policy, num_layers, batch, num_q_heads, num_kv_heads,
    head_dim, blocks_per_pool, budget, recent_window, obs_window,
    pool_kernel, theta_f."""

    def __init__(self, cfg, layers=None, store_kv=True):
        self.cfg = cfg
        self.g = cfg.num_q_heads // cfg.num_kv_heads
        self.n_lanes = cfg.batch * cfg.num_kv_heads
        W = cfg.obs_window if cfg.policy in (SNAPKV, DROPKV) and cfg.obs_window >= 1 else 1
        wanted = range(cfg.num_layers) if layers is None else layers
        self.layers = {l: PagedLayer(self.n_lanes, cfg.blocks_per_pool, cfg.head_dim, W, store_kv)
                       for l in wanted}
        self.deferred = 0
        self.layer_budget = {}
        self.defer_reloc = False

    def set_layer_budget(self, layer, budget, recent_window):
        """Per-layer budget (H2O Guide, "Asymmetric Layer Allocation"): later
        steps of ``layer`` keep ``budget`` tokens with a recent window of
        ``recent_window``; the same refusals as the configuration."""
        if recent_window < 1 or recent_window >= budget:
            raise ValueError("recent_window must be in [1, budget)")
        self.layer_budget[layer] = (budget, recent_window)

    def lane_of(self, b, kvh):
        return b * self.cfg.num_kv_heads + kvh

    def prefill(self, layer, K, V):
        """K, V [B, Hkv, n, d]."""
        B, H = self.cfg.batch, self.cfg.num_kv_heads
        Ks = [np.asarray(K[b, h]) for b in range(B) for h in range(H)]
        Vs = [np.asarray(V[b, h]) for b in range(B) for h in range(H)]
        self.layers[layer].prefill(Ks, Vs)

    def lane_keys(self, L, n_new=1):
        """Eviction keys over the kept tokens followed by the new token."""
        c = self.cfg
        if c.policy in (SNAPKV, DROPKV):
            hist = np.vstack([L.hist, np.zeros((n_new, L.hist.shape[1]), np.float32)])
            return snapkv.keys(hist, c.pool_kernel)
        return np.concatenate([L.score, np.zeros(n_new)])

    def decode_step(self, layer, q, k_new, v_new, new_pos):
        """q [B, Hq, d] or None; k_new, v_new [B, Hkv, d].

        Returns dict(out [B, Hq, d], lse [B, Hq], victims: list per lane,
        moves, freed, deferred)."""
        c = self.cfg
        PL = self.layers[layer]
        g = self.g
        budget, recent = self.layer_budget.get(layer, (c.budget, c.recent_window))
        out = np.zeros((c.batch, c.num_q_heads, c.head_dim))
        lse = np.zeros((c.batch, c.num_q_heads))
        victims, freed, pending, new_rows, all_keys, all_pos = [], [], [], {}, [], []
        for lane in range(self.n_lanes):
            b, h = divmod(lane, c.num_kv_heads)
            L = PL.lanes[lane]
            kn = np.asarray(k_new[b, h], dtype=np.float64)
            vn = np.asarray(v_new[b, h], dtype=np.float64)
            n = L.pos.size
            if q is not None:
                Kk, Vk = PL.rows(lane)
                Ka = np.vstack([Kk, kn[None, :]])
                Va = np.vstack([Vk, vn[None, :]])
                o, ls, p = decode_attention(np.asarray(q[b, h * g:(h + 1) * g], np.float64), Ka, Va)
                out[b, h * g:(h + 1) * g] = o
                lse[b, h * g:(h + 1) * g] = ls
                if c.policy == H2O:
                    L.score = h2o.accumulate(L.score, p)
                elif c.policy == SNAPKV:
                    L.ring_slot = snapkv.ring_write(L.hist, L.ring_slot, h2o.group_weights(p)[:n])
                elif c.policy == DROPKV:
                    L.ring_slot = snapkv.ring_write(L.hist, L.ring_slot, decode_scores(p, o, Va, n))
            keys = self.lane_keys(L)
            pos_all = np.append(L.pos, np.int64(new_pos))
            vict = select_lane(keys, pos_all, budget, recent)
            assert new_pos not in vict
            all_keys.append(keys)
            all_pos.append(pos_all)
            freed += PL.evict(lane, vict)
            if not PL.admit(lane, new_pos, kn, vn):
                pending.append(lane)
                new_rows[lane] = (kn, vn)
            victims.append(vict)
        moves, freed2, deferred = self._finish_layer(PL, pending, new_rows, forced=False,
                                                     relocate=not self.defer_reloc)
        return dict(out=out, lse=lse, victims=victims, moves=moves,
                    freed=sorted(freed + freed2), deferred=deferred, keys=all_keys, pos=all_pos)

    def _finish_layer(self, PL, pending, new_rows, forced, relocate=True):
        """Layer-level end of a step: admissions that need a block, then the
        lanes' relocation plans (computed after those admissions)."""
        PL.allocate_admissions(pending, new_rows)
        plans = {}
        for lane in (range(self.n_lanes) if relocate else ()):
            p = PL.plan(lane, forced, self.cfg.theta_f)
            if p is not None:
                plans[lane] = p
        moves, freed, deferred = PL.reclaim(plans)
        self.deferred += int(deferred)
        return moves, freed, deferred

    def score(self, layer, q_win, q_pos, token_idx=None, lanes=None):
        """DropKV prefill-window scoring.

        q_win [B, Hq, w, d]; q_pos [w].  Returns dict(lse [B, Hq, w],
        a [B, Hq, w, d], scores: list per lane of the kept tokens' scores).
        q_win None is inert (scores None)."""
        c = self.cfg
        PL = self.layers[layer]
        g = self.g
        if q_win is None:
            return None
        w = q_win.shape[2]
        lse = np.zeros((c.batch, c.num_q_heads, w))
        a = np.zeros((c.batch, c.num_q_heads, w, c.head_dim))
        scores = {}
        for lane in (range(self.n_lanes) if lanes is None else lanes):
            b, h = divmod(lane, c.num_kv_heads)
            L = PL.lanes[lane]
            K, V = PL.rows(lane)
            rows = np.asarray(q_win[b, h * g:(h + 1) * g], np.float64).reshape(g * w, c.head_dim)
            qp = np.tile(np.asarray(q_pos, np.int64), g)
            sc, ls, aa = window_scores(rows, qp, K, V, L.pos, token_idx)
            lse[b, h * g:(h + 1) * g] = ls.reshape(g, w)
            a[b, h * g:(h + 1) * g] = aa.reshape(g, w, c.head_dim)
            scores[lane] = sc
        return dict(lse=lse, a=a, scores=scores)

    def score_mass(self, layer, q_win, q_pos, kind, lanes=None):
        """Prefill-window attention mass of each kept token (no values).

        kind SNAPKV: the one-shot SnapKV prefill keys (window sums over the
        rows that see the token, pooled with pool_kernel); kind H2O: the
        causal-prefill cumulative scores (rows strictly after the token).
        q_win [B, Hq, w, d]; q_pos [w].  Returns dict(lse [B, Hq, w],
        scores: list per lane); q_win None is inert (returns None)."""
        c = self.cfg
        PL = self.layers[layer]
        g = self.g
        if q_win is None:
            return None
        w = q_win.shape[2]
        lse = np.zeros((c.batch, c.num_q_heads, w))
        scores = {}
        for lane in (range(self.n_lanes) if lanes is None else lanes):
            b, h = divmod(lane, c.num_kv_heads)
            L = PL.lanes[lane]
            K, V = PL.rows(lane)
            rows = np.asarray(q_win[b, h * g:(h + 1) * g], np.float64).reshape(g * w, c.head_dim)
            qp = np.tile(np.asarray(q_pos, np.int64), g)
            _, ls, p = causal_attention(rows, qp, K, V, L.pos)
            lse[b, h * g:(h + 1) * g] = ls.reshape(g, w)
            if kind == SNAPKV:
                scores[lane] = snapkv.prefill_keys(p, qp, L.pos, c.pool_kernel)
            elif kind == H2O:
                scores[lane] = h2o.prefill_scores(p, qp, L.pos)
            else:
                raise ValueError("kind must be SNAPKV or H2O")
        return dict(lse=lse, scores=scores)

    def relocate(self, layer):
        """Deferred relocation (vToken review, Sec. 3.3 Stage 4: the copy
        runs after the step, on its own stream): the theta_F-gated plans a
        decode step of ``layer`` would have run, now.  Returns dict(freed
        ascending, moves, deferred)."""
        moves, freed, deferred = self._finish_layer(self.layers[layer], [], {}, forced=False)
        return dict(freed=sorted(freed), moves=moves, deferred=deferred)

    def compact(self, layer, victims):
        """Forced compaction: evict ``victims`` (list per lane of positions),
        then relocate every lane whose plan frees blocks (no theta_F gate).
        Returns dict(freed ascending, moves, deferred)."""
        PL = self.layers[layer]
        freed = []
        for lane in range(self.n_lanes):
            freed += PL.evict(lane, victims[lane])
        moves, freed2, deferred = self._finish_layer(PL, [], {}, forced=True)
        return dict(freed=sorted(freed + freed2), moves=moves, deferred=deferred)


def select(keys, positions, counts, budget, recent_window):
    """Standalone selection over given keys: per lane, the first counts[l]
    entries of keys[l] / positions[l] (positions ascending)."""
    out = []
    for l in range(len(counts)):
        n = int(counts[l])
        out.append(select_lane(np.asarray(keys[l][:n], np.float64),
                               np.asarray(positions[l][:n], np.int64), budget, recent_window))
    return out

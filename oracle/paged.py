"""Oracle: token table over 16-token paged blocks (test infrastructure only).

vToken review:
* Sec. 2, Eq. (1): intra-block waste F = 1 - sum_i n_i / (N S).
* Sec. 3.2: per logical token a (block_id, offset) location and a liveness
  bit; evicting a token is a metadata write.
* Sec. 3.3 Stage 1: per-block live count n_b; Stage 3: choose low-utilisation
  source blocks, count their live tokens T_live, pack them into
  ceil(T_live / S) destination blocks, proceed only if that frees strictly
  more blocks than it consumes, fill each destination completely before the
  next, keep logical order, record (token, src_block, src_off, dst_block,
  dst_off) moves.
* Sec. 3.4, Eq. (2): slot = block_id * S + offset.
H2O Guide, "PagedAttention Memory Integration": a new token overwrites an
evicted slot in place.

Readings where the pages are silent (also listed in the design notes):
* blocks hold one lane's tokens (a lane is one (sequence, KV head), since
  eviction is decided per KV head) and come from one pool per layer;
* a block left with no live token is returned to the pool at once;
* the new token takes the lowest-numbered free slot among its lane's blocks
  after this step's evictions, else a new block;
* new blocks are the lowest free block ids, handed out in ascending lane
  order, first to admissions, then to reclamation destinations; if the pool
  cannot supply every destination of the layer, all relocation plans of that
  call are deferred;
* sources are the lane's blocks with 0 < n_b < S; a plan runs when the
  lane's F exceeds theta_F (Stage 2's threshold) or when forced.
"""
import math

import numpy as np

BLOCK = 16


class NoBlocks(RuntimeError):
    """The pool has fewer free blocks than a mandatory admission needs."""


def waste_ratio(live_counts, S=BLOCK):
    """Eq. (1): F = 1 - sum(n_b) / (N S); 0 for an empty set of blocks."""
    live_counts = list(live_counts)
    N = len(live_counts)
    if N == 0:
        return 0.0
    return 1.0 - float(sum(live_counts)) / float(N * S)


def slot_of(block, offset, S=BLOCK):
    """Eq. (2): slot = block_id * S + offset."""
    return int(block) * S + int(offset)


class Lane:
    """Token table of one lane, kept tokens in ascending position order."""

    def __init__(self, W):
        self.pos = np.zeros(0, dtype=np.int64)
        self.slot = np.zeros(0, dtype=np.int64)
        self.score = np.zeros(0, dtype=np.float64)
        self.hist = np.zeros((0, max(W, 1)), dtype=np.float32)
        self.ring_slot = 0
        self.blocks = set()

    def append(self, pos, slot):
        self.pos = np.append(self.pos, np.int64(pos))
        self.slot = np.append(self.slot, np.int64(slot))
        self.score = np.append(self.score, 0.0)
        self.hist = np.vstack([self.hist, np.zeros((1, self.hist.shape[1]), np.float32)])

    def keep(self, mask):
        self.pos = self.pos[mask]
        self.slot = self.slot[mask]
        self.score = self.score[mask]
        self.hist = self.hist[mask]


class PagedLayer:
    """One layer's block pool and the token tables of its lanes."""

    def __init__(self, n_lanes, n_blocks, d, W=1, store_kv=True):
        self.n_blocks = int(n_blocks)
        self.owner = np.full(self.n_blocks, -1, dtype=np.int64)
        self.live = np.zeros((self.n_blocks, BLOCK), dtype=bool)
        self.store_kv = store_kv
        if store_kv:
            # bf16 and fp32 values are exactly representable in float32
            self.K = np.zeros((self.n_blocks, BLOCK, d), dtype=np.float32)
            self.V = np.zeros((self.n_blocks, BLOCK, d), dtype=np.float32)
        self.lanes = [Lane(W) for _ in range(n_lanes)]

    # ---- block pool ---------------------------------------------------
    def free_blocks(self):
        return np.nonzero(self.owner < 0)[0]

    def assign(self, block, lane):
        assert self.owner[block] < 0
        self.owner[block] = lane
        self.lanes[lane].blocks.add(int(block))

    def release(self, block):
        lane = int(self.owner[block])
        self.owner[block] = -1
        self.live[block, :] = False
        self.lanes[lane].blocks.discard(int(block))

    def live_counts(self, lane):
        return {b: int(self.live[b].sum()) for b in self.lanes[lane].blocks}

    # ---- rows ---------------------------------------------------------
    def write_row(self, slot, k, v):
        if self.store_kv:
            self.K[slot // BLOCK, slot % BLOCK] = k
            self.V[slot // BLOCK, slot % BLOCK] = v

    def rows(self, lane):
        s = self.lanes[lane].slot
        return (self.K[s // BLOCK, s % BLOCK].astype(np.float64),
                self.V[s // BLOCK, s % BLOCK].astype(np.float64))

    # ---- token table operations ----------------------------------------
    def prefill(self, Kctx, Vctx):
        """Admit every lane's prompt: lane by lane, ceil(n/S) lowest free
        blocks, token i at (block i // S, offset i % S), positions 0..n-1."""
        for lane in range(len(self.lanes)):
            n = Kctx[lane].shape[0]
            nb = -(-n // BLOCK)
            free = self.free_blocks()
            if free.size < nb:
                raise NoBlocks("prefill")
            blocks = free[:nb]
            L = self.lanes[lane]
            for b in blocks:
                self.assign(b, lane)
            i = np.arange(n)
            blk, off = blocks[i // BLOCK], i % BLOCK          # Eq. (2): slot = block * S + offset
            self.live[blk, off] = True
            if self.store_kv:
                self.K[blk, off] = Kctx[lane]
                self.V[blk, off] = Vctx[lane]
            L.pos = i.astype(np.int64)
            L.slot = (blk * BLOCK + off).astype(np.int64)
            L.score = np.zeros(n)
            L.hist = np.zeros((n, L.hist.shape[1]), np.float32)
            L.ring_slot = 0

    def lowest_free_slot(self, lane):
        best = None
        for b in self.lanes[lane].blocks:
            row = self.live[b]
            if not row.all():
                s = slot_of(b, int(np.argmin(row)))
                best = s if best is None else min(best, s)
        return best

    def evict(self, lane, victim_positions):
        """Mark the victims dead (clear their live bits), drop them from the
        table, and release blocks left with no live token.  Returns the
        released block ids, ascending."""
        L = self.lanes[lane]
        vict = np.isin(L.pos, np.asarray(victim_positions, dtype=np.int64))
        slots = L.slot[vict]
        touched = sorted(set((slots // BLOCK).tolist()))
        self.live[slots // BLOCK, slots % BLOCK] = False
        L.keep(~vict)
        freed = [b for b in touched if not self.live[b].any()]
        for b in freed:
            self.release(b)
        return freed

    def admit(self, lane, pos, k, v):
        """Append the new token; returns True if it found a free slot in one
        of the lane's blocks, False if it waits for a new block."""
        slot = self.lowest_free_slot(lane)
        L = self.lanes[lane]
        if slot is None:
            L.append(pos, -1)
            return False
        self.live[slot // BLOCK, slot % BLOCK] = True
        self.write_row(slot, k, v)
        L.append(pos, slot)
        return True

    def plan(self, lane, forced, theta_f):
        """Stage 1 + Stage 3 for one lane: None, or (sources, T_live, n_dst)."""
        counts = self.live_counts(lane)
        F = waste_ratio(counts.values())
        if not forced and not F > theta_f:
            return None
        sources = sorted(b for b, c in counts.items() if 0 < c < BLOCK)
        t_live = sum(counts[b] for b in sources)
        n_dst = -(-t_live // BLOCK)
        if not len(sources) > n_dst:      # I4: the block count must strictly drop
            return None
        return sources, t_live, n_dst

    def relocate(self, lane, sources, dsts):
        """Move every live token of ``sources`` into ``dsts`` in ascending
        position, filling each destination before the next.  Returns the
        move tuples (lane, position, src_block, src_off, dst_block, dst_off)."""
        L = self.lanes[lane]
        src = set(int(b) for b in sources)
        for b in dsts:
            self.assign(b, lane)
        moves = []
        q = 0
        for i in range(L.pos.size):
            s = int(L.slot[i])
            if s // BLOCK in src:
                db, do = int(dsts[q // BLOCK]), q % BLOCK
                q += 1
                ns = slot_of(db, do)
                if self.store_kv:
                    self.K[db, do] = self.K[s // BLOCK, s % BLOCK]
                    self.V[db, do] = self.V[s // BLOCK, s % BLOCK]
                self.live[db, do] = True
                self.live[s // BLOCK, s % BLOCK] = False
                moves.append((lane, int(L.pos[i]), s // BLOCK, s % BLOCK, db, do))
                L.slot[i] = ns
        for b in sorted(src):
            self.release(b)
        return moves

    def allocate_admissions(self, pending, new_rows):
        """New blocks for the lanes whose new token found no free slot:
        ascending lanes take the lowest free block ids; the token goes to
        offset 0.  Raises NoBlocks if the pool is short."""
        free = self.free_blocks()
        if free.size < len(pending):
            raise NoBlocks("admission")
        for i, lane in enumerate(pending):
            b = int(free[i])
            self.assign(b, lane)
            slot = slot_of(b, 0)
            self.live[b, 0] = True
            k, v = new_rows[lane]
            self.write_row(slot, k, v)
            self.lanes[lane].slot[-1] = slot

    def reclaim(self, plans):
        """Run the relocation plans (lane -> (sources, T_live, n_dst)) of one
        call: ascending lanes take the lowest free blocks as destinations.  If
        the pool cannot supply them all, every plan is deferred.
        Returns (moves, freed_sources ascending, deferred)."""
        remaining = self.free_blocks()
        need = sum(p[2] for p in plans.values())
        if need > remaining.size:
            return [], [], True
        moves, freed = [], []
        cur = 0
        for lane in sorted(plans):
            sources, _, n_dst = plans[lane]
            dsts = [int(b) for b in remaining[cur:cur + n_dst]]
            cur += n_dst
            moves += self.relocate(lane, sources, dsts)
            freed += [int(b) for b in sources]
        return moves, sorted(freed), False

    # ---- metrics ----------------------------------------------------------
    def stats(self):
        """(allocated blocks N, live tokens, F, blocks at <= 50% utilisation)."""
        owned = self.owner >= 0
        n_b = self.live[owned].sum(axis=1)
        N = int(owned.sum())
        return N, int(n_b.sum()), waste_ratio(n_b.tolist()), int(np.sum(n_b <= BLOCK // 2))

    def check_invariants(self):
        """I2 (unique mapping): every kept token owns exactly one live slot of
        a block its lane owns, and every live slot is claimed exactly once."""
        claimed = np.zeros((self.n_blocks, BLOCK), dtype=np.int64)
        for lane, L in enumerate(self.lanes):
            assert np.all(np.diff(L.pos) > 0)
            for s in L.slot.tolist():
                if s < 0:
                    continue
                assert self.owner[s // BLOCK] == lane
                claimed[s // BLOCK, s % BLOCK] += 1
        assert np.array_equal(claimed > 0, self.live)
        assert claimed.max(initial=0) <= 1

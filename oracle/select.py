"""Oracle: budgeted bottom-k victim selection (test infrastructure only).

* Keep budget B = k_recent + k_heavy; tokens inside the recent window are
  never evicted; victims are the lowest-score tokens among the candidates
  outside the window -- H2O Guide, "The Dual-Pool Budget Partitioning" and
  "Step-by-Step Eviction Lifecycle" (argmin generalised to k victims, as the
  SnapKV page's evict(budget) and the DropKV page's "k lowest-scoring").
* Equal scores evict the lower position; victims come back in ascending
  position order -- SnapKV, "Tie-breaking".
"""
import numpy as np


def canonical_keys(keys):
    """Keys as compared by the selection.

    -0.0 is the same key as +0.0 (numeric order already says so); NaN sorts
    after +inf, i.e. a NaN-scored token is the last to be evicted.
    """
    k = np.array(keys, dtype=np.float64, copy=True)
    k[k == 0.0] = 0.0
    return k


def recent_cutoff(newest_position, recent_window):
    """Positions >= this value form the protected recent window: the last
    recent_window positions up to and including the newest token."""
    return newest_position - recent_window + 1


def num_victims(n_after_admit, budget):
    """k = max(0, n - budget): evict down to the budget."""
    return max(0, int(n_after_admit) - int(budget))


def bottom_k(keys, positions, k, candidate):
    """Positions of the k candidates with the smallest (key, position).

    keys, positions: arrays over the lane's kept tokens; candidate: bool mask.
    Returns the chosen positions sorted ascending.  If fewer than k tokens are
    candidates, all candidates are chosen.
    """
    keys = canonical_keys(keys)
    positions = np.asarray(positions, dtype=np.int64)
    idx = np.nonzero(np.asarray(candidate, dtype=bool))[0]
    if k <= 0 or idx.size == 0:
        return np.zeros(0, dtype=np.int64)
    # np.lexsort sorts by the LAST key first: primary = key, secondary = position.
    # NaN keys sort after every number.
    order = np.lexsort((positions[idx], keys[idx]))
    chosen = idx[order[: min(k, idx.size)]]
    return np.sort(positions[chosen])


def select_lane(keys, positions, budget, recent_window):
    """Victims of one lane whose kept tokens are ``positions`` (ascending, the
    newest token last) with scores ``keys``."""
    positions = np.asarray(positions, dtype=np.int64)
    n = positions.size
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    cut = recent_cutoff(int(positions[-1]), recent_window)
    k = num_victims(n, budget)
    return bottom_k(keys, positions, k, positions < cut)

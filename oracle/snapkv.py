"""Oracle: decode-time SnapKV (test infrastructure only).

SnapKV page, "How it works":
  on a decode step with weights, history[i][slot] = weight for every kept i,
  then slot = (slot + 1) mod obsWindow, then the new token is admitted with
  an all-zero history row;
  on eviction, sums[i] = sum(history[i]) recomputed afresh in slot order
  0 upward, pooled[i] = max(sums[i-r .. i+r]) with r = (poolKernel-1)/2,
  clamped at the ends, and the lowest pooled scores outside the recent window
  are dropped.
"On the adaptation": neighbours are adjacent KEPT entries, not adjacent
token positions.  A null weight vector is inert: nothing written, the ring
does not advance.  "Complexity": history is float32, the sums are doubles.
"""
import numpy as np


def ring_write(hist, slot, weights):
    """Write this step's weights into column ``slot`` of the float32 history
    [n, W] and return the advanced slot.  weights=None is inert."""
    if weights is None:
        return slot
    W = hist.shape[1]
    hist[:, slot] = np.asarray(weights, dtype=np.float64).astype(np.float32)
    return (slot + 1) % W


def window_sums(hist):
    """sums[i] = hist[i][0] + hist[i][1] + ... + hist[i][W-1], accumulated in
    float64 strictly in slot order 0 upward (no pairwise or running sums)."""
    hist = np.asarray(hist, dtype=np.float32)
    n, W = hist.shape
    s = np.zeros(n, dtype=np.float64)
    for t in range(W):
        s = s + hist[:, t].astype(np.float64)
    return s


def max_pool(sums, pool_kernel):
    """pooled[i] = max(sums[max(0, i-r) .. min(n-1, i+r)]), r = (pk-1)/2.

    The window shrinks at the ends (clamped, not padded).  pool_kernel = 1
    returns the sums unchanged (the page's "disables pooling")."""
    if pool_kernel % 2 == 0:
        raise ValueError("poolKernel must be odd")
    sums = np.asarray(sums, dtype=np.float64)
    n = sums.size
    r = (pool_kernel - 1) // 2
    out = np.empty(n, dtype=np.float64)
    for i in range(n):
        out[i] = np.max(sums[max(0, i - r): min(n, i + r + 1)])
    return out


def keys(hist, pool_kernel):
    """The eviction keys of a lane: max-pooled fresh window sums."""
    return max_pool(window_sums(hist), pool_kernel)


def validate(budget, recent_window, obs_window, pool_kernel):
    """Parameter refusals (SnapKV, "Parameters"): even poolKernel,
    recentWindow >= budget and obsWindow == 0 are refused."""
    if pool_kernel % 2 == 0 or pool_kernel < 1:
        return "pool_kernel_even"
    if recent_window >= budget:
        return "recent_ge_budget"
    if obs_window == 0:
        return "obs_window_zero"
    return None


def prefill_sums(p, q_pos, kpos):
    """SnapKV as the paper runs it ("On the adaptation"): one shot over a
    prompt, the attention the last few prompt queries pay to each key.

    p [r, n] are the causal softmax weights of every (window query, query
    head of the group) row over the kept keys at positions kpos [n], rows at
    positions q_pos [r] (a row gives weight 0 to keys after it).  Returns
    sums[j] = sum over rows of p[row, j], accumulated in float64 row by row
    in row order.  These are the window sums of the prefill observation."""
    p = np.asarray(p, dtype=np.float64)
    vis = np.asarray(kpos)[None, :] <= np.asarray(q_pos)[:, None]
    s = np.zeros(p.shape[1], dtype=np.float64)
    for i in range(p.shape[0]):
        s = s + np.where(vis[i], p[i], 0.0)
    return s


def prefill_keys(p, q_pos, kpos, pool_kernel):
    """Eviction keys of the one-shot prefill selection: the prefill window
    sums, max-pooled over kept neighbours with the same clamped window as the
    decode-time keys ("How it works")."""
    return max_pool(prefill_sums(p, q_pos, kpos), pool_kernel)

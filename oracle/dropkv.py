"""Oracle: DropKV residual-output scores (test infrastructure only).

DropKV explainer:
* Lemma 1 paragraph: removing token j and renormalising the remaining
  weights moves the attention output by p_j / (1 - p_j) * (a - v_j), with a
  the original output; the token's score is the length of that shift.
* "summed over a window of the last w queries, as SnapKV does".
* Greedy: drop the k smallest scores; the shift of the greedy set is at most
  1 / (c (1 - eps)(1 - k eps)) times the best set's when the candidates have
  small weights and their residuals lie in one cone.
* Worked example: weights (.5, .3, .15, .05), values (5, 5, 15, 5).
* Decode variant (a reading: the explainer scores a window of queries; at
  decode time the window is the current query of each head of the group,
  and the per-step scores go through the SnapKV history ring, whose window
  sums are the eviction keys).
"""
import itertools

import numpy as np

from .attention import causal_attention


def lemma1_shift(p, V, j):
    """Closed form of the output shift when token j is removed (Lemma 1)."""
    p = np.asarray(p, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    a = p @ V
    return p[j] / (1.0 - p[j]) * (a - V[j])


def removal_shift(p, V, removed):
    """Brute force: drop the tokens in ``removed``, renormalise the remaining
    weights, recompute the output, and return new output minus old output."""
    p = np.asarray(p, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    a = p @ V
    keep = np.ones(p.size, dtype=bool)
    keep[list(removed)] = False
    a_new = (p[keep] @ V[keep]) / np.sum(p[keep])
    return a_new - a


def token_scores(p, V, a=None):
    """score_j = || p_j / (1 - p_j) * (a - v_j) || for one query.

    Where 1 - p_j is not positive the token's removal is undefined and its
    score is +inf (never evicted).  Entries with p_j = 0 score 0.
    """
    p = np.asarray(p, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if a is None:
        a = p @ V
    r = np.linalg.norm(a[None, :] - V, axis=1)
    one_minus = 1.0 - p
    with np.errstate(divide="ignore", invalid="ignore"):
        s = np.where(one_minus > 0.0, p / one_minus * r, np.inf)
    s = np.where(p == 0.0, 0.0, s)
    return s


def window_scores(q_rows, q_pos, K, V, kpos, token_idx=None):
    """Prefill-window DropKV scores of one KV head.

    q_rows [r, d] are every (window query, query head of the group) row,
    q_pos [r] their positions; the score of token j is the sum over rows of
    the row's Lemma-1 shift length (rows that cannot see j contribute 0).
    token_idx restricts the (costly) residual norms to a subset of tokens;
    the softmax always runs over every key.
    Returns (scores [n] or [len(token_idx)], lse [r], a [r, d]).
    """
    a, lse, p = causal_attention(q_rows, q_pos, K, V, kpos)
    V = np.asarray(V, dtype=np.float64)
    idx = np.arange(V.shape[0]) if token_idx is None else np.asarray(token_idx)
    total = np.zeros(idx.size, dtype=np.float64)
    for i in range(p.shape[0]):
        total += token_scores(p[i, idx], V[idx], a[i])
    return total, lse, a


def decode_scores(p, A, V, n_kept):
    """DropKV decode variant, one step of one KV head: for each kept token j,
    the sum over the group's query heads h of || p_hj / (1 - p_hj) (a_h - v_j) ||.

    p [g, n] are the step's weights over the kept tokens and the new token
    (the new token last), A [g, d] the heads' outputs, V [n, d] the values;
    returns [n_kept] (the new token is not scored).  +inf where 1 - p <= 0.
    """
    p = np.atleast_2d(np.asarray(p, dtype=np.float64))
    A = np.atleast_2d(np.asarray(A, dtype=np.float64))
    V = np.asarray(V, dtype=np.float64)
    total = np.zeros(n_kept, dtype=np.float64)
    for h in range(p.shape[0]):
        total += token_scores(p[h, :n_kept], V[:n_kept], A[h])
    return total


def greedy_set(scores, k):
    """Indices of the k smallest scores (ties: lower index first)."""
    scores = np.asarray(scores, dtype=np.float64)
    order = np.lexsort((np.arange(scores.size), scores))
    return sorted(order[:k].tolist())


def best_set_bruteforce(p, V, k):
    """Exhaustive best k-subset (smallest removal shift); tiny n only --
    choosing the best set is NP-hard (DropKV explainer)."""
    best, best_norm = None, np.inf
    for S in itertools.combinations(range(len(p)), k):
        nrm = np.linalg.norm(np.atleast_1d(removal_shift(p, V, S)))
        if nrm < best_norm - 1e-15:
            best, best_norm = list(S), nrm
    return best, best_norm


def bound_constants(p, V, candidates, k):
    """(c, eps, bound) for the greedy guarantee, under this reading of the
    page's undefined constants: eps = max candidate weight; c = the cone
    constant min_j <r_j, u> / ||r_j|| with u the normalised mean direction of
    the candidates' residuals r_j = a - v_j; bound = 1/(c(1-eps)(1-k eps)).
    Returns None when the preconditions (c > 0, k eps < 1) fail."""
    p = np.asarray(p, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    a = p @ V
    R = a[None, :] - V[candidates]
    norms = np.linalg.norm(R, axis=1)
    if np.any(norms == 0):
        return None
    dirs = R / norms[:, None]
    u = dirs.mean(axis=0)
    if np.linalg.norm(u) == 0:
        return None
    u = u / np.linalg.norm(u)
    c = float(np.min(dirs @ u))
    eps = float(np.max(p[candidates]))
    if c <= 0 or k * eps >= 1:
        return None
    return c, eps, 1.0 / (c * (1 - eps) * (1 - k * eps))

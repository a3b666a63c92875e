"""Oracle: H2O cumulative attention scores (test infrastructure only).

S_j = sum_{t > j} sum_h A_{h,t,j}  -- H2O Guide, "Formulating Cumulative
Attention Scores"; per decode step S_j <- S_j + sum_h A_{h,T,j} for every
token already in the cache -- "Step-by-Step Eviction Lifecycle", score
accumulation.  Under GQA the sum runs over the query heads that share the
KV head -- FAQ "How does H2O handle Grouped-Query Attention (GQA)?".
"""
import numpy as np


def group_weights(p_group):
    """w_j = sum over the group's query heads of p_{h,j}; p_group [g, n]."""
    return np.sum(np.asarray(p_group, dtype=np.float64), axis=0)


def accumulate(S, p_group):
    """S + w for the tokens that were in the cache before this step.

    S [n] holds the kept tokens' scores; p_group [g, n+1] are this step's
    weights over the kept tokens followed by the new token.  The new token's
    weight on itself is not accumulated: Eq. "S_j" sums over t >= j+1 and the
    new token enters with score 0.
    """
    S = np.asarray(S, dtype=np.float64)
    w = group_weights(p_group)[: S.size]
    return S + w


def cumulative_scores_from_rows(A):
    """Literal S_j = sum_{t=j+1}^{T} sum_h A[h, t, j] over a full weight
    tensor A [H, T+1, T+1] (rows t, columns j); used to pin ``accumulate``."""
    A = np.asarray(A, dtype=np.float64)
    H, R, C = A.shape
    S = np.zeros(C)
    for j in range(C):
        for t in range(j + 1, R):
            S[j] += np.sum(A[:, t, j])
    return S


def prefill_scores(p, q_pos, kpos):
    """Causal-prefill initialisation of the cumulative scores: S_j = sum over
    the prompt query rows t at positions after j of A[t, j] (the score
    equation sums t >= j + 1: a token's weight on itself is not counted).

    p [r, n] are the causal softmax weights of the rows (every query of the
    window, for every query head of the group) over the kept keys at
    positions kpos [n]; rows at positions q_pos [r].  With every prompt
    position in the window this is the equation's S_j after the prompt; with
    the last w positions only, it is that sum restricted to those rows."""
    p = np.asarray(p, dtype=np.float64)
    later = np.asarray(kpos)[None, :] < np.asarray(q_pos)[:, None]
    S = np.zeros(p.shape[1], dtype=np.float64)
    for t in range(p.shape[0]):
        S = S + np.where(later[t], p[t], 0.0)
    return S

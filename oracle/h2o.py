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

"""Oracle: softmax attention (test infrastructure only).

A_{h,t,j} = softmax(Q_{h,t} K_j^T / sqrt(d_head)) -- H2O Guide,
"The Existence of Heavy Hitters".  All weights of one query sum to one --
DropKV explainer, jargon entry "Attention weight".
"""
import numpy as np


def softmax_rows(s):
    """Row-wise softmax of logits s [r, n] (float64).

    Returns (p [r, n], lse [r]) with lse the natural log of the softmax
    denominator (DropKV explainer, jargon entry "Log-sum-exp").  Entries equal
    to -inf (masked) get weight exactly 0.  The max subtraction changes nothing
    mathematically; it only keeps exp() finite.
    """
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    l = np.sum(e, axis=1, keepdims=True)
    p = e / l
    lse = (m + np.log(l))[:, 0]
    return p, lse


def logits(q, K):
    """s = q K^T / sqrt(d) for q [r, d], K [n, d] (float64)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    return (q @ K.T) / np.sqrt(q.shape[1])


def decode_attention(q, K, V):
    """One decode step of one KV head.

    q [g, d]: the g query heads that share this KV head (GQA; H2O Guide FAQ
    "How does H2O handle Grouped-Query Attention").  K, V [n, d]: every token
    the new query attends, including the new token itself.

    Returns out [g, d] = p V, lse [g], p [g, n].
    """
    p, lse = softmax_rows(logits(q, K))
    out = p @ np.asarray(V, dtype=np.float64)
    return out, lse, p


def causal_attention(q, qpos, K, V, kpos):
    """Window queries q [r, d] at positions qpos [r] over keys at kpos [n].

    Query i sees key j iff kpos[j] <= qpos[i] (causal prefill; the DropKV
    explainer scores with the last w queries of a prefill).  Returns
    out [r, d], lse [r], p [r, n] with p = 0 on masked entries.
    """
    s = logits(q, K)
    mask = np.asarray(kpos)[None, :] > np.asarray(qpos)[:, None]
    s = np.where(mask, -np.inf, s)
    p, lse = softmax_rows(s)
    out = p @ np.asarray(V, dtype=np.float64)
    return out, lse, p

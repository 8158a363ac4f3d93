"""O(T^2) pairwise-weight form of (causal) linear attention, fp64 numpy.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  This is the second,
independent formulation the recurrence is checked against.  It writes the
output directly from the kernel trick -- the similarity of query i and key j
is phi(q_i).phi(k_j) ("Linear Attention", section "The Kernel-Based
Insight") -- with the causal restriction j <= i including the current token
("[Feature] LinearAttention layer for Keras", Mathematical definition /
Causal), and, for the gated rule, the product of the per-step decays between
j and i (ONNX-light "LinearAttention", update rule "gated").  Meant for small
T only: it builds the (T, T) weight matrix the fast paths never build.
"""
from __future__ import annotations

import numpy as np


def phi(x, feature_map, eps):
    """Feature maps of the Keras request, section "Feature maps"."""
    x = np.asarray(x, dtype=np.float64)
    if feature_map == "elu_plus_one":
        return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    if feature_map == "relu":
        return np.maximum(x, 0.0) + eps
    if feature_map == "none":
        return x
    raise ValueError(feature_map)


def attention(q, k, v, *, causal=True, feature_map="elu_plus_one", use_normalizer=True,
              eps=1e-6, scale=1.0, decay=None, S0=None, Z0=None):
    """Single head.  q (T,Dk), k (T,Dk), v (T,Dv); decay (T,) or (T,Dk) in log space.

    y_i = scale * (sum_{j} w_ij v_j + a_i) / (sum_{j} w_ij + c_i + eps)
    with w_ij = sum_r phi(q_i)_r phi(k_j)_r exp(G_i,r - G_j,r) over j <= i (or
    all j when non-causal), G the inclusive cumulative sum of the decay, and
    a_i = (phi(q_i) * exp(G_i)) @ S0, c_i = phi(q_i) @ Z0 for a carried state.
    """
    fq = phi(q, feature_map, eps)
    fk = phi(k, feature_map, eps)
    v = np.asarray(v, dtype=np.float64)
    T, Dk = fq.shape
    if decay is None:
        W = fq @ fk.T
        qdec = fq
    else:
        g = np.asarray(decay, dtype=np.float64)
        if g.ndim == 1:
            g = np.repeat(g[:, None], Dk, axis=1)
        G = np.cumsum(g, axis=0)  # (T, Dk): log of the decay product up to and incl. t
        # w_ij = sum_r fq[i,r] fk[j,r] exp(G[i,r] - G[j,r])
        W = np.einsum("ir,jr,ijr->ij", fq, fk, np.exp(G[:, None, :] - G[None, :, :]))
        qdec = fq * np.exp(G)
    if causal:
        W = np.tril(W)
    num = W @ v
    den = W.sum(axis=1)
    if S0 is not None:
        num = num + qdec @ np.asarray(S0, dtype=np.float64)
    if Z0 is not None:
        den = den + fq @ np.asarray(Z0, dtype=np.float64)
    if use_normalizer:
        return scale * num / (den + eps)[:, None]
    return scale * num


def attention_bthd(q, k, v, *, q_heads, kv_heads, causal=True, **kw):
    """Multi-head wrapper over packed (B,T,H*D) or (B,T,H,D) arrays with GQA.

    Query head h reads kv head h // (q_heads // kv_heads) (ONNX-light
    "LinearAttention": each KV head is shared by q_num_heads/kv_num_heads
    query heads)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, T = q.shape[:2]
    q = q.reshape(B, T, q_heads, -1)
    k = k.reshape(B, T, kv_heads, -1)
    v = v.reshape(B, T, kv_heads, -1)
    G = q_heads // kv_heads
    decay = kw.pop("decay", None)
    S0 = kw.pop("S0", None)
    Z0 = kw.pop("Z0", None)
    y = np.zeros((B, T, q_heads, v.shape[-1]))
    for b in range(B):
        for h in range(q_heads):
            hk = h // G
            d = None
            if decay is not None:
                dd = np.asarray(decay, dtype=np.float64)
                d = dd[b, :, hk] if dd.ndim == 3 and dd.shape[2] == kv_heads else \
                    dd.reshape(B, T, kv_heads, -1)[b, :, hk, :]
            y[b, :, h] = attention(q[b, :, h], k[b, :, hk], v[b, :, hk], causal=causal,
                                   decay=d,
                                   S0=None if S0 is None else S0[b, hk],
                                   Z0=None if Z0 is None else Z0[b, hk], **kw)
    return y

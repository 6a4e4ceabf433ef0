"""Rounding model of the tensor-core chunked prefill, for deriving tolerances.

Test infrastructure (CPU, numpy).  It restates the chunked form of the gated
delta rule (cortex commit "feat(stage-8c): linear-attention layer", "chunked
algorithm ... chunk_size=64") with the operand precisions the bf16 tensor-core
path uses and nothing else from it: every product's operands are rounded to
bf16 where that path feeds bf16 operands to the tensor cores, accumulation and
the state stay in f64 (the path's f32 accumulation is finer than the bf16
operands), and (I + A)^-1 is exact.  The rel-L2 of this model against the
oracle is the error the operand precisions alone imply; a GPU result within a
small factor of it shows the kernel adds no error of its own.
"""
from __future__ import annotations

import math

import numpy as np

from test_solve_forms import bf16


def chunked_bf16_operands(q, k, v, g, beta, S0, scale, C=64):
    """One head of one sequence.  q, k: raw (not normalised) [L, d] from bf16
    inputs; v [L, d_v]; g, beta [L]; S0 [d, d_v].  Returns (o [L, d_v] rounded
    to bf16, S [d, d_v])."""
    L = len(g)
    rq = scale / np.sqrt((q ** 2).sum(-1) + 1e-6)
    rk = 1.0 / np.sqrt((k ** 2).sum(-1) + 1e-6)
    S = S0.copy()
    O = np.zeros((L, v.shape[1]))
    for c0 in range(0, L, C):
        sl = slice(c0, min(c0 + C, L))
        Q, K, V, gg, bb = q[sl], k[sl], v[sl], g[sl], beta[sl]
        n = len(gg)
        G = np.cumsum(gg)
        low = np.tril(np.ones((n, n), dtype=bool))
        Dm = np.exp(np.where(low, G[:, None] - G[None, :], -np.inf))
        KK = K @ K.T
        A = np.tril(bb[:, None] * rk[sl][:, None] * rk[sl][None, :] * Dm * KK, -1)
        Ti = np.linalg.solve(np.eye(n) + A, np.eye(n))
        W = bf16(bf16(Ti * (bb * np.exp(G) * rk[sl])[None, :]) @ K)
        U = bf16(bf16(Ti * bb[None, :]) @ V)
        P = bf16(rq[sl][:, None] * rk[sl][None, :] * Dm * (Q @ K.T))
        Sb = bf16(S)
        Up = U - W @ Sb
        dec = np.exp(G[-1] - G) * rk[sl]
        O[sl] = bf16((np.exp(G) * rq[sl])[:, None] * (Q @ Sb) + P @ bf16(Up))
        S = math.exp(G[-1]) * S + K.T @ bf16(dec[:, None] * Up)
    return O, S

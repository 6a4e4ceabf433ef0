"""Rounding model of the tensor-core chunked prefill, for reading its error.

Test infrastructure (CPU, numpy).  It restates the chunked form of the gated
delta rule (cortex commit "feat(stage-8c): linear-attention layer", "chunked
algorithm ... chunk_size=64") with the operand precisions the bf16 tensor-core
path uses and nothing else from it: the products with the raw bf16 q, [Q; W] S,
take W and S rounded to bf16; T', the row-scaled diag(beta e^G rk) K and
diag(beta) V, U, P, U' and diag(e^{G_n - G_j} rk) K are rounded to fp16 where
they meet the tensor cores; accumulation and the state stay in f64,
(I + A)^-1 is exact, and o is rounded to bf16.  The rel-L2 of this
model against the oracle is the error the operand precisions alone imply; a
GPU result close to it shows the kernels add little error of their own.  It
sets no tolerance.
"""
from __future__ import annotations

import math

import numpy as np

from test_solve_forms import bf16


def fp16(x):
    """x rounded to the nearest fp16 value."""
    return np.asarray(x, dtype=np.float16).astype(np.float64)


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
        Th = fp16(Ti)
        W = bf16(Th @ fp16((bb * np.exp(G) * rk[sl])[:, None] * K))
        U = fp16(Th @ fp16(bb[:, None] * V))
        P = fp16(rq[sl][:, None] * rk[sl][None, :] * Dm * (Q @ K.T))
        Sb = bf16(S)
        Up = fp16(U - W @ Sb)
        Kd = fp16((np.exp(G[-1] - G) * rk[sl])[:, None] * K)
        O[sl] = bf16((np.exp(G) * rq[sl])[:, None] * (Q @ Sb) + P @ Up)
        S = math.exp(G[-1]) * S + Kd.T @ Up
    return O, S

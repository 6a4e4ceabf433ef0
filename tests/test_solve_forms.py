"""Direct solve vs Neumann-style product for the chunk's triangular system.

NxD-Inference PR "Add Qwen3.6-27B hybrid DeltaNet/GQA contrib model and vLLM
serving path", "Known limitations": the stable direct-solve DeltaNet path
trades some speed for numerical stability against a faster Neumann-style path.
The chunked form needs T' = (I + A)^-1 for a strictly lower-triangular A (64 x
64 per chunk).  Since A is nilpotent (A^n = 0 for n rows), the Neumann series
sum_k (-A)^k ends after n terms and equals the product
    (I + N)(I + N^2)(I + N^4) ... (I + N^(2^(m-1))),   N = -A,  2^m >= n,
six factors for n = 64: five squarings and five products, all dense matrix
products -- the form that suits a matrix engine.  The direct solve is forward
substitution (here as the kernel does it: 16 x 16 diagonal blocks by forward
substitution in f32, the off-diagonal blocks by doubling).

The f64 forms are pinned to each other and to the recurrence; the error study
runs each form in the precision a GPU would use, on the chunks of the
Qwen3.6-27B prefill workload and on a slow-decay, correlated-key stress case.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from test_oracle_pins import _dr_case, chunked_dense, rel_l2


# ------------------------------------------------------------ the two forms
def neumann_inverse(A, rnd=None):
    """(I + A)^-1 for strictly lower-triangular A as the product of
    (I + N^(2^i)), N = -A.  `rnd` rounds each matrix product's operands and
    result (None: exact f64)."""
    r = (lambda x: x) if rnd is None else rnd
    n = A.shape[0]
    eye = np.eye(n)
    P = r(-A)          # N^(2^i)
    T = r(eye + P)     # running product
    span = 2
    while span < n:
        P = r(r(P) @ r(P))
        T = r(r(T) @ r(eye + P))
        span *= 2
    return T


def forward_inverse(A, dtype=np.float32):
    """(I + A)^-1 by forward substitution, row by row, in `dtype`."""
    n = A.shape[0]
    A = A.astype(dtype)
    T = np.zeros((n, n), dtype=dtype)
    for i in range(n):
        row = np.zeros(n, dtype=dtype)
        row[i] = 1
        for j in range(i):
            row -= A[i, j] * T[j]
        T[i] = row
    return T.astype(np.float64)


def blocked_inverse(A, rnd_mm, B=16):
    """The kernel's scheme: diagonal B x B blocks by forward substitution in
    f32, then the off-diagonal blocks by doubling, T'_ij = -T'_ii A_ij T'_jj
    over blocks of 16 and then of 32 rows, with rnd_mm rounding the operands
    of each block product (tf32 on the GPU)."""
    n = A.shape[0]
    T = np.zeros((n, n))
    for b0 in range(0, n, B):
        sl = slice(b0, min(b0 + B, n))
        T[sl, sl] = forward_inverse(A[sl, sl])
    size = B
    while size < n:
        for b0 in range(0, n, 2 * size):
            lo = slice(b0, min(b0 + size, n))
            hi = slice(b0 + size, min(b0 + 2 * size, n))
            if hi.start >= n:
                continue
            f32 = lambda x: rnd_mm(x).astype(np.float32).astype(np.float64)
            T[hi, lo] = -f32(f32(T[hi, hi]) @ f32(A[hi, lo])) @ f32(T[lo, lo])
            T[hi, lo] = T[hi, lo].astype(np.float32).astype(np.float64)
        size *= 2
    return T


# ------------------------------------------------------------ rounding
def _round_mantissa(x, drop):
    """Round an array to f32 with its low `drop` mantissa bits cleared, to
    nearest-even (bf16: drop 16, tf32: drop 13)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    half = np.uint64((1 << (drop - 1)) - 1)
    lsb = (u >> np.uint64(drop)) & np.uint64(1)
    u = (u + half + lsb) & np.uint64(~((1 << drop) - 1) & 0xFFFFFFFF)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16(x):
    return _round_mantissa(x, 16)


def tf32(x):
    return _round_mantissa(x, 13)


def f32(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64)


# ------------------------------------------------------------ pins (f64)
@pytest.mark.parametrize("n", [1, 2, 3, 16, 37, 64])
def test_neumann_product_equals_solve_in_f64(n):
    rng = np.random.default_rng(n)
    A = np.tril(rng.normal(scale=0.4, size=(n, n)), -1)
    ref = np.linalg.solve(np.eye(n) + A, np.eye(n))
    assert rel_l2(neumann_inverse(A), ref) < 1e-13
    assert rel_l2(forward_inverse(A, np.float64), ref) < 1e-13
    assert rel_l2(blocked_inverse(A, lambda x: x), ref) < 1e-6  # f32 diagonal blocks


def test_neumann_needs_every_factor():
    # closed form: with A = -S (S the sub-diagonal shift), (I + A)^-1 =
    # sum_k S^k is the lower triangle of ones; five factors instead of six
    # stop at S^31 and miss the 528 entries 32 or more rows below the diagonal
    n = 64
    A = -np.eye(n, k=-1)
    ref = np.tril(np.ones((n, n)))
    assert np.array_equal(neumann_inverse(A), ref)
    eye, P, T = np.eye(n), -A, np.eye(n) - A
    for _ in range(4):
        P = P @ P
        T = T @ (eye + P)
    assert np.array_equal(T, np.tril(ref, 0) - np.tril(ref, -32))
    assert abs(rel_l2(T, ref) - np.sqrt(528 / 2080)) < 1e-12


@pytest.mark.parametrize("C", [16, 64])
def test_chunked_form_with_neumann_inverse_equals_recurrence(oracle_mod, C):
    lengths = [100, 64]
    T = sum(lengths)
    q, k, v, g, beta, S0 = _dr_case(22, T=T, H_k=1, H_v=1, d_k=16, d_v=8, N=2, g_scale=0.5)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o, S, _ = oracle_mod.delta_rule(q, k, v, g, beta, cu, S0=S0, scale=0.25)
    qn = q / np.sqrt((q ** 2).sum(-1, keepdims=True) + 1e-6) * 0.25
    kn = k / np.sqrt((k ** 2).sum(-1, keepdims=True) + 1e-6)
    for i in range(2):
        sl = slice(cu[i], cu[i + 1])
        O2, S2 = chunked_dense(qn[sl, 0], kn[sl, 0], v[sl, 0], g[sl, 0], beta[sl, 0], S0[i, 0],
                               C, inverse=neumann_inverse)
        assert rel_l2(o[sl, 0], O2) < 1e-12
        assert rel_l2(S[i, 0], S2) < 1e-12


# ------------------------------------------------------------ error study
def _chunk_matrices(oracle_mod, kind, n_chunks=8, heads=(0, 17, 47), seed=3):
    """A (f64, from the bf16 inputs a GPU sees) of the first chunks of some
    value heads.  kind 'workload': the Qwen3.6-27B prefill inputs through the
    oracle's conv1d + SiLU, l2norm and gates.  kind 'stress': slow decay
    (A_log = ln U(1e-3, 1e-2)), keys sharing one direction (cosine ~0.8) and
    beta ~ 0.9, where (I + A)^-1 is far from the identity."""
    s = W.QWEN36_27B
    Tn = 64 * n_chunks
    rng = np.random.default_rng(seed)
    if kind == "workload":
        inp = W.workload_inputs("qwen36_27b_prefill")
        x = inp["mixed_qkv"][:Tn]
        y = bf16(oracle_mod.conv1d(W.to_f64(x), W.to_f64(inp["conv_w"]))[0])  # as a GPU stores it
        g, beta = oracle_mod.gates(W.to_f64(inp["a"][:Tn]), W.to_f64(inp["b"][:Tn]),
                                   W.to_f64(inp["A_log"]), W.to_f64(inp["dt_bias"]))
        kcols = lambda kh: y[:, s.H_k * s.d_k + kh * s.d_k: s.H_k * s.d_k + (kh + 1) * s.d_k]
    else:
        u = rng.normal(size=s.d_k)
        keys = bf16(u[None, :] + 0.5 * rng.normal(size=(Tn, s.d_k)))
        kcols = lambda kh: keys
        A_log = np.log(rng.uniform(1e-3, 1e-2, size=s.H_v))
        a = rng.normal(size=(Tn, s.H_v))
        b = rng.normal(2.2, 0.5, size=(Tn, s.H_v))
        g, beta = oracle_mod.gates(a, b, A_log, np.zeros(s.H_v))
    r = s.H_v // s.H_k
    out = []
    for h in heads:
        kn = oracle_mod.l2norm(kcols(h // r))
        for c in range(n_chunks):
            sl = slice(64 * c, 64 * (c + 1))
            G = np.cumsum(g[sl, h])
            K = kn[sl]
            A = np.tril(beta[sl, h][:, None] * np.exp(np.tril(G[:, None] - G[None, :])) * (K @ K.T), -1)
            out.append(A)
    return out


FORMS = {
    # name: (T' from f32 A, in the precision of the form); T' is rounded to bf16
    # after, as the W and U products take bf16 operands
    "direct, kernel scheme (f32 blocks + tf32 doubling)": lambda A: blocked_inverse(f32(A), tf32),
    "direct, f32 forward substitution": lambda A: forward_inverse(f32(A)),
    "Neumann product, f32": lambda A: neumann_inverse(f32(A), f32),
    "Neumann product, tf32 operands": lambda A: neumann_inverse(f32(A), tf32),
    "Neumann product, bf16 operands": lambda A: neumann_inverse(f32(A), bf16),
}


def solve_error_study(oracle_mod, kind):
    """Per form: median and max over chunks of rel-L2(bf16(T'), (I + A)^-1),
    and the largest |entry| of the exact inverse."""
    mats = _chunk_matrices(oracle_mod, kind)
    rows = {}
    growth = 0.0
    for A in mats:
        ref = np.linalg.solve(np.eye(64) + A, np.eye(64))
        growth = max(growth, float(np.abs(ref).max()))
        for name, fn in FORMS.items():
            rows.setdefault(name, []).append(rel_l2(bf16(fn(A)), ref))
    return {k: (float(np.median(v)), float(np.max(v))) for k, v in rows.items()}, growth, len(mats)


@pytest.mark.parametrize("kind", ["workload", "stress"])
def test_solve_error_study(oracle_mod, kind):
    """Prints the table (pytest -s) and checks what the kernel relies on: its
    scheme stays at the bf16 rounding of T' (2^-9 relative per entry), and the
    Neumann product is no better than it in any precision."""
    res, growth, n = solve_error_study(oracle_mod, kind)
    print(f"\n{kind}: {n} chunks of 64, max |(I + A)^-1| = {growth:.3g}")
    for name, (med, mx) in res.items():
        print(f"  {name:52s} median {med:.2e}  max {mx:.2e}")
    kern = res["direct, kernel scheme (f32 blocks + tf32 doubling)"]
    assert kern[1] < 4e-3
    for name in ("Neumann product, tf32 operands", "Neumann product, bf16 operands"):
        assert res[name][1] >= 0.9 * kern[1]

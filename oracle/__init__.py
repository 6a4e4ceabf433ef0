"""CPU float64 oracle of the Gated DeltaNet layer core.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The library's
compute path never calls it, and it shares no code with the CUDA kernels.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision, tokens in
order); this module compiles it with gcc on first use and exposes each step
with numpy float64 arrays.  The composite helpers below only slice channels
(the [q | k | v] split) and call the C steps in the order the cortex commit
"feat(stage-8c): linear-attention layer (Qwen3-Next GatedDeltaNet)" lists them
in its "Block" section.

Parity unpinned: none -- every step here is pinned by ``tests/test_oracle_*.py``
(closed forms, brute force, an independent dense chunked restatement and
hand-derived fixtures under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_gdn.so")
_lock = threading.Lock()
_lib = None

L2NORM_EPS = 1e-6
RMSNORM_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build (gcc, OpenMP, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_conv1d.argtypes = [P, P, P, I64, I64, I64, P, ctypes.c_int, P, P, I64, P,
                                          ctypes.c_int]
            lib.oracle_gates.argtypes = [P, P, P, P, I64, I64, P, P]
            lib.oracle_l2norm.argtypes = [P, I64, I64, ctypes.c_double]
            lib.oracle_delta_rule.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I64, P,
                                              ctypes.c_double, ctypes.c_int, ctypes.c_double,
                                              P, P, I64, P, ctypes.c_int]
            lib.oracle_rmsnorm_gated.argtypes = [P, P, P, ctypes.c_double, I64, I64, I64, P]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _cu(cu_seqlens, T):
    if cu_seqlens is None:
        return np.array([0, T], dtype=np.int64)
    return np.ascontiguousarray(np.asarray(cu_seqlens), dtype=np.int64)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def n_ckpt(cu_seqlens, every: int) -> int:
    if every <= 0:
        return 0
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return int(sum((cu[i + 1] - cu[i]) // every for i in range(len(cu) - 1)))


def conv1d(x, w, cu_seqlens=None, state_in=None, apply_silu=True, ckpt_every=0, nthreads=0):
    """Depthwise causal conv with state prepend (+SiLU).
    Returns (y [T, C], state_out [N, C, K-1], ckpt [n_ckpt, C, K-1] or None)."""
    x, w, st = _f64(x), _f64(w), _f64(state_in)
    T, C = x.shape
    K = w.shape[1]
    cu = _cu(cu_seqlens, T)
    N = len(cu) - 1
    y = np.empty_like(x)
    so = np.empty((N, C, K - 1))
    nck = n_ckpt(cu, ckpt_every)
    ck = np.empty((nck, C, K - 1)) if nck else None
    _load().oracle_conv1d(_p(x), _p(w), _p(cu), N, C, K, _p(st), int(bool(apply_silu)), _p(y),
                          _p(so), int(ckpt_every), _p(ck), int(nthreads))
    return y, so, ck


def gates(a, b, A_log, dt_bias):
    """Returns (g, beta), both [T, H] float64."""
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    T, H = a.shape
    g = np.empty_like(a)
    beta = np.empty_like(a)
    _load().oracle_gates(_p(a), _p(b), _p(A_log), _p(dt_bias), T, H, _p(g), _p(beta))
    return g, beta


def l2norm(x, eps=L2NORM_EPS):
    x = np.array(x, dtype=np.float64, copy=True)
    d = x.shape[-1]
    _load().oracle_l2norm(_p(x), x.size // d if d else 0, d, eps)
    return x


def delta_rule(q, k, v, g, beta, cu_seqlens=None, S0=None, scale=None, l2norm_qk=True,
               ckpt_every=0, eps=L2NORM_EPS, nthreads=0):
    """Per-token gated delta rule.  q, k [T, H_k, d_k]; v [T, H_v, d_v];
    g, beta [T, H_v].  Returns (o [T, H_v, d_v], S_final [N, H_v, d_k, d_v],
    ckpt [n_ckpt, H_v, d_k, d_v] or None)."""
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    T, H_k, d_k = q.shape
    H_v, d_v = v.shape[1], v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = len(cu) - 1
    if scale is None:
        scale = d_k ** -0.5
    o = np.empty((T, H_v, d_v))
    Sf = np.empty((N, H_v, d_k, d_v))
    nck = n_ckpt(cu, ckpt_every)
    ck = np.empty((nck, H_v, d_k, d_v)) if nck else None
    _load().oracle_delta_rule(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu), N, H_k, H_v, d_k,
                              d_v, _p(S0), float(scale), int(bool(l2norm_qk)), float(eps), _p(o),
                              _p(Sf), int(ckpt_every), _p(ck), int(nthreads))
    return o, Sf, ck


def rmsnorm_gated(o, z, w, eps=RMSNORM_EPS):
    """o [T, H, d]; z [T, H*d]; w [d].  Returns out [T, H*d]."""
    o, z, w = _f64(o), _f64(z), _f64(w)
    T, H, d = o.shape
    out = np.empty((T, H * d))
    _load().oracle_rmsnorm_gated(_p(o), _p(z), _p(w), float(eps), T, H, d, _p(out))
    return out


def split_qkv(y, H_k, H_v, d_k, d_v):
    """[q | k | v] channel split of the conv output, heads contiguous."""
    T = y.shape[0]
    q = y[:, :H_k * d_k].reshape(T, H_k, d_k)
    k = y[:, H_k * d_k:2 * H_k * d_k].reshape(T, H_k, d_k)
    v = y[:, 2 * H_k * d_k:2 * H_k * d_k + H_v * d_v].reshape(T, H_v, d_v)
    return q, k, v


def layer_prefill(x, z, a, b, conv_w, A_log, dt_bias, norm_w, H_k, H_v, d_k, d_v,
                  cu_seqlens=None, S0=None, conv_state0=None, scale=None, ckpt_every=0,
                  nthreads=0):
    """Whole layer core over packed sequences: conv1d+SiLU -> split -> l2norm,
    gates -> delta rule -> RMSNormGated.  Returns a dict of float64 arrays."""
    y, conv_state, conv_ck = conv1d(x, conv_w, cu_seqlens, conv_state0, True, ckpt_every,
                                    nthreads)
    q, k, v = split_qkv(y, H_k, H_v, d_k, d_v)
    g, beta = gates(a, b, A_log, dt_bias)
    o, S, ck = delta_rule(q, k, v, g, beta, cu_seqlens, S0, scale, True, ckpt_every,
                          nthreads=nthreads)
    out = rmsnorm_gated(o, z, norm_w)
    return {"y": y, "conv_state": conv_state, "conv_ckpt": conv_ck, "g": g, "beta": beta,
            "o": o, "S": S, "S_ckpt": ck, "out": out}


def layer_decode_step(x, z, a, b, conv_w, A_log, dt_bias, norm_w, H_k, H_v, d_k, d_v, S,
                      conv_state, scale=None, nthreads=0):
    """One single-token step for B sequences (x [B, conv_dim]): the same
    definitions with one token per sequence.  Returns (out, S_new,
    conv_state_new, o)."""
    B = x.shape[0]
    cu = np.arange(B + 1, dtype=np.int64)
    r = layer_prefill(x, z, a, b, conv_w, A_log, dt_bias, norm_w, H_k, H_v, d_k, d_v, cu, S,
                      conv_state, scale, 0, nthreads)
    return r["out"], r["S"], r["conv_state"], r["o"]

"""Helpers of the GPU parity tests: moving seeded inputs to the device, slicing
one value head out of a layer's inputs for the oracle, the oracle's decode step
with the activations rounded where the layer's calls hand them on, and
tolerance checks."""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
import workloads as W

TOL = {torch.float32: 1e-4, torch.bfloat16: 5e-3}


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((x - ref).ravel())
    return float(num / den) if den > 0 else float(num)


def host(t) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def to_dev(d: dict, dev="cuda") -> dict:
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def assert_close(name, got, ref, tol, per_head_axis=None):
    e = rel_l2(got, ref)
    msg = f"{name}: rel-L2 {e:.3e} > {tol:.1e}"
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{name}: non-finite output"
    assert e <= tol, msg
    if per_head_axis is not None:
        g = np.moveaxis(np.asarray(got, dtype=np.float64), per_head_axis, 0)
        r = np.moveaxis(np.asarray(ref, dtype=np.float64), per_head_axis, 0)
        worst = max(rel_l2(g[i], r[i]) for i in range(g.shape[0]))
        assert worst <= 2 * tol, f"{name}: worst head rel-L2 {worst:.3e} > {2 * tol:.1e}"
    return e


def head_channels(shape: W.GDNShape, h: int):
    """Channel indices of v-head h's q, k (its key head) and v in mixed_qkv."""
    kh = h // (shape.H_v // shape.H_k)
    D = shape.d_k
    q = np.arange(kh * D, (kh + 1) * D)
    k = shape.H_k * D + q
    v = 2 * shape.H_k * D + np.arange(h * shape.d_v, (h + 1) * shape.d_v)
    return np.concatenate([q, k, v])


def oracle_head_prefill(inp: dict, shape: W.GDNShape, h: int, ckpt_every=0):
    """Oracle of the whole layer core restricted to value head h: every
    channel, head and state involved in head h is sliced out (heads and conv
    channels are independent), and the oracle runs with H_k = H_v = 1."""
    f = W.to_f64
    ch = head_channels(shape, h)
    D = shape.d_v
    x = f(inp["mixed_qkv"][:, ch])
    cs = None if inp["conv_state0"] is None else f(inp["conv_state0"][:, ch])
    S0 = None if inp["S0"] is None else f(inp["S0"][:, h:h + 1])
    return oracle.layer_prefill(
        x, f(inp["z"][:, h * D:(h + 1) * D]), f(inp["a"][:, h:h + 1]), f(inp["b"][:, h:h + 1]),
        f(inp["conv_w"][ch]), f(inp["A_log"][h:h + 1]), f(inp["dt_bias"][h:h + 1]),
        f(inp["norm_w"]), 1, 1, shape.d_k, shape.d_v, cu_seqlens=inp["cu_seqlens"].numpy(),
        S0=S0, conv_state0=cs, ckpt_every=ckpt_every, nthreads=1)


def oracle_heads_prefill(inp, shape, heads, ckpt_every=0):
    with ThreadPoolExecutor(max(1, min(len(heads), oracle.max_threads()))) as ex:
        return dict(zip(heads, ex.map(lambda h: oracle_head_prefill(inp, shape, h, ckpt_every),
                                      heads)))


def rounded_to(dtype):
    """f64 array -> the nearest values of the activation dtype, as f64."""
    return lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dtype).to(torch.float64).numpy()


def oracle_step_in_activation_dtype(x, z, a, b, conv_w, A_log, dt_bias, norm_w, s, S, conv_state, rnd):
    """One decode step of B sequences by the oracle's definitions, with the
    conv output y and the rule's output o rounded to the activation dtype
    where the layer's calls hand them on (each call's output is an activation
    of that dtype).  Returns (out, S_new, conv_state_new)."""
    cu = np.arange(x.shape[0] + 1, dtype=np.int64)
    y, cs_new, _ = oracle.conv1d(x, conv_w, cu, conv_state, True, 0)
    q, k, v = oracle.split_qkv(rnd(y), s.H_k, s.H_v, s.d_k, s.d_v)
    g, beta = oracle.gates(a, b, A_log, dt_bias)
    o, S_new, _ = oracle.delta_rule(q, k, v, g, beta, cu, S, None, True, 0)
    return oracle.rmsnorm_gated(rnd(o), z, norm_w), S_new, cs_new

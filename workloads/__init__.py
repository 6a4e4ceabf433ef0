"""Seeded synthetic inputs for the Gated DeltaNet layer core.

This module is shared by the CPU oracle side and the CUDA side of the tests and
of ``bench.py``.  It only draws random numbers and lays them out; it holds none
of the layer's arithmetic (no convolution, gating, normalisation or state
update).

Every tensor is drawn blockwise: element block ``i`` of tensor stream ``s``
comes from ``numpy.random.Philox`` seeded with ``SeedSequence([seed, s, i])``,
so the values do not depend on how many threads draw them.  Values are drawn in
float32 and then rounded once to the workload dtype (bf16 or f32); both sides
read those same rounded values (the oracle widens them exactly to f64).

Distributions (the workloads of the Qwen3.6-27B / Qwen3-Coder-Next GDN layer
pages; "N(mu, s)" means mean mu and standard deviation s):

* mixed_qkv, z, a, b ~ N(0, 1)
* depthwise conv weight [conv_dim, 4] ~ N(0, 0.25)
* A_log = ln U(1, 16), dt_bias = ln(expm1(U(1e-3, 0.1)))      (f32)
* RMSNormGated weight [d_v] ~ N(1, 0.1)
* recurrent initial state ~ N(0, 0.02) (f32), conv initial state ~ N(0, 1)
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 1 << 22  # elements per independently seeded block

# stream ids: one per tensor role, so adding a tensor never shifts another's values
_STREAM = {
    "mixed_qkv": 1, "z": 2, "a": 3, "b": 4, "conv_w": 5, "A_log": 6, "dt_bias": 7,
    "norm_w": 8, "S0": 9, "conv_state0": 10, "lengths": 11,
    "dec_qkv": 21, "dec_z": 22, "dec_a": 23, "dec_b": 24,
}


@dataclass(frozen=True)
class GDNShape:
    """Head layout of one GDN layer (config fields linear_num_key_heads, ...)."""
    H_k: int
    H_v: int
    d_k: int
    d_v: int
    conv_k: int = 4

    @property
    def conv_dim(self) -> int:
        return 2 * self.H_k * self.d_k + self.H_v * self.d_v

    @property
    def z_dim(self) -> int:
        return self.H_v * self.d_v


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    shape: GDNShape
    dtype: torch.dtype
    lengths: tuple = ()
    init_state: bool = False
    ckpt_every: int = 0
    decode_batch: int = 0
    decode_steps: int = 0
    notes: str = ""

    @property
    def seed(self) -> int:
        return 1000 + self.index


QWEN36_27B = GDNShape(H_k=16, H_v=48, d_k=128, d_v=128)
CODER_NEXT = GDNShape(H_k=16, H_v=32, d_k=128, d_v=128)
TINY = GDNShape(H_k=2, H_v=4, d_k=16, d_v=16)


def _varlen_lengths(seed: int, n: int = 8, total: int = 32768, lo: int = 512,
                    hi: int = 8192) -> tuple:
    """n lengths drawn i.i.d. from U{lo..hi}, rescaled to sum to `total`,
    clamped to [lo, hi]; the residual is spread +-1 within the bounds.  The
    draw is repeated with the next sub-seed until at least one length is not a
    multiple of 64 (so a ragged last chunk is always exercised)."""
    for attempt in range(100):
        rng = np.random.Generator(np.random.Philox(
            np.random.SeedSequence([seed, _STREAM["lengths"], attempt])))
        raw = rng.integers(lo, hi + 1, size=n).astype(np.float64)
        L = np.clip(np.rint(raw * total / raw.sum()), lo, hi).astype(np.int64)
        i = 0
        while L.sum() != total:
            step = 1 if L.sum() < total else -1
            if lo <= L[i % n] + step <= hi:
                L[i % n] += step
            i += 1
        if np.any(L % 64 != 0):
            return tuple(int(x) for x in L)
    raise RuntimeError("no ragged length set found")


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_f32", 0, TINY, torch.float32, lengths=(64,),
                 notes="B=1, T=64, f32 everywhere, zero initial states"),
        Workload("qwen36_27b_prefill", 1, QWEN36_27B, torch.bfloat16, lengths=(4096,),
                 notes="B=1, T=4096, bf16 activations, f32 state, zero initial states"),
        Workload("qwen36_27b_decode", 2, QWEN36_27B, torch.bfloat16, init_state=True,
                 decode_batch=64, decode_steps=256,
                 notes="64 sequences x 256 single-token steps from N(0,0.02) state"),
        Workload("coder_next_varlen", 3, CODER_NEXT, torch.bfloat16,
                 lengths=_varlen_lengths(1003), init_state=True,
                 notes="8 packed sequences summing to 32768 tokens, resumed prefix"),
        Workload("qwen36_27b_long", 4, QWEN36_27B, torch.bfloat16, lengths=(262144,),
                 ckpt_every=4096, decode_batch=1, decode_steps=128,
                 notes="one 262144-token sequence, checkpoints every 4096 tokens, "
                       "then 128 decode steps"),
    ]
}


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _fill(out: np.ndarray, seed: int, stream: int, kind: str, p0: float, p1: float):
    flat = out.reshape(-1)
    nblk = (flat.size + BLOCK - 1) // BLOCK

    def one(i):
        rng = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream, i])))
        seg = flat[i * BLOCK:(i + 1) * BLOCK]
        if kind == "normal":
            rng.standard_normal(dtype=np.float32, out=seg)
            if p1 != 1.0:
                seg *= np.float32(p1)
            if p0 != 0.0:
                seg += np.float32(p0)
        else:  # uniform [p0, p1)
            rng.random(dtype=np.float32, out=seg)
            seg *= np.float32(p1 - p0)
            seg += np.float32(p0)

    if nblk == 1:
        one(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(one, range(nblk)))


def draw(shape, *, seed: int, stream: int, dtype: torch.dtype, kind: str = "normal",
         p0: float = 0.0, p1: float = 1.0) -> torch.Tensor:
    """A seeded tensor: N(p0, p1) for kind='normal', U(p0, p1) for 'uniform',
    drawn in float32 and rounded once to `dtype`."""
    buf = np.empty(tuple(shape), dtype=np.float32)
    if buf.size:
        _fill(buf, seed, stream, kind, p0, p1)
    t = torch.from_numpy(buf)
    return t if dtype == torch.float32 else t.to(dtype)


def layer_params(shape: GDNShape, dtype: torch.dtype, seed: int) -> dict:
    """Per-layer parameters: conv weight, A_log, dt_bias, RMSNormGated weight."""
    u_A = draw((shape.H_v,), seed=seed, stream=_STREAM["A_log"], dtype=torch.float32,
               kind="uniform", p0=1.0, p1=16.0)
    u_dt = draw((shape.H_v,), seed=seed, stream=_STREAM["dt_bias"], dtype=torch.float32,
                kind="uniform", p0=1e-3, p1=0.1)
    return {
        "conv_w": draw((shape.conv_dim, shape.conv_k), seed=seed, stream=_STREAM["conv_w"],
                       dtype=dtype, p1=0.25),
        "A_log": torch.log(u_A.double()).float(),
        "dt_bias": torch.log(torch.expm1(u_dt.double())).float(),
        "norm_w": draw((shape.d_v,), seed=seed, stream=_STREAM["norm_w"], dtype=dtype,
                       p0=1.0, p1=0.1),
    }


def cu_seqlens_of(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def layer_inputs(shape: GDNShape, dtype: torch.dtype, lengths, *, seed: int,
                 init_state: bool = False) -> dict:
    """Prefill inputs of one layer: packed tokens of len(lengths) sequences.

    Returns CPU tensors: mixed_qkv [T, conv_dim], z [T, H_v*d_v], a, b [T, H_v]
    (all `dtype`), the layer parameters, cu_seqlens int32 [N+1], and S0
    [N, H_v, d_k, d_v] f32 / conv_state0 [N, conv_dim, conv_k-1] (`dtype`), both
    None when init_state is False (zero initial state)."""
    T = int(sum(lengths))
    N = len(lengths)
    d = {
        "mixed_qkv": draw((T, shape.conv_dim), seed=seed, stream=_STREAM["mixed_qkv"], dtype=dtype),
        "z": draw((T, shape.z_dim), seed=seed, stream=_STREAM["z"], dtype=dtype),
        "a": draw((T, shape.H_v), seed=seed, stream=_STREAM["a"], dtype=dtype),
        "b": draw((T, shape.H_v), seed=seed, stream=_STREAM["b"], dtype=dtype),
        "cu_seqlens": cu_seqlens_of(lengths),
        "S0": None,
        "conv_state0": None,
    }
    d.update(layer_params(shape, dtype, seed))
    if init_state:
        d["S0"] = draw((N, shape.H_v, shape.d_k, shape.d_v), seed=seed, stream=_STREAM["S0"],
                       dtype=torch.float32, p1=0.02)
        d["conv_state0"] = draw((N, shape.conv_dim, shape.conv_k - 1), seed=seed,
                                stream=_STREAM["conv_state0"], dtype=dtype)
    return d


def decode_inputs(shape: GDNShape, dtype: torch.dtype, batch: int, steps: int, *,
                  seed: int) -> dict:
    """Per-step decode inputs: qkv [steps, B, conv_dim], z [steps, B, H_v*d_v],
    a, b [steps, B, H_v] (`dtype`)."""
    return {
        "qkv": draw((steps, batch, shape.conv_dim), seed=seed, stream=_STREAM["dec_qkv"], dtype=dtype),
        "z": draw((steps, batch, shape.z_dim), seed=seed, stream=_STREAM["dec_z"], dtype=dtype),
        "a": draw((steps, batch, shape.H_v), seed=seed, stream=_STREAM["dec_a"], dtype=dtype),
        "b": draw((steps, batch, shape.H_v), seed=seed, stream=_STREAM["dec_b"], dtype=dtype),
    }


def workload_inputs(name: str, *, lengths=None) -> dict:
    """Inputs of a named workload (optionally with other sequence lengths but
    the same shapes, distributions and seed)."""
    w = WORKLOADS[name]
    if w.decode_batch and not w.lengths:
        d = decode_inputs(w.shape, w.dtype, w.decode_batch, w.decode_steps, seed=w.seed)
        d.update(layer_params(w.shape, w.dtype, w.seed))
        d["S0"] = draw((w.decode_batch, w.shape.H_v, w.shape.d_k, w.shape.d_v), seed=w.seed,
                       stream=_STREAM["S0"], dtype=torch.float32, p1=0.02)
        d["conv_state0"] = draw((w.decode_batch, w.shape.conv_dim, w.shape.conv_k - 1),
                                seed=w.seed, stream=_STREAM["conv_state0"], dtype=w.dtype)
        return d
    return layer_inputs(w.shape, w.dtype, lengths or w.lengths, seed=w.seed,
                        init_state=w.init_state)


def to_f64(t):
    """Exact widening to a float64 numpy array (None passes through)."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()

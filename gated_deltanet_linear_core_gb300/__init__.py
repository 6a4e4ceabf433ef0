"""Gated DeltaNet (GDN) linear-attention layer core for GB300 (sm_103a).

A thin binding of the C ABI in include/gdn.h (libgdn.so, hand-written CUDA
kernels).  The functions below only marshal arguments: they check tensor
placement and layout, allocate outputs with torch when the caller passes none,
and call the library on the current CUDA stream.  Every step of the layer runs
in the library's kernels; if libgdn.so is missing, every call raises.

Layer core (cortex commit "feat(stage-8c): linear-attention layer (Qwen3-Next
GatedDeltaNet)"): conv1d(k=4)+SiLU -> split [q|k|v] -> l2norm(q,k), gates
g = -exp(A_log) softplus(a+dt_bias), beta = sigmoid(b) -> gated delta rule
(chunked prefill or per-token decode) -> RMSNormGated(o, z).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib
from ._lib import GDNError, GDN_QK_L2NORM, GDN_SOLVE_NEUMANN, GDN_CHUNK  # noqa: F401

__all__ = [
    "GDNDims", "GDNError", "gdn_conv1d_fwd", "gdn_conv1d_update", "gdn_chunk_prefill",
    "gdn_chunk_prefill_workspace_size", "gdn_chunk_prefill_launches", "gdn_chunk_prefill_noalloc", "gdn_recurrent_decode", "gdn_rmsnorm_gated",
    "gdn_ckpt_count", "gdn_check_cu_seqlens", "gdn_sync_status", "gdn_selftest_bounded_wait",
    "gdn_layer_prefill_host", "gdn_decode_step", "gdn_decode_verify", "gdn_layer_prefill",
    "gdn_layer_prefill_workspace_size", "gdn_layer_prefill_launches", "gdn_chunk_prefill_norm",
    "HeadShard", "head_shard",
    "gdn_layer_decode",
    "library_path",
]

RMSNORM_EPS = 1e-6


@dataclass(frozen=True)
class GDNDims:
    """H_k query/key heads, H_v value heads, head dims d_k = d_v, conv width 4."""
    H_k: int
    H_v: int
    d_k: int
    d_v: int
    conv_k: int = 4

    @property
    def conv_dim(self) -> int:
        return 2 * self.H_k * self.d_k + self.H_v * self.d_v


def library_path() -> str:
    return _lib.LIB_PATH


def _dims(d) -> _lib.Dims:
    return _lib.Dims(int(d.H_k), int(d.H_v), int(d.d_k), int(d.d_v), int(getattr(d, "conv_k", 4)))


def _conv_dim(d) -> int:
    return 2 * int(d.H_k) * int(d.d_k) + int(d.H_v) * int(d.d_v)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.GDN_BF16
    if t.dtype == torch.float32:
        return _lib.GDN_F32
    raise TypeError(f"unsupported activation dtype {t.dtype} (bfloat16 or float32)")


def _ptr(t, name, dtype=None, shape=None):
    """Device pointer of a contiguous CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr() if t.numel() else None


def _stream(t: torch.Tensor, stream):
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return torch.cuda.current_stream(t.device).cuda_stream


def _nseq(cu_seqlens):
    return 1 if cu_seqlens is None else int(cu_seqlens.numel()) - 1


def gdn_ckpt_count(cu_seqlens, every: int) -> int:
    """Checkpoint rows for packed sequences (host offsets: list, numpy or CPU tensor)."""
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int32, device="cpu").contiguous()
    r = _lib.load().gdn_ckpt_count(cu.data_ptr(), int(cu.numel()) - 1, int(every))
    if r < 0:
        raise ValueError("invalid cu_seqlens or checkpoint interval")
    return int(r)


def gdn_check_cu_seqlens(cu_seqlens: torch.Tensor, T_tot: int, stream=None) -> None:
    """Validates device offsets (synchronises the stream)."""
    p = _ptr(cu_seqlens, "cu_seqlens", torch.int32)
    _lib.check(_lib.load().gdn_check_cu_seqlens(p, _nseq(cu_seqlens), int(T_tot),
                                               _stream(cu_seqlens, stream)),
               "gdn_check_cu_seqlens")


def gdn_sync_status(device=None, stream=None) -> None:
    """Synchronises the stream and raises GDNError if a kernel gave up a
    bounded device-side wait (GDN_ERR_TIMEOUT) or the stream holds a CUDA error."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _lib.check(_lib.load().gdn_sync_status(s), "gdn_sync_status")


def gdn_selftest_bounded_wait(limit_ns: int = 1_000_000, device=None, stream=None) -> None:
    """Enqueues one kernel whose bounded wait runs out after limit_ns (nothing
    arrives at its barrier); the next gdn_sync_status raises GDN_ERR_TIMEOUT."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _lib.check(_lib.load().gdn_selftest_bounded_wait(int(limit_ns), s), "gdn_selftest_bounded_wait")


def gdn_conv1d_fwd(x, w, dims, cu_seqlens=None, conv_state_in=None, conv_state_out=None,
                   ckpt_every=0, conv_ckpt_out=None, apply_silu=True, y=None, stream=None):
    """Prefill depthwise causal conv1d(k=4) with state prepend (+SiLU).
    x [T, conv_dim]; w [conv_dim, 4]; states [n_seq, conv_dim, 3];
    checkpoints [rows, conv_dim, 3].  Returns y [T, conv_dim]."""
    dt = x.dtype
    T, C = x.shape
    if C != _conv_dim(dims):
        raise ValueError(f"x has {C} channels, dims give {_conv_dim(dims)}")
    if y is None:
        y = torch.empty_like(x)
    rows = 0 if conv_ckpt_out is None else int(conv_ckpt_out.shape[0])
    st = _lib.load().gdn_conv1d_fwd(
        _ptr(x, "x", dt), _ptr(w, "w", dt, (C, 4)), _ptr(cu_seqlens, "cu_seqlens", torch.int32),
        _nseq(cu_seqlens), T, _ptr(conv_state_in, "conv_state_in", dt),
        _ptr(conv_state_out, "conv_state_out", dt), int(ckpt_every),
        _ptr(conv_ckpt_out, "conv_ckpt_out", dt), rows, int(bool(apply_silu)),
        _ptr(y, "y", dt, (T, C)), _dims(dims), _dtype_code(x), _stream(x, stream))
    _lib.check(st, "gdn_conv1d_fwd")
    return y


def gdn_conv1d_update(x, w, conv_state, dims, apply_silu=True, y=None, stream=None):
    """Decode conv for B sequences; conv_state [B, conv_dim, 3] shifted in place."""
    dt = x.dtype
    B, C = x.shape
    if y is None:
        y = torch.empty_like(x)
    st = _lib.load().gdn_conv1d_update(
        _ptr(x, "x", dt), _ptr(w, "w", dt, (C, 4)), _ptr(conv_state, "conv_state", dt, (B, C, 3)),
        B, int(bool(apply_silu)), _ptr(y, "y", dt, (B, C)), _dims(dims), _dtype_code(x),
        _stream(x, stream))
    _lib.check(st, "gdn_conv1d_update")
    return y


def gdn_chunk_prefill_workspace_size(n_seq: int, T_tot: int, dims, dtype) -> int:
    code = _lib.GDN_BF16 if dtype == torch.bfloat16 else _lib.GDN_F32
    return int(_lib.load().gdn_chunk_prefill_workspace_size(int(n_seq), int(T_tot), _dims(dims),
                                                            code))


def gdn_chunk_prefill_launches(n_seq: int, T_tot: int, dims, dtype, cu_seqlens=True, chunk=64) -> int:
    """Kernel launches of one gdn_chunk_prefill call; cu_seqlens: whether the
    call passes cu_seqlens (a truthy value) or not (None / False); chunk: its
    chunk size (16, 32 or 64)."""
    code = _lib.GDN_BF16 if dtype == torch.bfloat16 else _lib.GDN_F32
    has_cu = 0 if cu_seqlens is None or cu_seqlens is False else 1
    return int(_lib.load().gdn_chunk_prefill_launches(int(n_seq), int(T_tot), has_cu, _dims(dims), code,
                                                      _flags(False, "direct", chunk)))


def _flags(l2norm_qk, solve, chunk) -> int:
    if solve not in ("direct", "neumann"):
        raise ValueError(f"solve must be 'direct' or 'neumann', not {solve!r}")
    return ((_lib.GDN_QK_L2NORM if l2norm_qk else 0) | (_lib.GDN_SOLVE_NEUMANN if solve == "neumann" else 0) |
            (0 if chunk == 64 else _lib.GDN_CHUNK(chunk)))


def _gate_ptrs(a, b, A_log, dt_bias, g, beta, dt):
    return (_ptr(a, "a", dt), _ptr(b, "b", dt), _ptr(A_log, "A_log", torch.float32),
            _ptr(dt_bias, "dt_bias", torch.float32), _ptr(g, "g", torch.float32),
            _ptr(beta, "beta", torch.float32))


def gdn_chunk_prefill(qkv, dims, a=None, b=None, A_log=None, dt_bias=None, g=None, beta=None,
                      cu_seqlens=None, initial_state=None, final_state=None, ckpt_every=0,
                      state_ckpt_out=None, scale=0.0, l2norm_qk=True, o=None, workspace=None,
                      stream=None, solve="direct", chunk=64):
    """Chunked gated delta rule over packed sequences.  qkv [T, conv_dim]
    (post-conv); states [n_seq, H_v, d_k, d_v] f32; returns o [T, H_v, d_v].
    solve="neumann" forms each chunk's (I + A)^-1 as the Neumann-style product
    (GDN_SOLVE_NEUMANN; tensor-core path only).  chunk: 16, 32 or 64 tokens
    (GDN_CHUNK; on the tensor-core path 16 and 32 need final_state)."""
    if solve not in ("direct", "neumann"):
        raise ValueError(f"solve must be 'direct' or 'neumann', not {solve!r}")
    dt = qkv.dtype
    T = int(qkv.shape[0])
    if o is None:
        o = torch.empty((T, dims.H_v, dims.d_v), dtype=dt, device=qkv.device)
    rows = 0 if state_ckpt_out is None else int(state_ckpt_out.shape[0])
    lib = _lib.load()
    if workspace is None:
        need = lib.gdn_chunk_prefill_workspace_size(_nseq(cu_seqlens), T, _dims(dims),
                                                    _dtype_code(qkv))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=qkv.device)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.gdn_chunk_prefill(
        _ptr(qkv, "qkv", dt), *_gate_ptrs(a, b, A_log, dt_bias, g, beta, dt),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32), _nseq(cu_seqlens), T,
        _ptr(initial_state, "initial_state", torch.float32),
        _ptr(final_state, "final_state", torch.float32), int(ckpt_every),
        _ptr(state_ckpt_out, "state_ckpt_out", torch.float32), rows, float(scale),
        _flags(l2norm_qk, solve, chunk), _ptr(o, "o", dt), _ptr(workspace, "workspace"),
        ws, _dims(dims), _dtype_code(qkv), _stream(qkv, stream))
    _lib.check(st, "gdn_chunk_prefill")
    return o


def gdn_chunk_prefill_norm(qkv, z, norm_w, dims, a=None, b=None, A_log=None, dt_bias=None, g=None,
                           beta=None, cu_seqlens=None, initial_state=None, final_state=None, ckpt_every=0,
                           state_ckpt_out=None, scale=0.0, l2norm_qk=True, norm_eps=RMSNORM_EPS, out=None,
                           workspace=None, stream=None, solve="direct", chunk=64):
    """gdn_chunk_prefill followed by RMSNormGated(o, z): returns out [T, H_v*d_v]
    (the rule's output is normalised in place in `out`)."""
    if solve not in ("direct", "neumann"):
        raise ValueError(f"solve must be 'direct' or 'neumann', not {solve!r}")
    dt = qkv.dtype
    T = int(qkv.shape[0])
    if out is None:
        out = torch.empty((T, dims.H_v * dims.d_v), dtype=dt, device=qkv.device)
    rows = 0 if state_ckpt_out is None else int(state_ckpt_out.shape[0])
    lib = _lib.load()
    if workspace is None:
        need = lib.gdn_chunk_prefill_workspace_size(_nseq(cu_seqlens), T, _dims(dims), _dtype_code(qkv))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=qkv.device)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.gdn_chunk_prefill_norm(
        _ptr(qkv, "qkv", dt), *_gate_ptrs(a, b, A_log, dt_bias, g, beta, dt),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32), _nseq(cu_seqlens), T,
        _ptr(initial_state, "initial_state", torch.float32),
        _ptr(final_state, "final_state", torch.float32), int(ckpt_every),
        _ptr(state_ckpt_out, "state_ckpt_out", torch.float32), rows, float(scale),
        _flags(l2norm_qk, solve, chunk), _ptr(z, "z", dt, (T, dims.H_v * dims.d_v)), _ptr(norm_w, "norm_w", dt, (dims.d_v,)), float(norm_eps),
        _ptr(out, "out", dt, (T, dims.H_v * dims.d_v)), _ptr(workspace, "workspace"), ws, _dims(dims),
        _dtype_code(qkv), _stream(qkv, stream))
    _lib.check(st, "gdn_chunk_prefill_norm")
    return out


def gdn_chunk_prefill_noalloc(qkv, dims, o, final_state, a=None, b=None, A_log=None,
                              dt_bias=None, g=None, beta=None, cu_seqlens=None,
                              initial_state=None, ckpt_every=0, state_ckpt_out=None, scale=0.0,
                              l2norm_qk=True, stream=None):
    """gdn_chunk_prefill for callers that cannot allocate device memory: its
    scratch is a fixed array inside the library, and this binding allocates
    nothing either -- the caller passes every output (o [T, H_v, d_v] and
    final_state [n_seq, H_v, d_k, d_v] f32, plus state_ckpt_out when
    checkpointing).  bf16, d = 128 only.  Calls that overlap on the GPU share
    the array and race; the first call on a device should precede any stream
    capture."""
    dt = qkv.dtype
    T = int(qkv.shape[0])
    rows = 0 if state_ckpt_out is None else int(state_ckpt_out.shape[0])
    st = _lib.load().gdn_chunk_prefill_noalloc(
        _ptr(qkv, "qkv", dt), *_gate_ptrs(a, b, A_log, dt_bias, g, beta, dt),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32), _nseq(cu_seqlens), T,
        _ptr(initial_state, "initial_state", torch.float32),
        _ptr(final_state, "final_state", torch.float32), int(ckpt_every),
        _ptr(state_ckpt_out, "state_ckpt_out", torch.float32), rows, float(scale),
        _lib.GDN_QK_L2NORM if l2norm_qk else 0, _ptr(o, "o", dt, (T, dims.H_v, dims.d_v)),
        _dims(dims), _dtype_code(qkv), _stream(qkv, stream))
    _lib.check(st, "gdn_chunk_prefill_noalloc")
    return o


def gdn_recurrent_decode(qkv, state, dims, a=None, b=None, A_log=None, dt_bias=None, g=None,
                         beta=None, scale=0.0, l2norm_qk=True, o=None, stream=None):
    """One decode step for B sequences; state [B, H_v, d_k, d_v] f32 in place.
    Returns o [B, H_v, d_v]."""
    dt = qkv.dtype
    B = int(qkv.shape[0])
    if o is None:
        o = torch.empty((B, dims.H_v, dims.d_v), dtype=dt, device=qkv.device)
    st = _lib.load().gdn_recurrent_decode(
        _ptr(qkv, "qkv", dt), *_gate_ptrs(a, b, A_log, dt_bias, g, beta, dt),
        _ptr(state, "state", torch.float32, (B, dims.H_v, dims.d_k, dims.d_v)), B, float(scale),
        _lib.GDN_QK_L2NORM if l2norm_qk else 0, _ptr(o, "o", dt), _dims(dims), _dtype_code(qkv),
        _stream(qkv, stream))
    _lib.check(st, "gdn_recurrent_decode")
    return o


def gdn_rmsnorm_gated(o, z, w, dims, eps=RMSNORM_EPS, out=None, stream=None):
    """RMSNormGated per value head: o [T, H_v, d_v], z [T, H_v*d_v] -> out [T, H_v*d_v]."""
    dt = o.dtype
    T = int(o.shape[0])
    if out is None:
        out = torch.empty((T, dims.H_v * dims.d_v), dtype=dt, device=o.device)
    st = _lib.load().gdn_rmsnorm_gated(
        _ptr(o, "o", dt), _ptr(z, "z", dt), _ptr(w, "w", dt, (dims.d_v,)), float(eps), T,
        _ptr(out, "out", dt), _dims(dims), _dtype_code(o), _stream(o, stream))
    _lib.check(st, "gdn_rmsnorm_gated")
    return out


def gdn_layer_prefill_workspace_size(n_seq: int, T_tot: int, dims, dtype) -> int:
    code = _lib.GDN_BF16 if dtype == torch.bfloat16 else _lib.GDN_F32
    return int(_lib.load().gdn_layer_prefill_workspace_size(int(n_seq), int(T_tot), _dims(dims), code))


def gdn_layer_prefill_launches(n_seq: int, T_tot: int, dims, dtype, cu_seqlens=True, chunk=64) -> int:
    """Kernel launches of one gdn_layer_prefill call (cu_seqlens and chunk as
    in gdn_chunk_prefill_launches)."""
    code = _lib.GDN_BF16 if dtype == torch.bfloat16 else _lib.GDN_F32
    has_cu = 0 if cu_seqlens is None or cu_seqlens is False else 1
    return int(_lib.load().gdn_layer_prefill_launches(int(n_seq), int(T_tot), has_cu, _dims(dims), code,
                                                      _flags(False, "direct", chunk)))


def gdn_layer_prefill(mixed_qkv, z, a, b, conv_w, A_log, dt_bias, norm_w, dims, cu_seqlens=None,
                      initial_state=None, conv_state=None, ckpt_every=0, scale=0.0,
                      return_intermediates=False, stream=None, norm_eps=RMSNORM_EPS, out=None,
                      final_state=None, conv_state_out=None, workspace=None, solve="direct", chunk=64,
                      state_ckpt_out=None, conv_ckpt_out=None):
    """Whole layer core over packed sequences: conv1d+SiLU -> chunked delta rule
    -> RMSNormGated, as one gdn_layer_prefill call (bf16, d = 128: the conv
    inside the chunk kernels).  Returns a dict with out
    [T, H_v*d_v], final_state [n_seq, H_v, d_k, d_v] f32, conv_state
    [n_seq, conv_dim, 3] and, when ckpt_every > 0, state_ckpt / conv_ckpt.
    return_intermediates=True runs the three calls one by one instead and adds
    the conv output y and the rule's output o to the dict.  state_ckpt_out and
    conv_ckpt_out may pass preallocated checkpoint buffers."""
    if solve not in ("direct", "neumann"):
        raise ValueError(f"solve must be 'direct' or 'neumann', not {solve!r}")
    dev, dt = mixed_qkv.device, mixed_qkv.dtype
    T = int(mixed_qkv.shape[0])
    n_seq = _nseq(cu_seqlens)
    C = _conv_dim(dims)
    rows = 0
    if ckpt_every:
        host_cu = (cu_seqlens.to("cpu") if cu_seqlens is not None
                   else torch.tensor([0, T], dtype=torch.int32))
        rows = gdn_ckpt_count(host_cu, ckpt_every)
    if conv_state_out is None:
        conv_state_out = torch.empty((n_seq, C, 3), dtype=dt, device=dev)
    conv_ck = conv_ckpt_out
    if conv_ck is None and rows:
        conv_ck = torch.empty((rows, C, 3), dtype=dt, device=dev)
    if final_state is None:
        final_state = torch.empty((n_seq, dims.H_v, dims.d_k, dims.d_v), dtype=torch.float32, device=dev)
    S_ck = state_ckpt_out
    if S_ck is None and rows:
        S_ck = torch.empty((rows, dims.H_v, dims.d_k, dims.d_v), dtype=torch.float32, device=dev)
    if rows and (tuple(S_ck.shape) != (rows, dims.H_v, dims.d_k, dims.d_v) or
                 tuple(conv_ck.shape) != (rows, C, 3)):
        raise ValueError(f"checkpoint buffers must hold {rows} rows")
    if return_intermediates:
        y = gdn_conv1d_fwd(mixed_qkv, conv_w, dims, cu_seqlens, conv_state, conv_state_out, ckpt_every,
                           conv_ck, True, stream=stream)
        o = gdn_chunk_prefill(y, dims, a, b, A_log, dt_bias, cu_seqlens=cu_seqlens,
                              initial_state=initial_state, final_state=final_state, ckpt_every=ckpt_every,
                              state_ckpt_out=S_ck, scale=scale, stream=stream, solve=solve, chunk=chunk)
        out = gdn_rmsnorm_gated(o, z, norm_w, dims, eps=norm_eps, out=out, stream=stream)
        return {"out": out, "final_state": final_state, "conv_state": conv_state_out, "state_ckpt": S_ck,
                "conv_ckpt": conv_ck, "y": y, "o": o}
    if out is None:
        out = torch.empty((T, dims.H_v * dims.d_v), dtype=dt, device=dev)
    lib = _lib.load()
    if workspace is None:
        need = lib.gdn_layer_prefill_workspace_size(n_seq, T, _dims(dims), _dtype_code(mixed_qkv))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.gdn_layer_prefill(
        _ptr(mixed_qkv, "mixed_qkv", dt, (T, C)), _ptr(z, "z", dt), _ptr(a, "a", dt), _ptr(b, "b", dt),
        _ptr(conv_w, "conv_w", dt, (C, 4)), _ptr(A_log, "A_log", torch.float32),
        _ptr(dt_bias, "dt_bias", torch.float32), _ptr(norm_w, "norm_w", dt, (dims.d_v,)), float(norm_eps),
        _ptr(cu_seqlens, "cu_seqlens", torch.int32), n_seq, T,
        _ptr(initial_state, "initial_state", torch.float32),
        _ptr(final_state, "final_state", torch.float32, (n_seq, dims.H_v, dims.d_k, dims.d_v)),
        _ptr(conv_state, "conv_state", dt), _ptr(conv_state_out, "conv_state_out", dt, (n_seq, C, 3)),
        int(ckpt_every), _ptr(S_ck, "state_ckpt", torch.float32), _ptr(conv_ck, "conv_ckpt", dt), rows,
        float(scale),
        _flags(True, solve, chunk),
        _ptr(out, "out", dt, (T, dims.H_v * dims.d_v)), _ptr(workspace, "workspace"), ws, _dims(dims),
        _dtype_code(mixed_qkv), _stream(mixed_qkv, stream))
    _lib.check(st, "gdn_layer_prefill")
    return {"out": out, "final_state": final_state, "conv_state": conv_state_out, "state_ckpt": S_ck,
            "conv_ckpt": conv_ck}


def _hptr(t, name, dtype=None, shape=None):
    """Address of a contiguous page-locked CPU tensor."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cpu" or not t.is_pinned():
        raise ValueError(f"{name}: must be a page-locked (pinned) CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr() if t.numel() else None


def gdn_layer_prefill_host(h_qkv, h_z, h_a, h_b, conv_w, A_log, dt_bias, norm_w, dims,
                           initial_state=None, conv_state_in=None, scale=0.0, l2norm=True,
                           norm_eps=1e-6, h_out=None, final_state=None, conv_state_out=None,
                           workspace=None, stream=None):
    """The layer core for one sequence whose activations (h_qkv [T, conv_dim],
    h_z [T, H_v*d_v], h_a, h_b [T, H_v]) and output h_out are pinned CPU tensors;
    parameters and states are CUDA tensors.  Copies in, kernels and copies out
    overlap piece by piece inside the library.  Returns a dict with out (the
    pinned host tensor; complete once the stream reaches this point),
    final_state [1, H_v, d_k, d_v] f32 and conv_state [1, conv_dim, 3]."""
    dt = h_qkv.dtype
    dev = conv_w.device
    T = int(h_qkv.shape[0])
    C, O = _conv_dim(dims), int(dims.H_v) * int(dims.d_v)
    code = _dtype_code(h_qkv)
    if h_out is None:
        h_out = torch.empty((T, O), dtype=dt).pin_memory()
    if final_state is None:
        final_state = torch.empty((1, dims.H_v, dims.d_k, dims.d_v), dtype=torch.float32, device=dev)
    if conv_state_out is None:
        conv_state_out = torch.empty((1, C, 3), dtype=dt, device=dev)
    lib = _lib.load()
    need = lib.gdn_layer_prefill_host_workspace_size(T, _dims(dims), code)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    st = lib.gdn_layer_prefill_host(
        _hptr(h_qkv, "h_qkv", dt, (T, C)), _hptr(h_z, "h_z", dt, (T, O)),
        _hptr(h_a, "h_a", dt, (T, dims.H_v)), _hptr(h_b, "h_b", dt, (T, dims.H_v)),
        _ptr(conv_w, "conv_w", dt, (C, 4)), _ptr(A_log, "A_log", torch.float32),
        _ptr(dt_bias, "dt_bias", torch.float32), _ptr(norm_w, "norm_w", dt), T,
        _ptr(initial_state, "initial_state", torch.float32), _ptr(final_state, "final_state", torch.float32),
        _ptr(conv_state_in, "conv_state_in", dt), _ptr(conv_state_out, "conv_state_out", dt),
        float(scale), _lib.GDN_QK_L2NORM if l2norm else 0, float(norm_eps),
        _hptr(h_out, "h_out", dt, (T, O)), _ptr(workspace, "workspace", torch.uint8),
        workspace.numel() if workspace is not None else 0, _dims(dims), code, _stream(conv_w, stream))
    _lib.check(st, "gdn_layer_prefill_host")
    return {"out": h_out, "final_state": final_state, "conv_state": conv_state_out}


def gdn_decode_step(x, z, a, b, conv_w, A_log, dt_bias, norm_w, dims, state, conv_state,
                    slots=None, scale=0.0, l2norm=True, norm_eps=1e-6, out=None, stream=None):
    """One fused decode step (conv update, gates, recurrence, RMSNormGated) in
    one kernel for B sequences; x [B, conv_dim], z [B, H_v*d_v], a, b [B, H_v];
    state [n_slots, H_v, d_k, d_v] f32 and conv_state [n_slots, conv_dim, 3]
    are updated in place at slots[b] (int32 [B], distinct) or at b.  Returns
    out [B, H_v*d_v]."""
    dt = x.dtype
    B = int(x.shape[0])
    C, O = _conv_dim(dims), int(dims.H_v) * int(dims.d_v)
    if out is None:
        out = torch.empty((B, O), dtype=dt, device=x.device)
    if state.dim() != 4 or tuple(state.shape[1:]) != (dims.H_v, dims.d_k, dims.d_v):
        raise ValueError("state: expected [n_slots, H_v, d_k, d_v]")
    if conv_state.dim() != 3 or tuple(conv_state.shape[1:]) != (C, 3):
        raise ValueError("conv_state: expected [n_slots, conv_dim, 3]")
    if slots is None and (state.shape[0] < B or conv_state.shape[0] < B):
        raise ValueError("state/conv_state: fewer slots than sequences")
    st = _lib.load().gdn_decode_step(
        _ptr(x, "x", dt, (B, C)), _ptr(conv_w, "conv_w", dt, (C, 4)), _ptr(conv_state, "conv_state", dt),
        _ptr(z, "z", dt, (B, O)), _ptr(a, "a", dt, (B, dims.H_v)), _ptr(b, "b", dt, (B, dims.H_v)),
        _ptr(A_log, "A_log", torch.float32), _ptr(dt_bias, "dt_bias", torch.float32),
        _ptr(state, "state", torch.float32), _ptr(norm_w, "norm_w", dt), float(norm_eps),
        _ptr(slots, "slots", torch.int32, (B,)) if slots is not None else None, B, float(scale),
        _lib.GDN_QK_L2NORM if l2norm else 0, _ptr(out, "out", dt, (B, O)), _dims(dims),
        _dtype_code(x), _stream(x, stream))
    _lib.check(st, "gdn_decode_step")
    return out


def gdn_decode_verify(x, z, a, b, conv_w, A_log, dt_bias, norm_w, dims, state, conv_state,
                      slots, scale=0.0, l2norm=True, norm_eps=1e-6, out=None, stream=None):
    """Speculative-decoding verification: K draft tokens of B sequences
    (x [B, K, conv_dim], z [B, K, H_v*d_v], a, b [B, K, H_v]) through the fused
    decode step in one kernel.  States are read from slot slots[b, 0] of
    state [n_slots, H_v, d_k, d_v] f32 / conv_state [n_slots, conv_dim, 3]; the
    states after draft token t are written to slot slots[b, t + 1] (slots int32
    [B, K + 1]).  Returns out [B, K, H_v*d_v]."""
    dt = x.dtype
    if x.dim() != 3:
        raise ValueError("x: expected [B, K, conv_dim]")
    B, K = int(x.shape[0]), int(x.shape[1])
    C, O = _conv_dim(dims), int(dims.H_v) * int(dims.d_v)
    if out is None:
        out = torch.empty((B, K, O), dtype=dt, device=x.device)
    if state.dim() != 4 or tuple(state.shape[1:]) != (dims.H_v, dims.d_k, dims.d_v):
        raise ValueError("state: expected [n_slots, H_v, d_k, d_v]")
    if conv_state.dim() != 3 or tuple(conv_state.shape[1:]) != (C, 3):
        raise ValueError("conv_state: expected [n_slots, conv_dim, 3]")
    st = _lib.load().gdn_decode_verify(
        _ptr(x, "x", dt, (B, K, C)), _ptr(conv_w, "conv_w", dt, (C, 4)),
        _ptr(conv_state, "conv_state", dt), _ptr(z, "z", dt, (B, K, O)),
        _ptr(a, "a", dt, (B, K, dims.H_v)), _ptr(b, "b", dt, (B, K, dims.H_v)),
        _ptr(A_log, "A_log", torch.float32), _ptr(dt_bias, "dt_bias", torch.float32),
        _ptr(state, "state", torch.float32), _ptr(norm_w, "norm_w", dt), float(norm_eps),
        _ptr(slots, "slots", torch.int32, (B, K + 1)), B, K, float(scale),
        _lib.GDN_QK_L2NORM if l2norm else 0, _ptr(out, "out", dt, (B, K, O)), _dims(dims),
        _dtype_code(x), _stream(x, stream))
    _lib.check(st, "gdn_decode_verify")
    return out


def gdn_layer_decode(x, z, a, b, conv_w, A_log, dt_bias, norm_w, dims, state, conv_state,
                     scale=0.0, stream=None):
    """One decode step of the layer core for B sequences (x [B, conv_dim]);
    state and conv_state are updated in place.  Returns out [B, H_v*d_v]."""
    y = gdn_conv1d_update(x, conv_w, conv_state, dims, True, stream=stream)
    o = gdn_recurrent_decode(y, state, dims, a, b, A_log, dt_bias, scale=scale, stream=stream)
    return gdn_rmsnorm_gated(o, z, norm_w, dims, stream=stream)


@dataclass(frozen=True)
class HeadShard:
    """One rank's part of the layer core under head sharding: key heads
    [kh0, kh1), their value heads [h0, h1), and the matching conv channels
    (its q, k and v slices of conv_dim, in that order)."""
    dims: GDNDims
    kh0: int
    kh1: int
    h0: int
    h1: int
    channels: torch.Tensor  # int64 [conv_dim of the shard], indices into the full conv_dim


def head_shard(dims, rank: int, world: int) -> HeadShard:
    """Head sharding of the layer core over `world` ranks: rank takes a contiguous
    block of H_k / world key heads with their H_v / H_k value heads each.  Heads,
    their conv channels and their states are independent through the whole core,
    so every rank calls the same entry points with `shard.dims` on its slices
    (q, k, v channels, z and out columns, a, b, A_log and dt_bias entries, state
    heads) and no exchange is needed inside the core; the pages' tensor-parallel
    runs split the layer this way, with the one all-reduce after out_proj.
    world must divide H_k."""
    if world < 1 or rank < 0 or rank >= world or dims.H_k % world != 0:
        raise ValueError(f"head_shard: world {world} must divide H_k {dims.H_k} (rank {rank})")
    r = dims.H_v // dims.H_k
    nk = dims.H_k // world
    kh0, kh1 = rank * nk, (rank + 1) * nk
    h0, h1 = kh0 * r, kh1 * r
    dk, dv = dims.d_k, dims.d_v
    ch = torch.cat([torch.arange(kh0 * dk, kh1 * dk), torch.arange(dims.H_k * dk + kh0 * dk, dims.H_k * dk + kh1 * dk),
                    torch.arange(2 * dims.H_k * dk + h0 * dv, 2 * dims.H_k * dk + h1 * dv)])
    return HeadShard(GDNDims(nk, h1 - h0, dk, dv, dims.conv_k), kh0, kh1, h0, h1, ch)

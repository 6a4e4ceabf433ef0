"""C ABI: the library loads, exports every symbol include/gdn.h declares, and
rejects bad arguments on the host with the documented status codes (CPU only:
no call here reaches a launch)."""
import ctypes
import os
import re

import pytest
import torch

from conftest import ROOT

import gated_deltanet_linear_core_gb300 as gdn
from gated_deltanet_linear_core_gb300 import _lib

HEADER = os.path.join(ROOT, "include", "gdn.h")

# Argument-validation cases hand the library fake (never dereferenced) device
# addresses.  Each case must be rejected before any launch.  On a machine with
# a GPU these CPU tests are skipped so that a validation regression can never
# launch a kernel on fake addresses.
no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="host-only validation tests use fake device addresses")


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_linear_core_gb300 import build
    build.build()
    return _lib.load()


def header_symbols():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_\w+)\s*\(", txt)))


def test_header_declares_the_boundary():
    syms = header_symbols()
    for name in ["gdn_conv1d_fwd", "gdn_conv1d_update", "gdn_chunk_prefill",
                 "gdn_recurrent_decode", "gdn_rmsnorm_gated"]:
        assert name in syms


def test_library_exports_every_header_symbol(lib):
    syms = header_symbols()
    assert syms
    for name in syms:
        assert hasattr(lib, name), name
    assert set(syms) == set(_lib.SIGNATURES), "binding signatures out of sync with gdn.h"


def test_no_torch_types_in_header():
    txt = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for bad in ("torch", "at::", "Tensor", "c10", "#include <cuda"):
        assert bad not in txt


def test_status_strings_and_version(lib):
    for code in range(7):
        s = lib.gdn_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert lib.gdn_status_string(99) == b"unknown status"
    assert lib.gdn_version() >> 16 == 1
    assert lib.gdn_last_cuda_error() == 0


def test_ckpt_count(lib):
    assert gdn.gdn_ckpt_count([0, 130, 194, 257, 457], 64) == 2 + 1 + 0 + 3
    assert gdn.gdn_ckpt_count([0, 262144], 4096) == 64
    assert gdn.gdn_ckpt_count([0, 100], 0) == 0
    with pytest.raises(ValueError):
        gdn.gdn_ckpt_count([0, 100, 50], 64)
    cu = (ctypes.c_int32 * 2)(0, 10)
    assert lib.gdn_ckpt_count(None, 1, 64) == -1
    assert lib.gdn_ckpt_count(cu, 0, 64) == -1
    assert lib.gdn_ckpt_count(cu, 1, -1) == -1


DIMS = _lib.Dims(16, 48, 128, 128, 4)
A = 0x7f0000000000  # fake 16-byte-aligned address (never dereferenced)


def conv_fwd(lib, **kw):
    args = dict(x=A, w=A + 0x10000, cu=None, n_seq=1, T=64, si=None, so=None, every=0, ck=None,
                rows=0, silu=1, y=A + 0x20000, dims=DIMS, dt=_lib.GDN_BF16)
    args.update(kw)
    return lib.gdn_conv1d_fwd(args["x"], args["w"], args["cu"], args["n_seq"], args["T"],
                              args["si"], args["so"], args["every"], args["ck"], args["rows"],
                              args["silu"], args["y"], args["dims"], args["dt"], None)


@no_gpu
def test_conv1d_fwd_validation(lib):
    E = _lib
    assert conv_fwd(lib, dims=_lib.Dims(16, 48, 128, 128, 3)) == E.GDN_ERR_UNSUPPORTED
    assert conv_fwd(lib, dims=_lib.Dims(16, 48, 64, 64, 4)) == E.GDN_ERR_UNSUPPORTED
    assert conv_fwd(lib, dims=_lib.Dims(16, 40, 128, 128, 4)) == E.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, dims=_lib.Dims(0, 48, 128, 128, 4)) == E.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, dt=7) == E.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, x=None) == E.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, w=None) == E.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, y=A) == E.GDN_ERR_INVALID_ARG  # y aliases x
    assert conv_fwd(lib, x=A + 8) == E.GDN_ERR_ALIGN
    assert conv_fwd(lib, so=A + 0x30004) == E.GDN_ERR_ALIGN
    assert conv_fwd(lib, T=-1) == E.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, n_seq=2) == E.GDN_ERR_INVALID_ARG  # n_seq > 1 needs cu_seqlens
    assert conv_fwd(lib, cu=A + 0x40000, n_seq=0) == E.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, cu=A + 0x40002, n_seq=2) == E.GDN_ERR_ALIGN
    assert conv_fwd(lib, every=100, ck=A + 0x50000, rows=1) == E.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, every=64, ck=None, rows=1) == E.GDN_ERR_INVALID_ARG
    assert conv_fwd(lib, every=-64) == E.GDN_ERR_INVALID_ARG


def chunk(lib, **kw):
    args = dict(qkv=A, a=A + 0x1000, b=A + 0x2000, A_log=A + 0x3000, dt_bias=A + 0x4000,
                g=None, beta=None, cu=None, n_seq=1, T=64, S0=None, Sf=None, every=0,
                ck=None, rows=0, scale=0.0, flags=_lib.GDN_QK_L2NORM, o=A + 0x10000, ws=None,
                ws_bytes=0, dims=DIMS, dt=_lib.GDN_BF16)
    args.update(kw)
    return lib.gdn_chunk_prefill(
        args["qkv"], args["a"], args["b"], args["A_log"], args["dt_bias"], args["g"],
        args["beta"], args["cu"], args["n_seq"], args["T"], args["S0"], args["Sf"],
        args["every"], args["ck"], args["rows"], args["scale"], args["flags"], args["o"],
        args["ws"], args["ws_bytes"], args["dims"], args["dt"], None)


@no_gpu
def test_chunk_prefill_validation(lib):
    E = _lib
    assert chunk(lib, a=None) == E.GDN_ERR_INVALID_ARG      # neither raw gates ...
    assert chunk(lib, a=None, g=A + 0x5000) == E.GDN_ERR_INVALID_ARG  # ... nor g AND beta
    assert chunk(lib, A_log=A + 0x3002) == E.GDN_ERR_ALIGN
    assert chunk(lib, a=A + 0x1001) == E.GDN_ERR_ALIGN       # bf16 needs 2-byte alignment
    assert chunk(lib, flags=4) == E.GDN_ERR_INVALID_ARG
    # the Neumann-style solve: tensor-core path only (bf16, d = 128); here the
    # flags pass and the missing workspace is what is reported
    neu = E.GDN_QK_L2NORM | E.GDN_SOLVE_NEUMANN
    assert chunk(lib, flags=neu) == E.GDN_ERR_WORKSPACE
    assert chunk(lib, flags=neu, dt=E.GDN_F32, a=A + 0x1000, b=A + 0x2000) == E.GDN_ERR_UNSUPPORTED
    # the chunk-size field (bits 8..15): 16, 32, 64 or 0; on the tensor-core path
    # 16 and 32 need final_state (the state crosses the extra segments in it)
    assert chunk(lib, flags=1 | E.GDN_CHUNK(48)) == E.GDN_ERR_INVALID_ARG
    assert chunk(lib, flags=1 | E.GDN_CHUNK(128)) == E.GDN_ERR_INVALID_ARG
    assert chunk(lib, flags=1 | E.GDN_CHUNK(8)) == E.GDN_ERR_INVALID_ARG
    assert chunk(lib, flags=1 | (1 << 16)) == E.GDN_ERR_INVALID_ARG
    assert chunk(lib, flags=1 | E.GDN_CHUNK(16)) == E.GDN_ERR_UNSUPPORTED
    assert chunk(lib, flags=1 | E.GDN_CHUNK(32)) == E.GDN_ERR_UNSUPPORTED
    assert chunk(lib, flags=1 | E.GDN_CHUNK(32), Sf=A + 0x20000) == E.GDN_ERR_WORKSPACE  # valid
    assert chunk(lib, flags=1 | E.GDN_CHUNK(64)) == E.GDN_ERR_WORKSPACE  # valid; no workspace given
    assert chunk(lib, scale=float("nan")) == E.GDN_ERR_INVALID_ARG
    assert chunk(lib, scale=float("inf")) == E.GDN_ERR_INVALID_ARG
    assert chunk(lib, o=None) == E.GDN_ERR_INVALID_ARG
    assert chunk(lib, qkv=A + 4) == E.GDN_ERR_ALIGN
    assert chunk(lib, S0=A + 0x6008) == E.GDN_ERR_ALIGN
    assert chunk(lib, Sf=A + 0x6004) == E.GDN_ERR_ALIGN
    assert chunk(lib, every=4000, ck=A + 0x7000, rows=1) == E.GDN_ERR_INVALID_ARG
    assert chunk(lib, every=4096, ck=None, rows=1) == E.GDN_ERR_INVALID_ARG
    assert chunk(lib, every=4096, ck=None, rows=-1) == E.GDN_ERR_INVALID_ARG
    # no rows allocated (every sequence shorter than the cadence): no buffer needed
    assert chunk(lib, every=4096, ck=None, rows=0) == E.GDN_ERR_WORKSPACE
    assert chunk(lib, dims=_lib.Dims(16, 48, 128, 64, 4)) == E.GDN_ERR_UNSUPPORTED
    assert chunk(lib, dims=_lib.Dims(16, 48, 32, 32, 4)) == E.GDN_ERR_UNSUPPORTED


@no_gpu
def test_decode_update_norm_validation(lib):
    E = _lib
    dec = lambda **kw: lib.gdn_recurrent_decode(
        kw.get("qkv", A), kw.get("a", A + 0x1000), kw.get("b", A + 0x2000),
        kw.get("A_log", A + 0x3000), kw.get("dt_bias", A + 0x4000), None, None,
        kw.get("state", A + 0x10000), kw.get("B", 4), kw.get("scale", 0.0),
        kw.get("flags", 1), kw.get("o", A + 0x20000), kw.get("dims", DIMS), _lib.GDN_BF16, None)
    assert dec(B=-1) == E.GDN_ERR_INVALID_ARG
    assert dec(state=None) == E.GDN_ERR_INVALID_ARG
    assert dec(state=A + 0x10008) == E.GDN_ERR_ALIGN
    assert dec(flags=4) == E.GDN_ERR_INVALID_ARG
    assert dec(a=None) == E.GDN_ERR_INVALID_ARG
    upd = lambda **kw: lib.gdn_conv1d_update(
        kw.get("x", A), kw.get("w", A + 0x1000), kw.get("st", A + 0x2000), kw.get("B", 4), 1,
        kw.get("y", A + 0x3000), kw.get("dims", DIMS), _lib.GDN_BF16, None)
    assert upd(B=-2) == E.GDN_ERR_INVALID_ARG
    assert upd(st=None) == E.GDN_ERR_INVALID_ARG
    assert upd(y=A + 2) == E.GDN_ERR_ALIGN
    assert upd(dims=_lib.Dims(16, 48, 128, 128, 2)) == E.GDN_ERR_UNSUPPORTED
    norm = lambda **kw: lib.gdn_rmsnorm_gated(
        kw.get("o", A), kw.get("z", A + 0x1000), kw.get("w", A + 0x2000), kw.get("eps", 1e-6),
        kw.get("T", 8), kw.get("out", A + 0x3000), DIMS, _lib.GDN_BF16, None)
    assert norm(eps=0.0) == E.GDN_ERR_INVALID_ARG
    assert norm(eps=-1.0) == E.GDN_ERR_INVALID_ARG
    assert norm(w=None) == E.GDN_ERR_INVALID_ARG
    assert norm(T=-3) == E.GDN_ERR_INVALID_ARG
    assert norm(z=A + 0x1008) == E.GDN_ERR_ALIGN


def _fused_decode(lib, verify, **kw):
    """gdn_decode_step / gdn_decode_verify with fake device addresses."""
    g = kw.get
    head = [g("x", A), g("w", A + 0x1000), g("cs", A + 0x2000), g("z", A + 0x3000), g("a", A + 0x4000),
            g("b", A + 0x5000), g("A_log", A + 0x6000), g("dt_bias", A + 0x7000), g("state", A + 0x10000),
            g("nw", A + 0x8000), g("eps", 1e-6), g("slots", A + 0x9000), g("B", 4)]
    tail = [g("scale", 0.0), g("flags", 1), g("out", A + 0x20000), g("dims", DIMS), _lib.GDN_BF16, None]
    if verify:
        return lib.gdn_decode_verify(*head, g("K", 4), *tail)
    return lib.gdn_decode_step(*head, *tail)


@no_gpu
@pytest.mark.parametrize("verify", [False, True], ids=["decode_step", "decode_verify"])
def test_fused_decode_validation(lib, verify):
    E = _lib
    call = lambda **kw: _fused_decode(lib, verify, **kw)
    assert call(B=-1) == E.GDN_ERR_INVALID_ARG
    assert call(dims=_lib.Dims(16, 40, 128, 128, 4)) == E.GDN_ERR_INVALID_ARG  # H_v % H_k != 0
    assert call(dims=_lib.Dims(2, 32, 128, 128, 4)) == E.GDN_ERR_UNSUPPORTED   # 16 value heads per key head
    assert call(dims=_lib.Dims(16, 48, 64, 64, 4)) == E.GDN_ERR_UNSUPPORTED
    assert call(flags=2) == E.GDN_ERR_INVALID_ARG                               # only GDN_QK_L2NORM
    assert call(eps=0.0) == E.GDN_ERR_INVALID_ARG
    assert call(eps=float("nan")) == E.GDN_ERR_INVALID_ARG
    assert call(scale=float("inf")) == E.GDN_ERR_INVALID_ARG
    for name in ("x", "w", "cs", "z", "a", "b", "A_log", "dt_bias", "state", "nw", "out"):
        assert call(**{name: None}) == E.GDN_ERR_INVALID_ARG, name
    assert call(z=A + 0x3008) == E.GDN_ERR_ALIGN
    assert call(state=A + 0x10008) == E.GDN_ERR_ALIGN
    assert call(a=A + 0x4001) == E.GDN_ERR_ALIGN                                # bf16 gate input
    assert call(slots=A + 0x9002) == E.GDN_ERR_ALIGN
    assert call(out=A + 0x20004) == E.GDN_ERR_ALIGN
    # no work: nothing is read, so no buffer is needed, and nothing is launched
    nulls = dict.fromkeys(("x", "w", "cs", "z", "a", "b", "A_log", "dt_bias", "state", "nw", "slots", "out"))
    assert call(B=0, **nulls) == E.GDN_OK
    if verify:
        assert call(K=-1) == E.GDN_ERR_INVALID_ARG
        assert call(K=17) == E.GDN_ERR_INVALID_ARG                              # at most 16 draft tokens
        assert call(slots=None) == E.GDN_ERR_INVALID_ARG                        # slots are required
        assert call(K=0, **nulls) == E.GDN_OK


def layer(lib, **kw):
    """gdn_layer_prefill with fake device addresses (never dereferenced)."""
    args = dict(x=A, z=A + 0x1000, a=A + 0x2000, b=A + 0x3000, w=A + 0x4000, A_log=A + 0x5000,
                dt_bias=A + 0x6000, nw=A + 0x7000, eps=1e-6, cu=None, n_seq=1, T=64, S0=None,
                Sf=A + 0x10000, cs_in=None, cs_out=A + 0x20000, every=0, sck=None, cck=None, rows=0,
                scale=0.0, flags=1, out=A + 0x30000, ws=None, ws_bytes=0, dims=DIMS, dt=_lib.GDN_BF16)
    args.update(kw)
    return lib.gdn_layer_prefill(
        args["x"], args["z"], args["a"], args["b"], args["w"], args["A_log"], args["dt_bias"], args["nw"],
        args["eps"], args["cu"], args["n_seq"], args["T"], args["S0"], args["Sf"], args["cs_in"],
        args["cs_out"], args["every"], args["sck"], args["cck"], args["rows"], args["scale"], args["flags"],
        args["out"], args["ws"], args["ws_bytes"], args["dims"], args["dt"], None)


@no_gpu
def test_layer_prefill_validation(lib):
    E = _lib
    # everything valid but the workspace: that is what is reported
    assert layer(lib) == E.GDN_ERR_WORKSPACE
    need = lib.gdn_layer_prefill_workspace_size(1, 64, DIMS, _lib.GDN_BF16)
    assert layer(lib, ws_bytes=need) == E.GDN_ERR_WORKSPACE        # NULL workspace
    assert layer(lib, ws=A + 0x100000, ws_bytes=need - 1) == E.GDN_ERR_WORKSPACE
    assert layer(lib, eps=0.0) == E.GDN_ERR_INVALID_ARG
    assert layer(lib, eps=float("nan")) == E.GDN_ERR_INVALID_ARG
    assert layer(lib, z=None) == E.GDN_ERR_INVALID_ARG
    assert layer(lib, out=None) == E.GDN_ERR_INVALID_ARG
    assert layer(lib, nw=None) == E.GDN_ERR_INVALID_ARG
    assert layer(lib, z=A + 0x1008) == E.GDN_ERR_ALIGN
    assert layer(lib, out=A + 0x30002) == E.GDN_ERR_ALIGN
    assert layer(lib, ws=A + 0x100008, ws_bytes=need) == E.GDN_ERR_ALIGN
    assert layer(lib, every=64, sck=A + 0x40000, cck=None, rows=1) == E.GDN_ERR_INVALID_ARG
    assert layer(lib, every=64, sck=None, cck=A + 0x50000, rows=1) == E.GDN_ERR_INVALID_ARG
    assert layer(lib, every=100, sck=A + 0x40000, cck=A + 0x50000, rows=1) == E.GDN_ERR_INVALID_ARG
    assert layer(lib, n_seq=2) == E.GDN_ERR_INVALID_ARG             # two sequences need cu_seqlens
    assert layer(lib, T=-1) == E.GDN_ERR_INVALID_ARG
    assert layer(lib, dims=_lib.Dims(16, 48, 128, 128, 3)) == E.GDN_ERR_UNSUPPORTED


def host_layer(lib, **kw):
    """gdn_layer_prefill_host with fake addresses (never dereferenced): every
    case below is rejected before the page-lock check, which asks the driver."""
    g = kw.get
    return lib.gdn_layer_prefill_host(
        g("hq", A), g("hz", A + 0x1000), g("ha", A + 0x2000), g("hb", A + 0x3000), g("w", A + 0x4000),
        g("A_log", A + 0x5000), g("dt_bias", A + 0x6000), g("nw", A + 0x7000), g("T", 64), None,
        g("Sf", A + 0x10000), None, g("cs_out", A + 0x20000), g("scale", 0.0), g("flags", 1), g("eps", 1e-6),
        g("hout", A + 0x30000), g("ws", A + 0x100000), g("ws_bytes", 1 << 30), g("dims", DIMS), _lib.GDN_BF16,
        None)


@no_gpu
def test_layer_prefill_host_validation(lib):
    E = _lib
    assert host_layer(lib, T=-1) == E.GDN_ERR_INVALID_ARG
    assert host_layer(lib, flags=2) == E.GDN_ERR_INVALID_ARG        # no Neumann option on this path
    assert host_layer(lib, eps=0.0) == E.GDN_ERR_INVALID_ARG         # as every RMSNormGated entry point
    assert host_layer(lib, eps=-1.0) == E.GDN_ERR_INVALID_ARG
    assert host_layer(lib, eps=float("nan")) == E.GDN_ERR_INVALID_ARG
    assert host_layer(lib, scale=float("inf")) == E.GDN_ERR_INVALID_ARG
    for name in ("w", "A_log", "dt_bias", "nw", "Sf", "cs_out", "hq", "hz", "ha", "hb", "hout"):
        assert host_layer(lib, **{name: None}) == E.GDN_ERR_INVALID_ARG, name
    assert host_layer(lib, w=A + 0x4008) == E.GDN_ERR_ALIGN
    assert host_layer(lib, Sf=A + 0x10004) == E.GDN_ERR_ALIGN
    assert host_layer(lib, ws=A + 0x100008) == E.GDN_ERR_ALIGN
    assert host_layer(lib, dims=_lib.Dims(16, 48, 64, 64, 4)) == E.GDN_ERR_UNSUPPORTED
    assert host_layer(lib, dims=_lib.Dims(16, 40, 128, 128, 4)) == E.GDN_ERR_INVALID_ARG


def test_layer_prefill_workspace_and_launches(lib):
    dims = gdn.GDNDims(16, 48, 128, 128)
    C = dims.conv_dim
    # bf16 with d = 128: the conv runs inside the chunk kernels, so no conv
    # output; the chunk intermediates plus the conv'd q tile of every chunk and
    # key head (4096 tokens: one segment of 65 chunk slots, 16 KiB per tile)
    ws_c = gdn.gdn_chunk_prefill_workspace_size(1, 4096, dims, torch.bfloat16)
    assert gdn.gdn_layer_prefill_workspace_size(1, 4096, dims, torch.bfloat16) == ws_c + 65 * 16 * 16384
    # f32: the conv output (rounded up to 256 bytes); the CUDA-core rule needs none
    assert gdn.gdn_layer_prefill_workspace_size(1, 100, dims, torch.float32) == (100 * C * 4 + 255) // 256 * 256
    assert gdn.gdn_layer_prefill_workspace_size(1, 0, dims, torch.bfloat16) == 0
    # the chunk kernels (the conv inside them) and the norm; f32: conv, rule, norm
    for cu in (True, None):
        assert gdn.gdn_layer_prefill_launches(1, 4096, dims, torch.bfloat16, cu_seqlens=cu) == \
            1 + gdn.gdn_chunk_prefill_launches(1, 4096, dims, torch.bfloat16, cu_seqlens=cu)
    assert gdn.gdn_layer_prefill_launches(1, 64, gdn.GDNDims(2, 4, 16, 16), torch.float32) == 3
    assert gdn.gdn_layer_prefill_launches(1, 0, dims, torch.bfloat16) == 0


def test_workspace_size(lib):
    dims = gdn.GDNDims(16, 32, 128, 128)
    # the CUDA-core (f32) path needs none; the bf16 tensor-core path holds per-chunk
    # intermediates (58,368 B per chunk and value head) plus chunk offsets
    assert gdn.gdn_chunk_prefill_workspace_size(8, 32768, dims, torch.float32) == 0
    ws = gdn.gdn_chunk_prefill_workspace_size(8, 32768, dims, torch.bfloat16)
    assert ws >= 32 * 58368
    assert gdn.gdn_chunk_prefill_workspace_size(8, 0, dims, torch.bfloat16) == 0
    assert gdn.gdn_chunk_prefill_workspace_size(1, 64, gdn.GDNDims(2, 4, 16, 16),
                                                torch.bfloat16) == 0


def test_prefill_launch_count(lib):
    # chunk offsets (with cu_seqlens), then an intra and a chain kernel per
    # workspace segment; the CUDA-core path is one kernel; nothing for an empty call
    dims = gdn.GDNDims(16, 48, 128, 128)
    assert gdn.gdn_chunk_prefill_launches(1, 4096, dims, torch.bfloat16) == 3
    assert gdn.gdn_chunk_prefill_launches(1, 4096, dims, torch.bfloat16, cu_seqlens=None) == 2
    long_run = gdn.gdn_chunk_prefill_launches(1, 262144, dims, torch.bfloat16)
    assert long_run > 3 and long_run % 2 == 1
    assert gdn.gdn_chunk_prefill_launches(1, 262144, dims, torch.bfloat16, cu_seqlens=None) == long_run - 1
    assert gdn.gdn_chunk_prefill_launches(1, 64, gdn.GDNDims(2, 4, 16, 16), torch.float32) == 1
    assert gdn.gdn_chunk_prefill_launches(1, 0, dims, torch.bfloat16) == 0
    # shorter chunks on the tensor-core path: the 65-chunk segments of the
    # 4096-token call hold 129 chunks of 32 tokens in 2 segments, 257 of 16 in 4
    assert gdn.gdn_chunk_prefill_launches(1, 4096, dims, torch.bfloat16, cu_seqlens=None, chunk=32) == 4
    assert gdn.gdn_chunk_prefill_launches(1, 4096, dims, torch.bfloat16, cu_seqlens=None, chunk=16) == 8
    assert gdn.gdn_layer_prefill_launches(1, 4096, dims, torch.bfloat16, cu_seqlens=None, chunk=32) == 5
    assert gdn.gdn_chunk_prefill_launches(1, 64, gdn.GDNDims(2, 4, 16, 16), torch.float32, chunk=16) == 1


def test_host_prefill_piece_plan(lib):
    # pieces of at most `piece` tokens, multiples of 64; a whole number (>= 2) of
    # full pieces has its last piece cut into 3/4 and 1/4; a short sequence is
    # one piece
    d = gdn._dims(gdn.GDNDims(16, 48, 128, 128))
    bf = gdn._lib.GDN_BF16
    piece = lib.gdn_layer_prefill_host_piece
    pieces = lib.gdn_layer_prefill_host_pieces
    assert piece(4096, d, bf) == 512 and pieces(4096, d, bf) == 7 + 2
    assert piece(3000, d, bf) == 512 and pieces(3000, d, bf) == 6
    assert piece(1024, d, bf) == 1024 and pieces(1024, d, bf) == 1
    assert piece(64, d, bf) == 64 and pieces(64, d, bf) == 1
    assert piece(65536, d, bf) == 4096 and pieces(65536, d, bf) == 15 + 2
    assert pieces(0, d, bf) == 0


def test_binding_rejects_host_tensors_before_the_library():
    x = torch.zeros(4, 128)
    with pytest.raises(ValueError, match="CUDA"):
        gdn.gdn_conv1d_fwd(x, torch.zeros(128, 4), gdn.GDNDims(2, 4, 16, 16), y=torch.zeros(4, 128))

"""ctypes loader of libgdn.so: symbol signatures and status codes of include/gdn.h."""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_ALIGN = 2
GDN_ERR_UNSUPPORTED = 3
GDN_ERR_WORKSPACE = 4
GDN_ERR_CUDA = 5
GDN_ERR_TIMEOUT = 6
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_ALIGN",
                3: "GDN_ERR_UNSUPPORTED", 4: "GDN_ERR_WORKSPACE", 5: "GDN_ERR_CUDA",
                6: "GDN_ERR_TIMEOUT"}

GDN_F32 = 0
GDN_BF16 = 1
GDN_QK_L2NORM = 1
GDN_SOLVE_NEUMANN = 2


def GDN_CHUNK(c: int) -> int:
    """The chunk-size field of the prefill flags (bits 8..15)."""
    return (int(c) & 0xFF) << 8


class Dims(ctypes.Structure):
    _fields_ = [("H_k", ctypes.c_int32), ("H_v", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("conv_k", ctypes.c_int32)]


P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
U32 = ctypes.c_uint32
F32 = ctypes.c_float
SZ = ctypes.c_size_t
ST = ctypes.c_int  # gdn_status_t

# name -> (restype, argtypes), in the order of include/gdn.h
SIGNATURES = {
    "gdn_status_string": (ctypes.c_char_p, [ST]),
    "gdn_last_cuda_error": (ctypes.c_int, []),
    "gdn_version": (ctypes.c_int, []),
    "gdn_ckpt_count": (I64, [P, I32, I32]),
    "gdn_check_cu_seqlens": (ST, [P, I32, I64, P]),
    "gdn_sync_status": (ST, [P]),
    "gdn_selftest_bounded_wait": (ST, [I64, P]),
    "gdn_layer_prefill_host_workspace_size": (SZ, [I64, Dims, ST]),
    "gdn_layer_prefill_host_piece": (I64, [I64, Dims, ST]),
    "gdn_layer_prefill_host_pieces": (I64, [I64, Dims, ST]),
    "gdn_layer_prefill_host": (ST, [P, P, P, P, P, P, P, P, I64, P, P, P, P, F32, U32, F32, P, P, SZ,
                                    Dims, ST, P]),
    "gdn_conv1d_fwd": (ST, [P, P, P, I32, I64, P, P, I32, P, I64, I32, P, Dims, ST, P]),
    "gdn_conv1d_update": (ST, [P, P, P, I32, I32, P, Dims, ST, P]),
    "gdn_chunk_prefill_workspace_size": (SZ, [I32, I64, Dims, ST]),
    "gdn_chunk_prefill_launches": (I32, [I32, I64, I32, Dims, ST, U32]),
    "gdn_chunk_prefill": (ST, [P, P, P, P, P, P, P, P, I32, I64, P, P, I32, P, I64, F32, U32, P,
                               P, SZ, Dims, ST, P]),
    "gdn_chunk_prefill_noalloc": (ST, [P, P, P, P, P, P, P, P, I32, I64, P, P, I32, P, I64, F32, U32,
                                       P, Dims, ST, P]),
    "gdn_recurrent_decode": (ST, [P, P, P, P, P, P, P, P, I32, F32, U32, P, Dims, ST, P]),
    "gdn_chunk_prefill_norm": (ST, [P, P, P, P, P, P, P, P, I32, I64, P, P, I32, P, I64, F32, U32, P, P, F32,
                                    P, P, SZ, Dims, ST, P]),
    "gdn_layer_prefill_workspace_size": (SZ, [I32, I64, Dims, ST]),
    "gdn_layer_prefill_launches": (I32, [I32, I64, I32, Dims, ST, U32]),
    "gdn_layer_prefill": (ST, [P, P, P, P, P, P, P, P, F32, P, I32, I64, P, P, P, P, I32, P, P, I64, F32, U32,
                               P, P, SZ, Dims, ST, P]),
    "gdn_rmsnorm_gated": (ST, [P, P, P, F32, I64, P, Dims, ST, P]),
    "gdn_decode_step": (ST, [P, P, P, P, P, P, P, P, P, P, F32, P, I32, F32, U32, P, Dims, ST, P]),
    "gdn_decode_verify": (ST, [P, P, P, P, P, P, P, P, P, P, F32, P, I32, I32, F32, U32, P, Dims, ST,
                               P]),
}

_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libgdn.so (built in-tree by gated_deltanet_linear_core_gb300.build).
    Raises if it is missing: there is no fallback implementation."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; "
                    f"g.build()'` (or python -m gated_deltanet_linear_core_gb300.build)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class GDNError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = lib.gdn_status_string(status).decode()
        extra = ""
        if status == GDN_ERR_CUDA:
            extra = f" (cudaError {lib.gdn_last_cuda_error()})"
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}{extra}")
        self.status = status


def check(status: int, where: str):
    if status != GDN_OK:
        raise GDNError(status, where)

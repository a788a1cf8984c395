"""ctypes mirror of include/ovc.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

c_i64 = ctypes.c_int64
c_i32 = ctypes.c_int32
c_ptr = ctypes.c_void_p

OVC_OK = 0
OVC_ERR_INVALID_ARG = 1
OVC_ERR_UNSUPPORTED = 2
OVC_ERR_WORKSPACE_TOO_SMALL = 3
OVC_ERR_CUDA = 4
OVC_ERR_TIMEOUT = 5
OVC_ERR_SCRATCH_LIMIT = 6
OVC_NOALLOC_MAX_HEADS = 4096
OVC_PREPARE_SMOOTH_K = 1
OVC_PREPARE_V_SMOOTH = 2
OVC_PREPARE_SMOOTH_Q = 4
OVC_ATTN_EXP_THEN_CAST = 1
OVC_ATTN_NATURAL_ORDER = 2
OVC_ATTN_BASELINE = 3
OVC_BF16 = 0
OVC_FP16 = 1


class OvcTensor(ctypes.Structure):
    _fields_ = [("ptr", c_ptr), ("dtype", c_i32), ("B", c_i64), ("S", c_i64), ("H", c_i64),
                ("D", c_i64), ("stride_b", c_i64), ("stride_s", c_i64), ("stride_h", c_i64)]


class OvcOutput(ctypes.Structure):
    _fields_ = [("ptr", c_ptr), ("stride_b", c_i64), ("stride_s", c_i64), ("stride_h", c_i64)]


class OvcPrepared(ctypes.Structure):
    _fields_ = [("B", c_i64), ("S", c_i64), ("H", c_i64), ("nb", c_i64), ("S_pad", c_i64),
                ("q", c_ptr), ("k", c_ptr), ("vt", c_ptr), ("sq", c_ptr), ("sk", c_ptr),
                ("sv", c_ptr), ("vamax", c_ptr), ("energy", c_ptr), ("vmean", c_ptr), ("perm", c_ptr),
                ("kbias", c_ptr)]


class OvcRepair(ctypes.Structure):
    _fields_ = [("B", c_i64), ("S", c_i64), ("H", c_i64), ("n", c_i64), ("n_pad", c_i64),
                ("idx", c_ptr), ("k_sel", c_ptr), ("dvt", c_ptr), ("sk_sel", c_ptr), ("sr", c_ptr),
                ("kb_sel", c_ptr)]


class OvcHostIO(ctypes.Structure):
    _fields_ = [("q", c_ptr), ("k", c_ptr), ("v", c_ptr), ("o", c_ptr), ("dtype", c_i32),
                ("B", c_i64), ("S", c_i64), ("H", c_i64)]


class OvcProbe(ctypes.Structure):
    _fields_ = [("dump_bh", c_i64), ("dump_qblock", c_i64), ("dump_kblock", c_i64),
                ("dump_codes", c_ptr), ("dump_m8", c_ptr), ("wait_timeout_ns", ctypes.c_uint64),
                ("skip_mma", c_i32), ("force_persistent", c_i32), ("trace", c_ptr),
                ("flags", ctypes.c_uint32)]


P = ctypes.POINTER
SIGNATURES = {
    "ovc_prepare_workspace_bytes": (ctypes.c_size_t, [c_i64, c_i64, c_i64, c_i64]),
    "ovc_prepare": (c_i32, [P(OvcTensor), P(OvcTensor), P(OvcTensor), c_ptr, ctypes.c_size_t,
                            P(OvcPrepared), c_ptr]),
    "ovc_attention": (c_i32, [P(OvcPrepared), ctypes.c_float, P(OvcOutput), c_ptr]),
    "ovc_attention_ex": (c_i32, [P(OvcPrepared), P(OvcRepair), ctypes.c_float, P(OvcOutput),
                                 ctypes.c_uint32, c_i32, c_ptr, ctypes.c_size_t, c_ptr]),
    "ovc_attention_workspace_bytes": (ctypes.c_size_t, [P(OvcPrepared), c_i32]),
    "ovc_repair_workspace_bytes": (ctypes.c_size_t, [c_i64, c_i64, c_i64, ctypes.c_float]),
    "ovc_prepare_v_repair": (c_i32, [P(OvcTensor), P(OvcPrepared), ctypes.c_float, c_ptr,
                                     ctypes.c_size_t, P(OvcRepair), c_ptr]),
    "ovc_attention_v_repair": (c_i32, [P(OvcPrepared), P(OvcRepair), ctypes.c_float,
                                       P(OvcOutput), c_ptr]),
    "ovc_get_device_status": (c_i32, [c_ptr]),
    "ovc_status_string": (ctypes.c_char_p, [c_i32]),
    "ovc_attention_probe": (c_i32, [P(OvcPrepared), P(OvcRepair), ctypes.c_float, P(OvcOutput),
                                    P(OvcProbe), c_ptr]),
    "ovc_prepare_noalloc": (c_i32, [P(OvcTensor), P(OvcTensor), P(OvcTensor), P(OvcPrepared), c_ptr]),
    "ovc_prepare_workspace_bytes_ex": (ctypes.c_size_t, [c_i64, c_i64, c_i64, c_i64, ctypes.c_uint32]),
    "ovc_prepare_ex": (c_i32, [P(OvcTensor), P(OvcTensor), P(OvcTensor), ctypes.c_uint32, c_ptr,
                               ctypes.c_size_t, P(OvcPrepared), c_ptr]),
    "ovc_vsmooth_group_workspace_bytes": (ctypes.c_size_t, [c_i64, c_i64, c_i64, c_i32]),
    "ovc_vsmooth_group": (c_i32, [P(OvcTensor), c_i32, c_i32, c_ptr, ctypes.c_size_t, c_ptr, c_ptr]),
    "ovc_prepare_grouped": (c_i32, [P(OvcTensor), P(OvcTensor), P(OvcTensor), c_ptr, ctypes.c_uint32, c_ptr,
                                    ctypes.c_size_t, P(OvcPrepared), c_ptr]),
    "ovc_attention_host": (c_i32, [P(OvcHostIO), ctypes.c_float, ctypes.c_uint32, ctypes.c_float, c_ptr, c_i32,
                                   c_ptr, ctypes.c_size_t]),
    "ovc_attention_host_workspace_bytes": (ctypes.c_size_t, [c_i64, c_i64, c_i64, c_i32, ctypes.c_uint32,
                                                             ctypes.c_float]),
    "ovc_host_chunk_plan": (c_i32, [c_i64, c_i64, c_i32, c_ptr, c_i32]),
}

_lock = threading.Lock()
_lib = None


class OvcError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _lib.ovc_status_string(status).decode() if _lib is not None else f"status {status}"
        super().__init__(f"{what}: {msg} (status {status})" if what else msg)


def lib():
    """Load the in-tree libovc.so; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(
                    f"libovc is not built ({_build.LIB} missing); run "
                    "`python -m fp8_bit_attention_gb300.build` on a machine with nvcc")
            L = ctypes.CDLL(_build.LIB)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def check(status: int, what: str = "") -> None:
    if status != OVC_OK:
        raise OvcError(status, what)

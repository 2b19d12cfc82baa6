"""ctypes view of libkda.so (the C ABI declared in include/kda.h)."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_WORKSPACE = 3
KDA_ERR_CUDA = 4
KDA_ERR_DEVICE = 5

KDA_DTYPE_F32 = 0
KDA_DTYPE_BF16 = 1
KDA_DECAY_SCALAR = 0
KDA_DECAY_PER_CHANNEL = 1
KDA_FLAG_CHECKED = 1
KDA_FLAG_CUDA_CORES = 2
KDA_FLAG_COMPACT = 4
KDA_FLAG_NO_DELTA = 8

KDA_DEVERR_NONE = 0
KDA_DEVERR_OFFSETS = 1
KDA_DEVERR_SLOT_RANGE = 2
KDA_DEVERR_SLOT_DUP = 3
KDA_DEVERR_TIMEOUT = 4
KDA_DEVERR_DECAY_RANGE = 5
KDA_DEVERR_ACCEPTED = 6

# every function include/kda.h declares
EXPORTS = ("kda_abi_version", "kda_status_string", "kda_prefill_workspace_size",
           "kda_prefill_fwd", "kda_decode_step", "kda_get_device_error",
           "kda_set_stage_events", "kda_prefill_fwd_no_alloc",
           "kda_prefill_uses_tensor_cores", "kda_ring_record_elems", "kda_verify_window",
           "kda_fold_accepted", "kda_gdp_prefill_fwd", "kda_gdp_decode_step",
           "kda_gdp_workspace_size", "kda_prefill_bwd", "kda_prefill_bwd_workspace_size",
           "kda_conv_gates_fwd", "kda_prefill_no_alloc_form")

KDA_NO_ALLOC_SCRATCH_BYTES = 64 << 20


class KdaParams(ctypes.Structure):
    """Mirror of kda_params_t (natural alignment, same field order)."""

    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("num_k_heads", ctypes.c_int32),
        ("num_v_heads", ctypes.c_int32),
        ("d_k", ctypes.c_int32),
        ("d_v", ctypes.c_int32),
        ("num_slots", ctypes.c_int32),
        ("total_tokens", ctypes.c_int64),
        ("chunk", ctypes.c_int32),
        ("qkv_dtype", ctypes.c_int32),
        ("state_dtype", ctypes.c_int32),
        ("decay_kind", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("l2norm_qk", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("q_row_stride", ctypes.c_int64),
        ("k_row_stride", ctypes.c_int64),
        ("v_row_stride", ctypes.c_int64),
    ]


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})" if what
                         else f"{status_string(status)} (status {status})")


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libkda.so.  Raises if it has not been built: there is no fallback path."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libkda.so is not built ({path}); run "
                "`python -m gated_delta_rule_deltanet_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        pp = ctypes.POINTER(KdaParams)
        L.kda_abi_version.argtypes = []
        L.kda_abi_version.restype = ctypes.c_int
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_prefill_workspace_size.argtypes = [pp, ctypes.POINTER(ctypes.c_size_t)]
        L.kda_prefill_workspace_size.restype = ctypes.c_int
        L.kda_prefill_fwd.argtypes = [pp, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        L.kda_prefill_fwd.restype = ctypes.c_int
        L.kda_decode_step.argtypes = [pp, P, P, P, P, P, P, P, P, P]
        L.kda_decode_step.restype = ctypes.c_int
        L.kda_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
        L.kda_get_device_error.restype = ctypes.c_int
        L.kda_ring_record_elems.argtypes = [pp]
        L.kda_ring_record_elems.restype = ctypes.c_int
        L.kda_verify_window.argtypes = [pp, P, P, P, P, P, P, ctypes.c_int32, P, P, P, P]
        L.kda_verify_window.restype = ctypes.c_int
        L.kda_fold_accepted.argtypes = [pp, P, ctypes.c_int32, P, P, P, P]
        L.kda_fold_accepted.restype = ctypes.c_int
        L.kda_prefill_uses_tensor_cores.argtypes = [pp]
        L.kda_prefill_uses_tensor_cores.restype = ctypes.c_int
        L.kda_prefill_fwd_no_alloc.argtypes = [pp, P, P, P, P, P, P, P, P, P, P]
        L.kda_prefill_fwd_no_alloc.restype = ctypes.c_int
        L.kda_prefill_no_alloc_form.argtypes = [pp]
        L.kda_prefill_no_alloc_form.restype = ctypes.c_int
        L.kda_gdp_prefill_fwd.argtypes = [pp, ctypes.c_int32, P, P, P, P, P, P, P, P, P, P,
                                          ctypes.c_size_t, P]
        L.kda_gdp_prefill_fwd.restype = ctypes.c_int
        L.kda_gdp_decode_step.argtypes = [pp, ctypes.c_int32, P, P, P, P, P, P, P, P, P,
                                          ctypes.c_size_t, P]
        L.kda_gdp_decode_step.restype = ctypes.c_int
        L.kda_gdp_workspace_size.argtypes = [pp, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.POINTER(ctypes.c_size_t)]
        L.kda_gdp_workspace_size.restype = ctypes.c_int
        L.kda_prefill_bwd.argtypes = [pp] + [P] * 17 + [ctypes.c_size_t, P]
        L.kda_prefill_bwd.restype = ctypes.c_int
        L.kda_prefill_bwd_workspace_size.argtypes = [pp, ctypes.POINTER(ctypes.c_size_t)]
        L.kda_prefill_bwd_workspace_size.restype = ctypes.c_int
        L.kda_conv_gates_fwd.argtypes = [pp, ctypes.c_int32] + [P] * 14
        L.kda_conv_gates_fwd.restype = ctypes.c_int
        L.kda_set_stage_events.argtypes = [P, ctypes.c_int32]
        L.kda_set_stage_events.restype = ctypes.c_int
        _lib = L
        return L


def status_string(status: int) -> str:
    try:
        return load().kda_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - only when the library itself is missing
        return "unknown"

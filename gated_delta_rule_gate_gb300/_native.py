"""ctypes view of the C ABI declared in include/gdn.h (libgdn.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind these symbols.  There is no CPU fallback; if the library is
missing and cannot be built, loading raises.
"""
import ctypes
import os
import threading

from . import build as _build

GDN_OK, GDN_ERR_INVALID, GDN_ERR_UNSUPPORTED, GDN_ERR_WORKSPACE, GDN_ERR_CUDA = range(5)
DTYPE_F32, DTYPE_F16, DTYPE_BF16 = 0, 1, 2
RULES = {"linear": 0, "gated": 1, "delta": 2, "gated_delta": 3, "gdn2": 4}
FLAG_L2NORM_Q, FLAG_L2NORM_K, FLAG_BETA_SIGMOID, FLAG_DECAY_PER_KEY = 0x1, 0x2, 0x4, 0x8
FLAG_BETA_SHARED = 0x10
FLAG_STATE_KMAJOR = 0x20
DEVERR_BAD_SLOT, DEVERR_TIMEOUT, DEVERR_OVERLAP, DEVERR_DECAY_RANGE = 0x1, 0x2, 0x4, 0x8

EXPORTS = ("gdn_gate", "gdn_recurrent_step", "gdn_chunked_prefill_workspace_size",
           "gdn_chunked_prefill_workspace_size_min", "gdn_chunked_prefill", "gdn_chunked_prefill_noalloc",
           "gdn_status_string", "gdn_last_error_message")

_vp = ctypes.c_void_p


class GdnProblem(ctypes.Structure):
    """Mirror of ``gdn_problem`` (include/gdn.h)."""
    _fields_ = [
        ("batch", ctypes.c_int32), ("total_tokens", ctypes.c_int32), ("seq_len", ctypes.c_int32),
        ("num_heads_q", ctypes.c_int32), ("num_heads_v", ctypes.c_int32),
        ("head_dim_k", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
        ("num_state_rows", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
        ("decay_dtype", ctypes.c_int32), ("beta_dtype", ctypes.c_int32),
        ("rule", ctypes.c_int32), ("flags", ctypes.c_uint32), ("scale", ctypes.c_float),
        ("state_update_capacity", ctypes.c_int32),
        ("q", _vp), ("k", _vp), ("v", _vp), ("o", _vp), ("decay", _vp),
        ("gate_bias", _vp), ("gate_scale", _vp), ("beta", _vp),
        ("cu_seqlens", _vp), ("slot_ids", _vp), ("initial_state", _vp),
        ("final_state", _vp), ("error_word", _vp), ("seq_lens", _vp),
        ("erase_gate", _vp), ("write_gate", _vp),
    ]


class GdnGateArgs(ctypes.Structure):
    """Mirror of ``gdn_gate_args`` (include/gdn.h)."""
    _fields_ = [
        ("n", ctypes.c_int64), ("heads", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("a", _vp), ("dt_bias", _vp), ("decay_scale", _vp), ("b", _vp),
        ("decay_out", _vp), ("beta_out", _vp),
    ]


class GdnError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__("%s: %s" % (status_string(status), message))


_lib = None
_lock = threading.Lock()


def library_path():
    return _build.LIB


def load():
    """Loads libgdn.so (building it first when out of date and nvcc exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not _build.up_to_date():
            try:
                _build.build()
            except RuntimeError:
                if not os.path.exists(_build.LIB):
                    raise
        if not os.path.exists(_build.LIB):
            raise RuntimeError("libgdn.so is missing: build it with gated_delta_rule_gate_gb300.build.build()")
        lib = ctypes.CDLL(_build.LIB)
        lib.gdn_gate.argtypes = [ctypes.POINTER(GdnGateArgs), _vp]
        lib.gdn_gate.restype = ctypes.c_int
        lib.gdn_recurrent_step.argtypes = [ctypes.POINTER(GdnProblem), _vp]
        lib.gdn_recurrent_step.restype = ctypes.c_int
        lib.gdn_chunked_prefill_workspace_size.argtypes = [ctypes.POINTER(GdnProblem), ctypes.c_int32]
        lib.gdn_chunked_prefill_workspace_size.restype = ctypes.c_size_t
        lib.gdn_chunked_prefill_workspace_size_min.argtypes = [ctypes.POINTER(GdnProblem), ctypes.c_int32]
        lib.gdn_chunked_prefill_workspace_size_min.restype = ctypes.c_size_t
        lib.gdn_chunked_prefill.argtypes = [ctypes.POINTER(GdnProblem), ctypes.c_int32, _vp,
                                            ctypes.c_size_t, _vp]
        lib.gdn_chunked_prefill.restype = ctypes.c_int
        lib.gdn_chunked_prefill_noalloc.argtypes = [ctypes.POINTER(GdnProblem), ctypes.c_int32, _vp]
        lib.gdn_chunked_prefill_noalloc.restype = ctypes.c_int
        lib.gdn_status_string.argtypes = [ctypes.c_int]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_last_error_message.argtypes = []
        lib.gdn_last_error_message.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status):
    return load().gdn_status_string(int(status)).decode()


def last_error_message():
    return load().gdn_last_error_message().decode()


def check(status):
    if status != GDN_OK:
        raise GdnError(status, last_error_message())
    return status

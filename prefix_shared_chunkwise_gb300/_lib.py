"""ctypes binding of the C ABI in ``include/harts.h`` (argument marshalling only).

Loads the in-tree ``_harts.so``.  There is no fallback: if the library is missing
or fails to load, every call raises."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
SO_PATH = os.path.join(_HERE, "_harts.so")

HARTS_FP32, HARTS_BF16 = 0, 1
HARTS_KERNEL_AUTO, HARTS_KERNEL_SIMT, HARTS_KERNEL_TC = 0, 1, 2
HARTS_PLAN_NODEWISE = 1                       # harts_plan_calls flags
HARTS_PLAN_NOREPLAY = 2

ERRORS = {0: "HARTS_OK", -1: "HARTS_EINVAL", -2: "HARTS_EUNSUPPORTED", -3: "HARTS_EOVERFLOW",
          -4: "HARTS_ESMALLBUF", -5: "HARTS_ECUDA", -6: "HARTS_ETIMEOUT", -7: "HARTS_EDEVICE",
          -8: "HARTS_ENOPLAN"}

EXPORTED = [
    "harts_plan_calls", "harts_plan_get_info", "harts_plan_export", "harts_plan_device_bytes",
    "harts_plan_upload", "harts_plan_device_error", "harts_plan_free", "harts_selftest_timeout",
    "harts_kda_chunk_state_bytes", "harts_kda_fwd", "harts_kda_bwd_workspace_bytes",
    "harts_kda_bwd", "harts_kda_bwd_state", "harts_kda_bwd_grad", "harts_kda_bwd_static",
    "harts_kda_bwd_static_max_bytes", "harts_conv_fwd", "harts_conv_bwd_workspace_bytes",
    "harts_conv_bwd", "harts_plan_semantic_map", "harts_logprob_fwd", "harts_logprob_bwd",
    "harts_attn_fwd", "harts_attn_bwd_workspace_bytes", "harts_attn_bwd", "harts_last_error",
]

_i32, _i64, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
_pi32, _pi64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)


class PlanInfo(ctypes.Structure):
    _fields_ = [("n_seg", _i32), ("n_roots", _i32), ("n_leaves", _i32), ("chunk", _i32),
                ("n_rounds", _i32), ("n_seq", _i32), ("n_states", _i32), ("n_cons", _i32),
                ("C", _i64), ("S", _i64), ("R", _i64), ("n_chunks", _i64),
                ("max_seq_chunks", _i32), ("n_fold_rows", _i32), ("flags", ctypes.c_uint32)]


PLAN_ARRAY_FIELDS = [
    ("seg_offset", "i64", "n_seg"), ("seg_pos", "i64", "n_seg"), ("seg_seq", "i32", "n_seg"),
    ("seg_ctop", "i32", "n_seg"), ("seg_tpre", "i32", "n_seg"), ("seg_tin", "i32", "n_seg"),
    ("round_seq_ptr", "i32", "n_rounds+1"), ("cu_seqlens", "i64", "n_seq+1"),
    ("seq_round", "i32", "n_seq"), ("seq_first_seg", "i32", "n_seq"),
    ("seq_anchor", "i64", "n_seq"), ("seq_replay", "i32", "n_seq"), ("seq_src", "i32", "n_seq"),
    ("replay_ptr", "i64", "n_seq+1"), ("replay_idx", "i64", "R"),
    ("seq_state_ptr", "i32", "n_seq+1"), ("state_seq", "i32", "n_states"),
    ("state_pos", "i64", "n_states"), ("state_cons_ptr", "i32", "n_states+1"),
    ("state_cons", "i32", "n_cons"), ("root_cons_ptr", "i32", "n_roots+1"),
    ("root_cons", "i32", "n_seq-n_cons"),
]


class PlanArrays(ctypes.Structure):
    _fields_ = [(n, _pi64 if t == "i64" else _pi32) for n, t, _ in PLAN_ARRAY_FIELDS]


class FwdArgs(ctypes.Structure):
    _fields_ = [("H", _i32), ("dk", _i32), ("dv", _i32), ("dtype", _i32), ("kernel", _i32),
                ("scale", ctypes.c_float),
                ("q", _vp), ("k", _vp), ("v", _vp), ("g", _vp), ("beta", _vp), ("o", _vp),
                ("states", _vp), ("final_state", _vp), ("h0", _vp), ("chunk_states", _vp)]


class BwdArgs(ctypes.Structure):
    _fields_ = [("fwd", FwdArgs), ("d_o", _vp), ("d_final", _vp), ("dq", _vp), ("dk", _vp),
                ("dv", _vp), ("dg", _vp), ("dbeta", _vp), ("dh0", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t)]


class ConvFwdArgs(ctypes.Structure):
    _fields_ = [("channels", _i32), ("width", _i32), ("dtype", _i32), ("activation", _i32),
                ("x", _vp), ("weight", _vp), ("bias", _vp), ("y", _vp)]


class ConvBwdArgs(ctypes.Structure):
    _fields_ = [("fwd", ConvFwdArgs), ("dy", _vp), ("dx", _vp), ("dweight", _vp), ("dbias", _vp),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t)]


class LogprobFwdArgs(ctypes.Structure):
    _fields_ = [("C", _i64), ("V", _i32), ("dtype", _i32), ("S", _i64), ("logits", _vp),
                ("row_ptr", _vp), ("row_sem", _vp), ("target", _vp), ("lse", _vp), ("logp", _vp)]


class LogprobBwdArgs(ctypes.Structure):
    _fields_ = [("fwd", LogprobFwdArgs), ("dlogp", _vp), ("dlogits", _vp)]


class AttnFwdArgs(ctypes.Structure):
    _fields_ = [("H", _i32), ("d", _i32), ("dtype", _i32), ("scale", ctypes.c_float),
                ("q", _vp), ("k", _vp), ("v", _vp), ("o", _vp), ("lse", _vp)]


class AttnBwdArgs(ctypes.Structure):
    _fields_ = [("fwd", AttnFwdArgs), ("d_o", _vp), ("dq", _vp), ("dk", _vp), ("dv", _vp),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t)]


_lib = None


def lib():
    """The loaded library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(SO_PATH):
            raise RuntimeError(f"{SO_PATH} is missing: build it with "
                               "prefix_shared_chunkwise_gb300.build.build()")
        L = ctypes.CDLL(SO_PATH)
        L.harts_plan_calls.argtypes = [_i32, _pi32, _pi64, _i32, ctypes.c_uint32,
                                       ctypes.POINTER(_vp)]
        L.harts_plan_get_info.argtypes = [_vp, ctypes.POINTER(PlanInfo)]
        L.harts_plan_export.argtypes = [_vp, ctypes.POINTER(PlanArrays)]
        L.harts_plan_device_bytes.argtypes = [_vp]
        L.harts_plan_device_bytes.restype = ctypes.c_size_t
        L.harts_plan_upload.argtypes = [_vp, _vp, ctypes.c_size_t, _vp]
        L.harts_plan_device_error.argtypes = [_vp, _vp, _pi32]
        L.harts_plan_free.argtypes = [_vp]
        L.harts_plan_free.restype = None
        L.harts_selftest_timeout.argtypes = [_vp, ctypes.c_uint32, _vp]
        L.harts_selftest_timeout.restype = ctypes.c_int
        L.harts_kda_chunk_state_bytes.argtypes = [_vp, _i32, _i32, _i32, _i32]
        L.harts_kda_chunk_state_bytes.restype = ctypes.c_size_t
        L.harts_kda_fwd.argtypes = [_vp, ctypes.POINTER(FwdArgs), _vp]
        L.harts_kda_bwd_workspace_bytes.argtypes = [_vp, _i32, _i32, _i32]
        L.harts_kda_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.harts_kda_bwd_static_max_bytes.argtypes = []
        L.harts_kda_bwd_static_max_bytes.restype = ctypes.c_size_t
        for fn in ("harts_kda_bwd", "harts_kda_bwd_state", "harts_kda_bwd_grad", "harts_kda_bwd_static"):
            getattr(L, fn).argtypes = [_vp, ctypes.POINTER(BwdArgs), _vp]
            getattr(L, fn).restype = ctypes.c_int
        L.harts_conv_fwd.argtypes = [_vp, ctypes.POINTER(ConvFwdArgs), _vp]
        L.harts_conv_fwd.restype = ctypes.c_int
        L.harts_conv_bwd.argtypes = [_vp, ctypes.POINTER(ConvBwdArgs), _vp]
        L.harts_conv_bwd.restype = ctypes.c_int
        L.harts_conv_bwd_workspace_bytes.argtypes = [_vp, _i32, _i32]
        L.harts_conv_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.harts_plan_semantic_map.argtypes = [_vp, _pi32, _pi32, _pi32]
        L.harts_plan_semantic_map.restype = ctypes.c_int
        L.harts_logprob_fwd.argtypes = [ctypes.POINTER(LogprobFwdArgs), _vp]
        L.harts_logprob_fwd.restype = ctypes.c_int
        L.harts_logprob_bwd.argtypes = [ctypes.POINTER(LogprobBwdArgs), _vp]
        L.harts_logprob_bwd.restype = ctypes.c_int
        L.harts_attn_fwd.argtypes = [_vp, ctypes.POINTER(AttnFwdArgs), _vp]
        L.harts_attn_fwd.restype = ctypes.c_int
        L.harts_attn_bwd_workspace_bytes.argtypes = [_vp, _i32]
        L.harts_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.harts_attn_bwd.argtypes = [_vp, ctypes.POINTER(AttnBwdArgs), _vp]
        L.harts_attn_bwd.restype = ctypes.c_int
        L.harts_last_error.argtypes = []
        L.harts_last_error.restype = ctypes.c_char_p
        for fn in ("harts_plan_calls", "harts_plan_get_info", "harts_plan_export",
                   "harts_plan_upload", "harts_plan_device_error", "harts_kda_fwd",
                   "harts_kda_bwd"):
            getattr(L, fn).restype = ctypes.c_int
        _lib = L
    return _lib


class HartsError(RuntimeError):
    def __init__(self, rc, where):
        msg = lib().harts_last_error().decode(errors="replace")
        super().__init__(f"{where}: {ERRORS.get(rc, rc)}: {msg}")
        self.rc = rc


def check(rc, where):
    if rc != 0:
        raise HartsError(rc, where)

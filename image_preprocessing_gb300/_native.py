"""ctypes binding to libtrfn.so: argument marshalling only.

Every step of the fused path runs in the library's CUDA kernels; this module
only turns tensors into pointers and sizes and status codes into exceptions.
It never falls back to another implementation: if the library is missing the
import of any entry point raises.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtrfn.so")
LIB_BOUNDS_PATH = os.path.join(_HERE, "libtrfn_bounds.so")

TR_OK = 0
STATUS_NAMES = {0: "TR_OK", 1: "TR_ERR_INVALID_ARGUMENT", 2: "TR_ERR_NOT_SUPPORTED", 3: "TR_ERR_CUDA",
                4: "TR_ERR_TIMEOUT", 5: "TR_ERR_DEVICE", 6: "TR_END_OF_DATA"}


class TrError(RuntimeError):
    """A non-zero tr_status from the library."""

    def __init__(self, status, where, detail=""):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        msg = "%s returned %s" % (where, name)
        if detail:
            msg += ": " + detail
        super().__init__(msg)


class AugParam(ctypes.Structure):
    _fields_ = [("flip", ctypes.c_int32), ("y0", ctypes.c_int32), ("x0", ctypes.c_int32),
                ("h", ctypes.c_int32), ("w", ctypes.c_int32)]


class StageSlot(ctypes.Structure):
    _fields_ = [("image", ctypes.c_void_p), ("record", ctypes.c_void_p), ("sample", ctypes.c_longlong),
                ("batch", ctypes.c_longlong), ("index", ctypes.c_int), ("zone", ctypes.c_int)]


class StageBatch(ctypes.Structure):
    _fields_ = [("images", ctypes.c_void_p), ("records", ctypes.c_void_p), ("batch", ctypes.c_longlong),
                ("count", ctypes.c_int), ("zone", ctypes.c_int)]


class Batch(ctypes.Structure):
    """tr_batch: one batch of a tr_fused_norm_batches call."""
    _fields_ = [("src_u8", ctypes.c_void_p), ("dst", ctypes.c_void_p), ("aug_params", ctypes.c_void_p)]


class AugSampling(ctypes.Structure):
    _fields_ = [("flip_enabled", ctypes.c_int), ("flip_p", ctypes.c_float), ("erase_enabled", ctypes.c_int),
                ("erase_p", ctypes.c_float), ("scale_lo", ctypes.c_float), ("scale_hi", ctypes.c_float),
                ("ratio_lo", ctypes.c_float), ("ratio_hi", ctypes.c_float)]


_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_fp = ctypes.POINTER(ctypes.c_float)
_u64 = ctypes.c_uint64

_SIGNATURES = {
    "tr_fused_norm": (_i, [_vp, _vp, _i, _i, _i, _i, _fp, _fp, _vp, _i, _i, _vp]),
    "tr_fused_norm_variant": (_i, [_vp, _vp, _i, _i, _i, _i, _fp, _fp, _vp, _i, _i, _vp, _i]),
    "tr_fused_norm_ws": (_i, [_vp, _vp, _i, _i, _i, _i, _fp, _fp, _vp, _i, _i, _vp, _i, _vp]),
    "tr_fused_norm_ex": (_i, [_vp, _vp, _i, _i, _i, _i, _fp, _fp, _vp, _i, _i, _vp, _i, _vp, ctypes.c_uint]),
    "tr_workspace_bytes": (ctypes.c_size_t, []),
    "tr_fused_norm_batches": (_i, [ctypes.POINTER(Batch), _i, _i, _i, _i, _i, _fp, _fp, _i, _i, _vp, _vp,
                                   ctypes.c_uint]),
    "tr_fused_norm_sampled": (_i, [_vp, _vp, _i, _i, _i, _i, _fp, _fp, _u64, _u64, ctypes.POINTER(AugSampling), _vp,
                                   ctypes.POINTER(_u64), _i, _i, _vp, _i, _vp]),
    "tr_fused_norm_sampled_ex": (_i, [_vp, _vp, _i, _i, _i, _i, _fp, _fp, _u64, _u64, ctypes.POINTER(AugSampling), _vp,
                                      ctypes.POINTER(_u64), _i, _i, _vp, _i, _vp, ctypes.c_uint]),
    "tr_fused_norm_crop": (_i, [_vp, _i, _i, ctypes.c_size_t, ctypes.c_size_t, _vp, _vp, _i, _i, _i, _i, _fp, _fp,
                                _vp, _i, _i, _vp, _i, _vp]),
    "tr_fused_norm_crop_ex": (_i, [_vp, _i, _i, ctypes.c_size_t, ctypes.c_size_t, _vp, _vp, _i, _i, _i, _i, _fp, _fp,
                                   _vp, _i, _i, _vp, _i, _vp, ctypes.c_uint]),
    "tr_fused_norm_noalloc": (_i, [_vp, _vp, _i, _i, _i, _i, _fp, _fp, _vp, _i, _i, _vp]),
    "tr_fused_norm_geometry": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.c_uint, ctypes.POINTER(_i),
                                    ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    "tr_fused_norm_plan": (_i, [_vp, _vp, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_i)]),
    "tr_norm_preset": (_i, [_i, _fp, _fp, ctypes.POINTER(_i)]),
    "tr_sample_aug_params": (_i, [_u64, _u64, _i, _i, _i, _i, _f, _i, _f, _f, _f, _f, _f, _vp,
                                  ctypes.POINTER(_u64)]),
    "tr_sample_aug_params_device": (_i, [_u64, _u64, _i, _i, _i, _i, _f, _i, _f, _f, _f, _f, _f, _vp,
                                         ctypes.POINTER(_u64), _vp]),
    "tr_validate_aug_params": (_i, [_vp, _i, _i, _i, ctypes.POINTER(_i)]),
    "tr_ts_slot_bytes": (ctypes.c_size_t, [_i, _i, _i, _i]),
    "tr_ts_create": (_i, [_i, ctypes.POINTER(_vp), ctypes.c_size_t, _vp, _vp, _vp, ctypes.POINTER(_vp)]),
    "tr_ts_submit": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _fp, _fp, _i, _i,
                          ctypes.POINTER(ctypes.c_longlong)]),
    "tr_ts_submit_partial": (_i, [_vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _fp, _fp, _i, _i,
                                  ctypes.POINTER(ctypes.c_longlong)]),
    "tr_ts_submit_staged": (_i, [_vp, _vp, ctypes.POINTER(StageBatch), _i, _vp, _vp, _i, _i, _i, _i, _fp, _fp,
                                 _i, _i, ctypes.POINTER(ctypes.c_longlong)]),
    "tr_stage_zone_bytes": (ctypes.c_size_t, [_i, _i, _i, _i]),
    "tr_stage_create": (_i, [ctypes.POINTER(_vp), ctypes.c_size_t, _i, _i, _i, _i, _i, ctypes.POINTER(_vp)]),
    "tr_stage_acquire": (_i, [_vp, ctypes.c_longlong, _i, ctypes.POINTER(StageSlot)]),
    "tr_stage_commit": (_i, [_vp, ctypes.POINTER(StageSlot)]),
    "tr_stage_close": (_i, [_vp, ctypes.c_longlong]),
    "tr_stage_wait_readable": (_i, [_vp, _i, ctypes.POINTER(StageBatch)]),
    "tr_stage_release": (_i, [_vp, ctypes.c_longlong]),
    "tr_stage_destroy": (_i, [_vp]),
    "tr_ts_sync": (_i, [_vp, _i]),
    "tr_ts_destroy": (_i, [_vp]),
    "tr_device_status": (_i, [ctypes.POINTER(_i), _i]),
    "tr_launch_count": (_u64, []),
    "tr_tune_tiled": (_i, [_i, _i, _i, _i]),
    "tr_status_string": (ctypes.c_char_p, [_i]),
    "tr_last_error_message": (ctypes.c_char_p, []),
    "tr_version": (_i, []),
}


def _load(path):
    if not os.path.exists(path):
        raise ImportError(
            "%s is not built; build it with `python -m image_preprocessing_gb300.build` "
            "or __graft_entry__.build()" % path)
    L = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    """The loaded libtrfn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


_checked = None


def checked_lib():
    """libtrfn_bounds.so: the same C ABI with the tiled kernel's bounds and
    alignment checks compiled in (tr_device_status bit 1, site number in bits
    8..15, on a failed check).  A separate library with its own device status
    word; for tests only."""
    global _checked
    if _checked is None:
        _checked = _load(LIB_BOUNDS_PATH)
    return _checked


def check(status, where):
    if status != TR_OK:
        detail = ""
        if status == 3:
            detail = lib().tr_last_error_message().decode(errors="replace")
        raise TrError(status, where, detail)


def float_array(values):
    arr = (ctypes.c_float * 4)()
    for i, v in enumerate(values):
        arr[i] = float(v)
    return arr

"""CPU oracle for FusedNormalization — TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline / reference legs
of `bench.py` may import this package.  The product library and its Python
binding never import it; nothing here is shared with the CUDA path.

Every function wraps the plain C restatement in `fused_norm_oracle.c`, which
follows the Tech-Renaissance FusedNormalization article
(tech-renaissance.cn/blog/?p=487): §五 (what is fused), §六/§八 (FP32 and
FP16 outputs, 4-channel padding), §九 (normalisation presets), §十 (the
Philox-driven random decisions) and §十二 (random erasing).

Parity status: every function here is pinned by tests/test_oracle.py; none is
"parity unpinned" except the mapping from (seed, offset) to a uniform number,
which the article defers to a post that is not available (the sampler's
*distribution* is pinned, its exact stream against the article's is not).
"""
import ctypes
import os

import numpy as np

from .build import build_oracle

OUT_F32, OUT_F16 = 0, 1
LAYOUT_NHWC, LAYOUT_NCHW, LAYOUT_NHWC4 = 0, 1, 2
PRESETS = {"NO_NORM": 0, "MNIST": 1, "CIFAR": 2, "IMAGENET": 3, "MLPERF": 4}

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = bind(build_oracle())
    return _lib


def bind(path):
    """Load a library built from fused_norm_oracle.c and declare its functions."""
    L = ctypes.CDLL(path)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    f32p = ctypes.POINTER(ctypes.c_float)
    i32p = ctypes.POINTER(ctypes.c_int32)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    u32p = ctypes.POINTER(ctypes.c_uint32)
    u64p = ctypes.POINTER(ctypes.c_uint64)
    L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
    L.oracle_f32_to_f16.restype = ctypes.c_uint16
    L.oracle_f32_to_f16_array.argtypes = [f32p, u16p, ctypes.c_size_t]
    L.oracle_f32_to_f16_bits_range.argtypes = [ctypes.c_uint32, ctypes.c_uint32, u16p]
    L.oracle_norm_preset.argtypes = [ctypes.c_int, f32p, f32p, ctypes.POINTER(ctypes.c_int)]
    L.oracle_norm_preset.restype = ctypes.c_int
    L.oracle_fused_norm.argtypes = [u8p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, f32p, f32p, i32p, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int]
    L.oracle_fused_norm.restype = ctypes.c_int
    L.oracle_fused_norm_crop.argtypes = [u8p, ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                         i32p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, f32p, f32p, i32p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int]
    L.oracle_fused_norm_crop.restype = ctypes.c_int
    L.oracle_exp_f32_array.argtypes = [f32p, f32p, ctypes.c_size_t]
    L.oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
    L.oracle_uniform01.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
    L.oracle_uniform01.restype = ctypes.c_float
    L.oracle_sample_aug_params.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                           ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                           ctypes.c_float, ctypes.c_float, ctypes.c_float, i32p, u64p]
    L.oracle_sample_aug_params.restype = ctypes.c_int
    L.oracle_sample_aug_params_blocked.argtypes = L.oracle_sample_aug_params.argtypes
    L.oracle_sample_aug_params_blocked.restype = ctypes.c_int
    return L


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def f32_to_f16_bits(x):
    """binary32 array -> binary16 bit patterns (uint16), RNE."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().oracle_f32_to_f16_array(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint16), x.size)
    return out


def f32_bits_range_to_f16(first, count):
    out = np.empty(count, dtype=np.uint16)
    lib().oracle_f32_to_f16_bits_range(first, count, _ptr(out, ctypes.c_uint16))
    return out


def norm_preset(name_or_id):
    pid = PRESETS[name_or_id] if isinstance(name_or_id, str) else int(name_or_id)
    mean = np.zeros(3, np.float32)
    std = np.zeros(3, np.float32)
    ch = ctypes.c_int(0)
    rc = lib().oracle_norm_preset(pid, _ptr(mean, ctypes.c_float), _ptr(std, ctypes.c_float), ctypes.byref(ch))
    if rc != 0:
        raise ValueError("unknown preset %r" % (name_or_id,))
    return mean[: ch.value].copy(), std[: ch.value].copy(), ch.value


def fused_norm(src, mean, std, aug=None, out_dtype=OUT_F32, layout=LAYOUT_NHWC, n_range=None):
    """Oracle output for a uint8 NHWC batch `src` of shape (N, H, W, C).

    Returns float32 (OUT_F32) or uint16 binary16 bit patterns (OUT_F16), shaped
    (N,H,W,C), (N,C,H,W) or (N,H,W,4) for NHWC, NCHW and NHWC4.
    `n_range=(a, b)` computes only images a..b-1 (others stay zero)."""
    src = np.ascontiguousarray(src, dtype=np.uint8)
    N, H, W, C = src.shape
    mean = np.ascontiguousarray(mean, dtype=np.float32)
    std = np.ascontiguousarray(std, dtype=np.float32)
    assert mean.size >= C and std.size >= C
    if layout == LAYOUT_NCHW:
        shape = (N, C, H, W)
    elif layout == LAYOUT_NHWC4:
        shape = (N, H, W, 4)
    else:
        shape = (N, H, W, C)
    dst = np.zeros(shape, dtype=np.float32 if out_dtype == OUT_F32 else np.uint16)
    augp = None
    if aug is not None:
        aug = np.ascontiguousarray(aug, dtype=np.int32).reshape(N, 5)
        augp = _ptr(aug, ctypes.c_int32)
    a, b = (0, N) if n_range is None else n_range
    rc = lib().oracle_fused_norm(_ptr(src, ctypes.c_uint8), dst.ctypes.data_as(ctypes.c_void_p), N, H, W, C,
                                 _ptr(mean, ctypes.c_float), _ptr(std, ctypes.c_float), augp,
                                 int(out_dtype), int(layout), a, b)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dst


def fused_norm_crop(src_bytes, image_stride, row_stride, src_H, src_W, N, H, W, C, mean, std, crop=None,
                    aug=None, out_dtype=OUT_F32, layout=LAYOUT_NHWC):
    """Oracle output for H x W windows of a strided uint8 source.

    src_bytes: 1-D uint8 array holding N images, image n's byte (sy, sx, c) at
    n*image_stride + sy*row_stride + sx*C + c; crop: int32 (N, 2) {top, left}."""
    src_bytes = np.ascontiguousarray(src_bytes, dtype=np.uint8).reshape(-1)
    mean = np.ascontiguousarray(mean, dtype=np.float32)
    std = np.ascontiguousarray(std, dtype=np.float32)
    if layout == LAYOUT_NCHW:
        shape = (N, C, H, W)
    elif layout == LAYOUT_NHWC4:
        shape = (N, H, W, 4)
    else:
        shape = (N, H, W, C)
    dst = np.zeros(shape, dtype=np.float32 if out_dtype == OUT_F32 else np.uint16)
    cp = None
    if crop is not None:
        crop = np.ascontiguousarray(crop, dtype=np.int32).reshape(N, 2)
        cp = _ptr(crop, ctypes.c_int32)
    ap = None
    if aug is not None:
        aug = np.ascontiguousarray(aug, dtype=np.int32).reshape(N, 5)
        ap = _ptr(aug, ctypes.c_int32)
    rc = lib().oracle_fused_norm_crop(_ptr(src_bytes, ctypes.c_uint8), image_stride, row_stride, src_H, src_W, cp,
                                      dst.ctypes.data_as(ctypes.c_void_p), N, H, W, C, _ptr(mean, ctypes.c_float),
                                      _ptr(std, ctypes.c_float), ap, int(out_dtype), int(layout), 0, N)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return dst


def philox4x32_10(ctr, key):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_ptr(c, ctypes.c_uint32), _ptr(k, ctypes.c_uint32), _ptr(out, ctypes.c_uint32))
    return out


def uniform01(seed, offset):
    return lib().oracle_uniform01(seed, offset)


def sample_aug_params(seed, offset, N, H, W, flip=True, flip_p=0.5, erase=True, erase_p=0.5,
                      scale=(0.02, 0.33), ratio=(0.3, 3.3)):
    """Per-image {flip, y0, x0, h, w} records (int32, shape (N,5)) and the next offset."""
    out = np.zeros((N, 5), np.int32)
    nxt = ctypes.c_uint64(0)
    rc = lib().oracle_sample_aug_params(seed, offset, N, H, W, int(flip), flip_p, int(erase), erase_p,
                                        scale[0], scale[1], ratio[0], ratio[1],
                                        _ptr(out, ctypes.c_int32), ctypes.byref(nxt))
    if rc != 0:
        raise ValueError("oracle sampler rejected the arguments")
    return out, nxt.value


def exp_f32(x):
    """The oracle's own binary32 exp (Cody-Waite reduction, degree-7 Taylor)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    lib().oracle_exp_f32_array(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_float), x.size)
    return out


DRAWS_PER_IMAGE = 24


def sample_aug_params_blocked(seed, offset, N, H, W, flip=True, flip_p=0.5, erase=True, erase_p=0.5,
                              scale=(0.02, 0.33), ratio=(0.3, 3.3)):
    """Records with one counter block of 24 draws per image (image n uses
    offsets offset + 24n + k); returns (int32 (N, 5), offset + 24N)."""
    out = np.zeros((N, 5), np.int32)
    nxt = ctypes.c_uint64(0)
    rc = lib().oracle_sample_aug_params_blocked(seed, offset, N, H, W, int(flip), flip_p, int(erase), erase_p,
                                                scale[0], scale[1], ratio[0], ratio[1],
                                                _ptr(out, ctypes.c_int32), ctypes.byref(nxt))
    if rc != 0:
        raise ValueError("oracle sampler rejected the arguments")
    return out, nxt.value

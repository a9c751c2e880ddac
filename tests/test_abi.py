"""Host-side tests of the C ABI: symbols, argument checks, presets, the
sampler against the oracle's independent sampler, planning.  No GPU needed:
every call here either stops at host validation or never touches CUDA."""
import ctypes
import os
import re
import subprocess
import sys

import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, NOT_SUPPORTED = 0, 1, 2


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(tr_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_library_exports_every_declared_function():
    names = _declared_functions()
    assert "tr_fused_norm" in names and "tr_ts_submit" in names and len(names) >= 16
    L = _native.lib()
    for n in names:
        assert hasattr(L, n), n


def test_binding_covers_every_declared_function():
    assert set(_declared_functions()) <= set(_native._SIGNATURES)


def _f4(v):
    return _native.float_array(v)


M3, S3 = _f4([0.485, 0.456, 0.406]), _f4([0.229, 0.224, 0.225])


@pytest.mark.parametrize("args,status", [
    ((-1, 2, 2, 3, 0, 0), INVALID),      # N < 0
    ((1, 0, 2, 3, 0, 0), INVALID),       # H < 1
    ((1, 2, 0, 3, 0, 0), INVALID),       # W < 1
    ((1, 2, 2, 0, 0, 0), INVALID),       # C < 1
    ((1, 2, 2, 5, 0, 0), NOT_SUPPORTED),  # C > 4
    ((1, 2, 2, 3, 2, 0), INVALID),       # unknown dtype
    ((1, 2, 2, 3, 0, 3), INVALID),       # unknown layout
    ((1, 1 << 20, 1 << 20, 3, 0, 0), INVALID),  # beyond 2^40 elements
])
def test_invalid_shapes_rejected_before_launch(args, status):
    N, H, W, C, dt, lay = args
    L = _native.lib()
    assert L.tr_fused_norm(0x10000, 0x100000000, N, H, W, C, M3, S3, None, dt, lay, None) == status


def test_null_and_bad_constants_rejected():
    L = _native.lib()
    assert L.tr_fused_norm(None, 0x1000, 1, 2, 2, 3, M3, S3, None, 0, 0, None) == INVALID
    assert L.tr_fused_norm(0x1000, None, 1, 2, 2, 3, M3, S3, None, 0, 0, None) == INVALID
    assert L.tr_fused_norm(0x1000, 0x100000, 1, 2, 2, 3, None, S3, None, 0, 0, None) == INVALID
    for bad in ([0.2, 0.0, 0.2], [0.2, float("nan"), 0.2], [0.2, float("inf"), 0.2]):
        assert L.tr_fused_norm(0x1000, 0x100000, 1, 2, 2, 3, M3, _f4(bad), None, 0, 0, None) == INVALID
    assert L.tr_fused_norm(0x1000, 0x100000, 1, 2, 2, 3, _f4([0, float("nan"), 0]), S3, None, 0, 0, None) == INVALID
    # an output off its element alignment, records off int32 alignment
    assert L.tr_fused_norm(0x1000, 0x100002, 1, 2, 2, 3, M3, S3, None, 0, 0, None) == INVALID
    assert L.tr_fused_norm(0x1000, 0x100001, 1, 2, 2, 3, M3, S3, None, 1, 0, None) == INVALID
    assert L.tr_fused_norm(0x1000, 0x100000, 1, 2, 2, 3, M3, S3, 0x2002, 0, 0, None) == INVALID
    # a workspace off a 16-byte boundary
    assert L.tr_fused_norm_ws(0x1000, 0x100000, 1, 2, 2, 3, M3, S3, None, 0, 0, None, 0, 0x3004) == INVALID
    assert L.tr_workspace_bytes() == 2048
    # launch options: unknown bits, and the flag on otherwise bad arguments
    assert L.tr_fused_norm_ex(0x1000, 0x100000, 1, 2, 2, 3, M3, S3, None, 0, 0, None, 0, None, 2) == INVALID
    assert L.tr_fused_norm_ex(0x1000, 0x100000, 1, 2, 2, 3, M3, S3, None, 0, 0, None, 0, 0x3004, 1) == INVALID
    assert L.tr_fused_norm_ex(0x1000, 0x100000, 0, 2, 2, 3, M3, S3, None, 0, 0, None, 0, None, 1) == 0
    assert L.tr_fused_norm_crop_ex(0x1000, 2, 2, 6, 12, None, 0x100000, 1, 2, 2, 3, M3, S3, None, 0, 0, None, 0,
                                   None, 4) == INVALID
    # geometry diagnostic: argument checks before any device query
    r = [ctypes.c_int(0) for _ in range(5)]
    refs = [ctypes.byref(x) for x in r]
    assert L.tr_fused_norm_geometry(0x1000, 0x100000, 0, 224, 224, 3, 1, 0, 0, *refs) == INVALID        # N < 1
    assert L.tr_fused_norm_geometry(0x1000, 0x100000, 8, 224, 224, 3, 1, 0, 2, *refs) == INVALID        # flags
    assert L.tr_fused_norm_geometry(0x1000, 0x100000, 8, 224, 224, 3, 1, 0, 0, None, *refs[1:]) == INVALID
    assert L.tr_fused_norm_geometry(0x1001, 0x100000, 8, 224, 224, 3, 1, 0, 0, *refs) == 2   # unaligned source
    # overlapping src and dst
    assert L.tr_fused_norm(0x1000, 0x1004, 1, 2, 2, 3, M3, S3, None, 0, 0, None) == INVALID
    # a bad kernel choice
    assert L.tr_fused_norm_variant(0x1000, 0x100000, 1, 2, 2, 3, M3, S3, None, 0, 0, None, 9) == INVALID


def test_empty_batch_is_a_no_op():
    L = _native.lib()
    assert L.tr_fused_norm(None, None, 0, 2, 2, 3, M3, S3, None, 1, 0, None) == OK


def test_forced_tiled_on_unsupported_shape_is_not_supported():
    L = _native.lib()
    # rows of more than 2^24 bytes
    assert L.tr_fused_norm_variant(0x1000, 0x40000000, 1, 1, 1 << 23, 3, M3, S3, None, 0, 0, None, 1) == NOT_SUPPORTED
    # misaligned source pointer
    assert L.tr_fused_norm_variant(0x1001, 0x100000, 2, 32, 32, 3, M3, S3, None, 0, 0, None, 1) == NOT_SUPPORTED


@pytest.mark.parametrize("shape,dt,lay,src,dst,want", [
    ((256, 224, 224, 3), 1, 0, 0x1000, 0x10000000, 1),
    ((256, 224, 224, 3), 0, 1, 0x1000, 0x10000000, 1),
    ((16, 32, 32, 3), 0, 0, 0x1000, 0x10000000, 2),   # small batch: the per-element kernel
    ((86, 32, 32, 3), 0, 0, 0x1000, 0x10000000, 1),   # 264,192 output elements
    ((200, 28, 28, 1), 0, 0, 0x1000, 0x10000000, 2),  # W*C = 28
    ((128, 64, 12, 4), 1, 1, 0x1000, 0x10000000, 1),  # NCHW fp16 row of 24 bytes: the odd-row form
    ((256, 227, 227, 3), 1, 0, 0x1000, 0x10000000, 1),  # 681-byte rows: the odd-row form
    ((256, 224, 224, 3), 1, 0, 0x1000, 0x10000002, 1),  # dst 2 bytes off 16: the odd-row form
    ((128, 64, 12, 4), 0, 1, 0x1000, 0x10000000, 1),
    ((4, 8, 16, 3), 1, 0, 0x1008, 0x10000000, 2),     # src not 16-byte aligned
    ((4, 8, 16, 3), 1, 0, 0x1000, 0x10000004, 2),     # dst not 16-byte aligned
])
def test_plan_picks_the_kernel(shape, dt, lay, src, dst, want):
    assert trfn.tr_fused_norm_plan(src, dst, *shape, dt, lay) == want


def test_presets_match_the_article_table():
    expect = {
        "NO_NORM": ([0, 0, 0], [1, 1, 1], 3),
        "MNIST": ([0.1307], [0.3081], 1),
        "CIFAR": ([0.4914, 0.4822, 0.4465], [0.2470, 0.2435, 0.2616], 3),
        "IMAGENET": ([0.485, 0.456, 0.406], [0.229, 0.224, 0.225], 3),
        "MLPERF": ([123.68 / 255, 116.78 / 255, 103.94 / 255], [1 / 255] * 3, 3),
    }
    for name, (m, s, ch) in expect.items():
        mean, std, c = trfn.tr_norm_preset(name)
        assert c == ch
        np.testing.assert_allclose(mean, m, rtol=1e-6)
        np.testing.assert_allclose(std, s, rtol=1e-6)
    L = _native.lib()
    m, s, ch = (ctypes.c_float * 3)(), (ctypes.c_float * 3)(), ctypes.c_int()
    assert L.tr_norm_preset(5, m, s, ctypes.byref(ch)) == INVALID


@pytest.mark.parametrize("kw", [
    dict(seed=2003, offset=0, N=512, H=224, W=224),
    dict(seed=1, offset=12345, N=300, H=32, W=32, erase_p=0.9),
    dict(seed=7, offset=0, N=200, H=28, W=28, flip=False),
    dict(seed=9, offset=5, N=100, H=5, W=3, erase_p=1.0),
    dict(seed=2 ** 40 + 3, offset=2 ** 33, N=64, H=224, W=224, scale=(0.1, 0.5), ratio=(0.5, 2.0)),
    dict(seed=3, offset=0, N=50, H=224, W=224, erase=False),
    dict(seed=3, offset=0, N=50, H=224, W=224, flip_p=0.25, erase_p=0.3),
])
def test_sampler_matches_the_oracle_sampler(kw):
    kw = dict(kw)
    seed, offset, N, H, W = kw.pop("seed"), kw.pop("offset"), kw.pop("N"), kw.pop("H"), kw.pop("W")
    a, na = trfn.tr_sample_aug_params(seed, offset, N, H, W, **kw)
    b, nb = oracle.sample_aug_params(seed, offset, N, H, W, **kw)
    assert np.array_equal(a, b) and na == nb


def test_sampler_rejects_bad_arguments():
    L = _native.lib()
    nxt = ctypes.c_uint64()
    assert L.tr_sample_aug_params(0, 0, -1, 4, 4, 1, 0.5, 1, 0.5, 0.02, 0.33, 0.3, 3.3, None,
                                  ctypes.byref(nxt)) == INVALID
    assert L.tr_sample_aug_params(0, 0, 3, 4, 4, 1, 0.5, 1, 0.5, 0.02, 0.33, 0.3, 3.3, None,
                                  ctypes.byref(nxt)) == INVALID
    with pytest.raises(trfn.TrError):
        trfn.tr_sample_aug_params(0, 0, 4, 4, 4, ratio=(0.0, 3.3))
    with pytest.raises(trfn.TrError):
        trfn.tr_sample_aug_params(0, 0, 4, 4, 4, scale=(0.5, 0.1))


def test_validate_aug_params():
    good = np.array([[0, 0, 0, 0, 0], [1, 2, 3, 4, 5], [0, 0, 0, 10, 10], [1, 9, 9, -1, 3]], np.int32)
    assert trfn.tr_validate_aug_params(good, 10, 10) == -1
    bad = good.copy()
    bad[2, 3] = 11
    assert trfn.tr_validate_aug_params(bad, 10, 10) == 2
    bad = good.copy()
    bad[1, 2] = -1
    assert trfn.tr_validate_aug_params(bad, 10, 10) == 1


def test_slot_bytes_layout():
    # [images][records][filler image][filler record][workspace], each zone on a 256-byte boundary
    img = 224 * 224 * 3
    assert trfn.tr_ts_slot_bytes(256, 224, 224, 3) == 256 * img + 5120 + img + 256 + 2048
    assert trfn.tr_ts_slot_bytes(3, 5, 7, 3) == 512 + 256 + 256 + 256 + 2048
    assert trfn.tr_ts_slot_bytes(-1, 5, 7, 3) == 0


def test_status_strings():
    L = _native.lib()
    for s in range(6):
        assert L.tr_status_string(s)
    assert L.tr_status_string(99) == b"unknown status"
    assert L.tr_version() >= 100


def test_package_does_not_import_the_oracle_and_fails_without_library():
    code = (
        "import sys, image_preprocessing_gb300 as t;"
        "assert 'oracle' not in sys.modules;"
        "from image_preprocessing_gb300 import _native;"
        "_native.LIB_PATH = '/nonexistent/libtrfn.so'; _native._lib = None\n"
        "try:\n    _native.lib()\nexcept ImportError:\n    print('raised')\n"
    )
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert "raised" in out.stdout


def test_product_sources_never_reference_the_oracle():
    pkg = os.path.join(ROOT, "image_preprocessing_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cpp", ".h")):
                text = open(os.path.join(dirpath, fn), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text and "liboracle" not in text, fn


def test_crop_arguments_rejected_before_launch():
    L = _native.lib()
    # src_H < H, row stride below a row, image stride below an image
    assert L.tr_fused_norm_crop(0x1000, 10, 20, 60, 600, None, 0x100000, 1, 12, 16, 3, M3, S3, None, 0, 0,
                                None, 0, None) == INVALID
    assert L.tr_fused_norm_crop(0x1000, 20, 20, 50, 1200, None, 0x100000, 1, 12, 16, 3, M3, S3, None, 0, 0,
                                None, 0, None) == INVALID
    assert L.tr_fused_norm_crop(0x1000, 20, 20, 64, 600, None, 0x100000, 1, 12, 16, 3, M3, S3, None, 0, 0,
                                None, 0, None) == INVALID
    # crop origins off int32 alignment
    assert L.tr_fused_norm_crop(0x1000, 20, 20, 64, 1280, 0x5002, 0x100000, 1, 12, 16, 3, M3, S3, None, 0, 0,
                                None, 0, None) == INVALID
    # forced TILED where the source strides are not 16-byte multiples
    assert L.tr_fused_norm_crop(0x1000, 20, 20, 60, 1200, None, 0x100000, 1, 12, 16, 3, M3, S3, None, 0, 0,
                                None, 1, None) == NOT_SUPPORTED
    assert L.tr_fused_norm_crop(None, 20, 20, 64, 1280, None, None, 0, 12, 16, 3, M3, S3, None, 0, 0,
                                None, 0, None) == OK


def test_fused_sampled_host_checks():
    """tr_fused_norm_sampled's checks run on the host: an empty batch is a
    no-op that still reports the next offset; bad sampling settings, a
    missing sampling struct or missing records are rejected."""
    L = _native.lib()
    m = _native.float_array([0.5, 0.5, 0.5])
    s = _native.float_array([0.25, 0.25, 0.25])
    good = _native.AugSampling(1, 0.5, 1, 0.5, 0.02, 0.33, 0.3, 3.3)
    nxt = ctypes.c_uint64(7)
    assert L.tr_fused_norm_sampled(None, None, 0, 8, 8, 3, m, s, 1, 40, ctypes.byref(good), None,
                                   ctypes.byref(nxt), 1, 0, None, 0, None) == 0
    assert nxt.value == 40
    for bad in (_native.AugSampling(1, 0.5, 1, 0.5, 0.5, 0.1, 0.3, 3.3),        # scale bounds out of order
                _native.AugSampling(1, 0.5, 1, 0.5, 0.02, 0.33, 0.0, 3.3),      # ratio_lo <= 0
                _native.AugSampling(1, float("nan"), 0, 0.0, 0, 0, 0, 0)):      # non-finite p
        assert L.tr_fused_norm_sampled(None, None, 0, 8, 8, 3, m, s, 1, 0, ctypes.byref(bad), None, None,
                                       1, 0, None, 0, None) == 1
    assert L.tr_fused_norm_sampled(None, None, 0, 8, 8, 3, m, s, 1, 0, None, None, None, 1, 0, None, 0, None) == 1
    # N > 0 without a records buffer
    assert L.tr_fused_norm_sampled(0x1000, 0x200000, 4, 8, 8, 3, m, s, 1, 0, ctypes.byref(good), None, None,
                                   1, 0, None, 0, None) == 1


def test_batches_arguments_rejected_before_launch():
    """tr_fused_norm_batches checks everything on the host first: the batch
    count, the descriptors, every batch's pointers and that no output
    overlaps a source or another output (no GPU is touched here)."""
    L = _native.lib()
    B = _native.Batch

    def call(bs, K=None, N=2, H=4, W=16, C=3, dt=1, lay=0, ws=None, flags=0):
        arr = (B * max(1, len(bs)))(*bs) if bs else None
        return L.tr_fused_norm_batches(arr, len(bs) if K is None else K, N, H, W, C, M3, S3, dt, lay, None, ws,
                                       flags)

    img_in, img_out = 2 * 4 * 16 * 3, 2 * 4 * 16 * 3 * 2
    good = [B(0x100000 + k * 0x10000, 0x900000 + k * 0x10000, None) for k in range(3)]
    assert call([]) == 0                                   # K = 0: nothing to do
    assert call(good, N=0) == 0                            # N = 0: nothing to do
    assert call(good, K=-1) == INVALID
    assert call(good * 6) == INVALID                       # 18 > TR_MAX_BATCHES
    assert call([], K=2) == INVALID                        # no descriptors
    assert call(good, C=5) == NOT_SUPPORTED
    assert call(good, flags=2) == INVALID
    assert call(good, ws=0x3008) == INVALID                # workspace off 16 bytes
    assert call([good[0], B(None, 0x990000, None)]) == INVALID
    assert call([good[0], B(0x180000, 0x990001, None)]) == INVALID   # output off its element size
    assert call([good[0], B(0x180000, 0x990000, 0x2002)]) == INVALID  # records off int32
    # batch 1 writes over batch 0's source; batch 1 writes into batch 0's output
    assert call([good[0], B(0x180000, 0x100000 + img_in - 2, None)]) == INVALID
    assert call([good[0], B(0x180000, 0x900000 + img_out - 2, None)]) == INVALID

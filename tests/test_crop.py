"""GPU parity for windows of a strided source (tr_fused_norm_crop) against
the oracle's crop form: the TMA tensor-copy path (16-byte multiple strides),
the generic path (any stride), clamping of out-of-range origins, both
schedules, every layout and dtype."""
import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import synth
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

F32, F16 = trfn.OUT_F32, trfn.OUT_F16
NHWC, NCHW, NHWC4 = trfn.LAYOUT_NHWC, trfn.LAYOUT_NCHW, trfn.LAYOUT_NHWC4
MEAN = np.array(synth.IMAGENET_MEAN + (0.5,), np.float32)
STD = np.array(synth.IMAGENET_STD + (0.25,), np.float32)


def _strided(src, row_pad, image_pad):
    N, SH, SW, C = src.shape
    row_stride = SW * C + row_pad
    image_stride = SH * row_stride + image_pad
    buf = np.full(N * image_stride, 0xEE, np.uint8)
    for n in range(N):
        for y in range(SH):
            o = n * image_stride + y * row_stride
            buf[o:o + SW * C] = src[n, y].reshape(-1)
    return buf, image_stride, row_stride


def _run(buf, istr, rstr, SH, SW, N, H, W, C, crop, aug, dt, layout, variant=trfn.VARIANT_AUTO, ws=None,
         src_offset=0):
    import torch
    d_buf = torch.zeros(buf.size + src_offset + 64, dtype=torch.uint8, device="cuda")
    d_buf[src_offset:src_offset + buf.size].copy_(torch.from_numpy(buf))
    d_crop = None if crop is None else torch.from_numpy(np.ascontiguousarray(crop, np.int32)).cuda()
    d_aug = None if aug is None else torch.from_numpy(np.ascontiguousarray(aug, np.int32)).cuda()
    tdt = torch.float16 if dt == F16 else torch.float32
    out = torch.empty(trfn.out_shape(N, H, W, C, layout), dtype=tdt, device="cuda")
    trfn.tr_fused_norm_crop(d_buf.data_ptr() + src_offset, SH, SW, rstr, istr, out, N, H, W, C, MEAN[:C],
                            STD[:C], crop=d_crop, aug=d_aug, out_dtype=dt, layout=layout, variant=variant,
                            workspace=ws)
    torch.cuda.synchronize()
    o = out.cpu()
    return o.view(torch.int16).numpy().view(np.uint16) if dt == F16 else o.numpy()


CASES = [
    # (N, SH, SW, C, H, W, row_pad, image_pad): TMA path when strides are 16-byte multiples
    (8, 64, 80, 3, 48, 64, 0, 0),
    (6, 40, 64, 3, 32, 48, 16, 32),
    (4, 36, 32, 1, 20, 16, 0, 16),
    (5, 30, 40, 2, 24, 32, 32, 0),
    (3, 20, 28, 4, 12, 16, 0, 0),
    (2, 256, 256, 3, 224, 224, 0, 0),
    # generic path: strides off 16 bytes, odd widths
    (4, 21, 23, 3, 10, 13, 5, 7),
    (3, 17, 50, 3, 9, 16, 0, 0),     # src_W*C = 150, not a multiple of 16
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("dt", [F32, F16])
@pytest.mark.parametrize("layout", [NHWC, NCHW, NHWC4])
def test_crop_windows_match_the_oracle(case, dt, layout):
    N, SH, SW, C, H, W, rp, ip = case
    src = synth.pixels_uniform(SH + SW + C, N, SH, SW, C)
    buf, istr, rstr = _strided(src, rp, ip)
    g = np.random.default_rng(N * SH + W)
    crop = np.stack([g.integers(0, SH - H + 1, N), g.integers(0, SW - W + 1, N)], axis=1).astype(np.int32)
    crop[0] = (0, 0)
    crop[-1] = (SH - H, SW - W)
    aug = synth.random_records(7 + N, N, H, W, allow_outside=True)
    ref = oracle.fused_norm_crop(buf, istr, rstr, SH, SW, N, H, W, C, MEAN[:C], STD[:C], crop, aug, dt, layout)
    got = _run(buf, istr, rstr, SH, SW, N, H, W, C, crop, aug, dt, layout)
    assert_parity(got, ref, dt, str(case))
    tma = (rp % 16 == 0 and ip % 16 == 0 and (SW * C) % 16 == 0 and (W * C) % 16 == 0 and
           not (layout == NCHW and (W * (2 if dt == F16 else 4)) % 16))
    if tma:   # the TMA tensor path, whatever AUTO picks for a batch this size
        got = _run(buf, istr, rstr, SH, SW, N, H, W, C, crop, aug, dt, layout, trfn.VARIANT_TILED)
        assert_parity(got, ref, dt, str(case) + " tiled")


@pytest.mark.parametrize("case", CASES[:5])
def test_crop_tiled_and_generic_agree(case):
    N, SH, SW, C, H, W, rp, ip = case
    src = synth.pixels_uniform(3 * SW, N, SH, SW, C)
    buf, istr, rstr = _strided(src, rp, ip)
    crop = np.stack([np.arange(N) % (SH - H + 1), (3 * np.arange(N)) % (SW - W + 1)], axis=1).astype(np.int32)
    aug = synth.random_records(11, N, H, W)
    for dt in (F32, F16):
        a = _run(buf, istr, rstr, SH, SW, N, H, W, C, crop, aug, dt, NHWC, trfn.VARIANT_TILED)
        b = _run(buf, istr, rstr, SH, SW, N, H, W, C, crop, aug, dt, NHWC, trfn.VARIANT_GENERIC)
        assert np.array_equal(a, b)


def test_crop_origins_are_clamped_into_the_source():
    N, SH, SW, C, H, W = 4, 40, 48, 3, 24, 32
    src = synth.pixels_uniform(5, N, SH, SW, C)
    buf, istr, rstr = _strided(src, 0, 0)
    crop = np.array([[-5, -7], [100, 100], [SH - H, -1], [3, SW]], np.int32)
    clamped = np.stack([np.clip(crop[:, 0], 0, SH - H), np.clip(crop[:, 1], 0, SW - W)], axis=1)
    for variant in (trfn.VARIANT_TILED, trfn.VARIANT_GENERIC):
        got = _run(buf, istr, rstr, SH, SW, N, H, W, C, crop, None, F16, NHWC, variant)
        ref = oracle.fused_norm_crop(buf, istr, rstr, SH, SW, N, H, W, C, MEAN[:3], STD[:3], clamped, None, F16)
        assert_parity(got, ref, F16)


def test_crop_with_dynamic_schedule_and_null_origins():
    import torch
    N, SH, SW, C, H, W = 64, 256, 256, 3, 224, 224
    src = synth.pixels_gaussian(9, N, SH, SW, C)
    buf, istr, rstr = _strided(src, 0, 0)
    ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda")
    aug = oracle.sample_aug_params(13, 0, N, H, W)[0]
    crop = np.full((N, 2), 16, np.int32)   # a centre crop 256 -> 224
    for c in (crop, None):
        got = _run(buf, istr, rstr, SH, SW, N, H, W, C, c, aug, F16, NHWC, ws=ws)
        ref = oracle.fused_norm_crop(buf, istr, rstr, SH, SW, N, H, W, C, MEAN[:3], STD[:3], c, aug, F16)
        assert_parity(got, ref, F16)
        assert int(ws.count_nonzero()) == 0
    assert trfn.tr_device_status() == 0


def test_crop_misaligned_source_takes_the_generic_kernel():
    N, SH, SW, C, H, W = 3, 32, 32, 3, 16, 16
    src = synth.pixels_uniform(2, N, SH, SW, C)
    buf, istr, rstr = _strided(src, 0, 0)
    crop = np.array([[1, 2], [3, 4], [5, 6]], np.int32)
    got = _run(buf, istr, rstr, SH, SW, N, H, W, C, crop, None, F32, NCHW, src_offset=3)
    ref = oracle.fused_norm_crop(buf, istr, rstr, SH, SW, N, H, W, C, MEAN[:3], STD[:3], crop, None, F32, NCHW)
    assert_parity(got, ref, F32)

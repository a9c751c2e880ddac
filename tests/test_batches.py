"""tr_fused_norm_batches: K batches of one shape in one launch.

Each batch's output must equal the oracle's (binary32 max-abs 2e-6, binary16
1 ulp, exact +0) and, bit for bit, tr_fused_norm's on that batch alone: the
launch only changes which band of which batch a CTA converts.  The article's
execute() runs once per batch (FusedNormalization article §五); one launch
over K batches pays the per-launch ramp and drain once."""
import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import synth
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

F32, F16 = trfn.OUT_F32, trfn.OUT_F16
NHWC, NCHW, NHWC4 = trfn.LAYOUT_NHWC, trfn.LAYOUT_NCHW, trfn.LAYOUT_NHWC4
# ImageNet constants, and a fourth channel for 4-channel images
MEAN = np.array(synth.IMAGENET_MEAN + (0.5,), np.float32)
STD = np.array(synth.IMAGENET_STD + (0.25,), np.float32)


def _host(t, dt):
    import torch
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if dt == F16 else t.numpy()


def _make(K, N, H, W, C, dt, layout, seed, coords=False, records=True):
    """K batches on the device: pixels, records (every third batch none),
    outputs filled with a pattern the kernel must overwrite."""
    import torch
    tdt = torch.float16 if dt == F16 else torch.float32
    shape = trfn.out_shape(N, H, W, C, layout)
    batches, host = [], []
    for k in range(K):
        px = synth.coordinate_image(N, H, W, C) if coords else synth.pixels_uniform(seed + k, N, H, W, C)
        if coords:
            px = np.ascontiguousarray(np.roll(px, k, axis=0))
        rec = None
        if records and k % 3 != 2:
            rec = synth.random_records(seed + 50 + k, N, H, W, allow_outside=True)
        src = torch.from_numpy(px).cuda()
        aug = torch.from_numpy(rec).cuda() if rec is not None else None
        dst = torch.full(shape, float("nan"), dtype=tdt, device="cuda")
        batches.append((src, dst, aug))
        host.append((px, rec))
    return batches, host


def _check(batches, host, dt, layout, what):
    import torch
    for k, ((src, dst, aug), (px, rec)) in enumerate(zip(batches, host)):
        got = _host(dst, dt)
        ref = oracle.fused_norm(px, MEAN[:px.shape[3]], STD[:px.shape[3]], rec, out_dtype=dt, layout=layout)
        assert_parity(got, ref, dt, "%s batch %d" % (what, k))
        alone = torch.empty_like(dst)
        trfn.tr_fused_norm(src, alone, MEAN[:px.shape[3]], STD[:px.shape[3]], aug, out_dtype=dt, layout=layout)
        torch.cuda.synchronize()
        assert np.array_equal(_host(alone, dt).view(np.uint8), got.view(np.uint8)), "%s batch %d" % (what, k)


@pytest.mark.parametrize("K", [2, 4, 8])
def test_headline_shape_one_launch(K):
    import torch
    N, H, W, C = 48, 224, 224, 3
    batches, host = _make(K, N, H, W, C, F16, NHWC, 100 * K)
    before = trfn.tr_launch_count()
    trfn.tr_fused_norm_batches(batches, MEAN[:C], STD[:C], out_dtype=F16, layout=NHWC)
    torch.cuda.synchronize()
    assert trfn.tr_launch_count() == before + 1, "K batches in one launch"
    _check(batches, host, F16, NHWC, "K=%d" % K)
    assert trfn.tr_device_status() == 0


@pytest.mark.parametrize("dt", [F32, F16])
@pytest.mark.parametrize("layout", [NHWC, NCHW, NHWC4])
@pytest.mark.parametrize("shape", [(16, 40, 64, 3), (40, 33, 48, 1), (20, 24, 32, 4), (40, 17, 40, 2),
                                   (2, 8, 16, 3)])
def test_layouts_and_channels_with_coordinate_images(shape, layout, dt):
    """Coordinate images (a misplaced element shows) and records that stick
    out of the image; five batches in one launch of the tiled kernel, whereas
    each batch alone is small enough for the per-element kernel (the two
    agree bit for bit).  The last shape is below the tiled kernel's threshold
    even for all five batches together: one per-element launch per batch."""
    import torch
    N, H, W, C = shape
    K = 5
    batches, host = _make(K, N, H, W, C, dt, layout, 7 + N, coords=True)
    oc = 4 if layout == NHWC4 else C
    one = K * N * H * W * oc >= 1 << 18
    before = trfn.tr_launch_count()
    trfn.tr_fused_norm_batches(batches, MEAN[:C], STD[:C], out_dtype=dt, layout=layout)
    torch.cuda.synchronize()
    assert trfn.tr_launch_count() == before + (1 if one else K)
    _check(batches, host, dt, layout, "shape %s" % (shape,))


@pytest.mark.parametrize("dt,layout", [(F16, NHWC), (F32, NHWC), (F16, NCHW)])
def test_odd_rows_one_launch(dt, layout):
    """227-pixel RGB rows (681 bytes, not a multiple of 16): the odd-row form
    of the kernel, with each batch's bytes realigned from its own base."""
    import torch
    K, N, H, W, C = 3, 12, 227, 227, 3
    batches, host = _make(K, N, H, W, C, dt, layout, 31)
    before = trfn.tr_launch_count()
    trfn.tr_fused_norm_batches(batches, MEAN[:C], STD[:C], out_dtype=dt, layout=layout)
    torch.cuda.synchronize()
    assert trfn.tr_launch_count() == before + 1
    _check(batches, host, dt, layout, "odd rows")


def test_unaligned_output_launches_each_batch():
    """An output off a 16-byte boundary: each batch gets its own launch,
    with the same results."""
    import torch
    K, N, H, W, C = 3, 16, 64, 64, 3
    batches, host = _make(K, N, H, W, C, F16, NHWC, 41)
    n_el = N * H * W * C
    buf = torch.full((n_el + 8,), float("nan"), dtype=torch.float16, device="cuda")
    off = buf[1:1 + n_el].view(N, H, W, C)   # 2 bytes past a 16-byte boundary
    batches[1] = (batches[1][0], off, batches[1][2])
    before = trfn.tr_launch_count()
    trfn.tr_fused_norm_batches(batches, MEAN[:C], STD[:C], out_dtype=F16, layout=NHWC)
    torch.cuda.synchronize()
    assert trfn.tr_launch_count() == before + K
    _check(batches, host, F16, NHWC, "unaligned")


def test_dynamic_schedule_and_overlapped_chain():
    """Six launches of four batches each in a stream, overlapping one another
    (independent buffers, workspaces alternating), against the oracle; the
    workspaces are zero again afterwards."""
    import torch
    K, N, H, W, C = 4, 32, 160, 160, 3
    stream = torch.cuda.Stream()
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    groups = [_make(K, N, H, W, C, F16, NHWC, 500 + 10 * g) for g in range(6)]
    with torch.cuda.stream(stream):
        for g, (batches, _) in enumerate(groups):
            trfn.tr_fused_norm_batches(batches, MEAN[:C], STD[:C], out_dtype=F16, layout=NHWC, stream=stream,
                                       workspace=wss[g % 2], overlap_previous=True)
    stream.synchronize()
    for g, (batches, host) in enumerate(groups):
        _check(batches, host, F16, NHWC, "chain %d" % g)
    assert not any(bool(torch.any(w)) for w in wss)
    assert trfn.tr_device_status() == 0


def test_empty_and_rejected_calls():
    import torch
    N, H, W, C = 4, 32, 32, 3
    batches, _ = _make(2, N, H, W, C, F16, NHWC, 9)
    trfn.tr_fused_norm_batches([], MEAN[:C], STD[:C], shape=(N, H, W, C))           # K = 0: nothing to do
    a = batches[0]
    with pytest.raises(trfn.TrError):
        trfn.tr_fused_norm_batches([a, (batches[1][0], a[1], None)], MEAN[:C], STD[:C])   # two batches, one output
    with pytest.raises(trfn.TrError):
        trfn.tr_fused_norm_batches([a] * (17), MEAN[:C], STD[:C])                        # more than TR_MAX_BATCHES
    torch.cuda.synchronize()

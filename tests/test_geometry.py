"""The tiled kernel's launch geometry (tr_fused_norm_geometry) for the shapes
whose planning the measurements rest on: band heights, stages, CTAs per SM
and grid as the planner chooses them on a GB300 (152 SMs, 228 KB of shared
memory per SM).  The values are the device's: other GPUs skip."""
import pytest

import image_preprocessing_gb300 as trfn

pytestmark = pytest.mark.gpu

F16, F32 = trfn.OUT_F16, trfn.OUT_F32
NHWC, NCHW, NHWC4 = trfn.LAYOUT_NHWC, trfn.LAYOUT_NCHW, trfn.LAYOUT_NHWC4


@pytest.fixture(autouse=True)
def _gb300():
    import torch
    p = torch.cuda.get_device_properties(0)
    if p.multi_processor_count != 152:
        pytest.skip("geometry values are those of a 152-SM GB300")
    trfn.tr_tune_tiled(0, 0, 0, 0)


CASES = [
    # (N, H, W, C, dtype, layout, overlap) -> expected subset
    ((256, 224, 224, 3, F16, NHWC, False), dict(rows=16, stages=3, ctas_per_sm=3, grid=448, odd_form=0)),
    ((256, 224, 224, 3, F16, NHWC, True), dict(rows=16, stages=3, ctas_per_sm=3, grid=448, odd_form=0)),
    ((256, 224, 224, 3, F32, NHWC, False), dict(rows=8, stages=4, ctas_per_sm=3, odd_form=0)),
    # 32 KB bands fit two CTAs: lowered to three (3-stage plans)
    ((256, 256, 256, 3, F16, NHWC, False), dict(rows=14, stages=3, ctas_per_sm=3)),
    ((64, 512, 512, 3, F16, NHWC, False), dict(rows=7, stages=3, ctas_per_sm=3)),
    ((256, 224, 224, 3, F16, NHWC4, False), dict(rows=13, stages=3, ctas_per_sm=3)),
    # 4-stage plans keep two CTAs when waiting, take three when overlapping
    ((256, 224, 224, 1, F32, NHWC, False), dict(rows=32, stages=4, ctas_per_sm=2)),
    ((256, 224, 224, 1, F32, NHWC, True), dict(rows=28, stages=4, ctas_per_sm=3)),
    # one channel: NCHW is planned as NHWC
    ((256, 224, 224, 1, F32, NCHW, True), dict(rows=28, stages=4, ctas_per_sm=3)),
    # odd-row form streaming many bands: two stages, four CTAs, strides >= 84 % full
    ((256, 299, 299, 3, F16, NHWC, True), dict(rows=10, stages=2, ctas_per_sm=4, odd_form=1)),
    ((256, 299, 299, 3, F32, NHWC, False), dict(rows=5, odd_form=1)),
    # odd-row NCHW (plane-aligned windows): compiled for four CTAs per SM
    ((256, 299, 299, 3, F16, NCHW, True), dict(rows=10, stages=2, ctas_per_sm=4, odd_form=1)),
    ((256, 299, 299, 3, F32, NCHW, True), dict(rows=5, stages=4, ctas_per_sm=4, odd_form=1)),
    # odd-row form with few bands a CTA: the aligned planning, even band heights
    ((256, 75, 75, 3, F16, NHWC, False), dict(rows=38, stages=3, odd_form=1)),
]


@pytest.mark.parametrize("args,expect", CASES)
def test_planned_geometry(args, expect):
    N, H, W, C, dt, lay, ov = args
    g = trfn.tr_fused_norm_geometry(N, H, W, C, out_dtype=dt, layout=lay, overlap_previous=ov)
    got = {k: g[k] for k in expect}
    assert got == expect, (args, g)


def test_geometry_follows_alignment_and_knobs():
    # an output pointer 2 bytes off 16: the odd-row form
    g = trfn.tr_fused_norm_geometry(256, 224, 224, 3, dst=0x200000002)
    assert g["odd_form"] == 1
    # tr_tune_tiled's band height and stage count are what the launch takes
    try:
        trfn.tr_tune_tiled(8 * 672, 4, 0, 0)
        g = trfn.tr_fused_norm_geometry(256, 224, 224, 3)
        assert (g["rows"], g["stages"]) == (8, 4)
        trfn.tr_tune_tiled(0, 0, 2, 0)
        g = trfn.tr_fused_norm_geometry(256, 224, 224, 3)
        assert g["ctas_per_sm"] == 2 and g["grid"] <= 2 * 152
    finally:
        trfn.tr_tune_tiled(0, 0, 0, 0)
    with pytest.raises(trfn.TrError):
        trfn.tr_fused_norm_geometry(4, 32, 32, 3, src=0x100000001)   # unaligned source: no tiled kernel

"""tr_fused_norm_sampled: records drawn on the GPU and the fused step in one
call.  The records it writes equal the oracle's per-image sampler bit for
bit (counter block offset + 24n per image), and its output equals the
oracle's fused normalisation under those records, for the tiled kernel
(static and dynamic schedules, every layout) and for the per-element kernel
(small batches), and bit for bit the separate calls (GPU sampler, then the
kernel)."""
import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import synth
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

MEAN = np.array(synth.IMAGENET_MEAN + (0.5,), np.float32)
STD = np.array(synth.IMAGENET_STD + (0.25,), np.float32)


def _bits(t, dt):
    import torch
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if dt == trfn.OUT_F16 else t.numpy()


def _run(src, seed, offset, dt, layout, variant=trfn.VARIANT_AUTO, ws=False, **kw):
    import torch
    N, H, W, C = src.shape
    d_src = torch.from_numpy(src).cuda()
    tdt = torch.float16 if dt == trfn.OUT_F16 else torch.float32
    dst = torch.full(trfn.out_shape(N, H, W, C, layout), 3.0, dtype=tdt, device="cuda")
    rec = torch.full((N, 5), -7, dtype=torch.int32, device="cuda")
    work = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") if ws else None
    nxt = trfn.tr_fused_norm_sampled(d_src, dst, MEAN[:C], STD[:C], seed, offset, rec, out_dtype=dt, layout=layout,
                                     variant=variant, workspace=work, **kw)
    torch.cuda.synchronize()
    if work is not None:
        assert int(work.count_nonzero()) == 0
    return _bits(dst, dt), rec.cpu().numpy(), nxt


CASES = [
    # (N, H, W, C, dtype, layout, variant, workspace, sampling)
    (256, 224, 224, 3, trfn.OUT_F16, trfn.LAYOUT_NHWC, trfn.VARIANT_AUTO, True, {}),
    (64, 224, 224, 3, trfn.OUT_F16, trfn.LAYOUT_NHWC, trfn.VARIANT_TILED, False, dict(erase_p=1.0)),
    (33, 64, 96, 3, trfn.OUT_F32, trfn.LAYOUT_NCHW, trfn.VARIANT_TILED, True, dict(flip=False)),
    (17, 40, 48, 1, trfn.OUT_F16, trfn.LAYOUT_NHWC4, trfn.VARIANT_TILED, True, dict(flip_p=0.25, erase_p=0.7)),
    (9, 37, 32, 4, trfn.OUT_F32, trfn.LAYOUT_NHWC, trfn.VARIANT_TILED, False, dict(erase=False)),
    (5, 31, 16, 2, trfn.OUT_F16, trfn.LAYOUT_NHWC, trfn.VARIANT_TILED, True, dict(scale=(0.1, 0.5), ratio=(0.5, 2))),
    (16, 32, 32, 3, trfn.OUT_F32, trfn.LAYOUT_NHWC, trfn.VARIANT_AUTO, False, {}),          # small: per-element
    (7, 11, 13, 3, trfn.OUT_F16, trfn.LAYOUT_NHWC, trfn.VARIANT_GENERIC, False, dict(erase_p=1.0)),
]


@pytest.mark.parametrize("case", CASES)
def test_records_and_output_match_the_oracle(case):
    N, H, W, C, dt, layout, variant, ws, kw = case
    src = synth.pixels_uniform(40 + N, N, H, W, C)
    seed, offset = 1000 + N, 24 * 7 + N
    out, rec, nxt = _run(src, seed, offset, dt, layout, variant, ws, **kw)
    ref_rec, ref_nxt = oracle.sample_aug_params_blocked(seed, offset, N, H, W, **kw)
    assert nxt == ref_nxt == offset + 24 * N
    assert np.array_equal(rec, ref_rec)
    ref = oracle.fused_norm(src, MEAN[:C], STD[:C], ref_rec, out_dtype=dt, layout=layout)
    assert_parity(out, ref, dt, "sampled %s" % (case[:7],))


@pytest.mark.parametrize("flags", [0, 32])
def test_same_bits_as_sampler_then_kernel(flags):
    """One call against two (the record sampler, then the kernel reading
    them): identical records and output."""
    import torch
    N, H, W, C = 128, 224, 224, 3
    src = synth.pixels_uniform(77, N, H, W, C)
    d_src = torch.from_numpy(src).cuda()
    try:
        trfn.tr_tune_tiled(0, 0, 0, flags)
        one, rec1, _ = _run(src, 5, 0, trfn.OUT_F16, trfn.LAYOUT_NHWC, ws=True)
        rec = torch.empty((N, 5), dtype=torch.int32, device="cuda")
        trfn.tr_sample_aug_params_device(5, 0, N, H, W, rec)
        dst = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
        trfn.tr_fused_norm(d_src, dst, MEAN[:C], STD[:C], rec, out_dtype=trfn.OUT_F16)
        torch.cuda.synchronize()
    finally:
        trfn.tr_tune_tiled(0, 0, 0, 0)
    assert np.array_equal(rec1, rec.cpu().numpy())
    assert np.array_equal(one, _bits(dst, trfn.OUT_F16))


def test_bad_arguments_launch_nothing():
    import torch
    N, H, W, C = 4, 32, 32, 3
    src = torch.zeros((N, H, W, C), dtype=torch.uint8, device="cuda")
    dst = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
    rec = torch.empty((N, 5), dtype=torch.int32, device="cuda")
    before = trfn.tr_launch_count()
    with pytest.raises(trfn.TrError):
        trfn.tr_fused_norm_sampled(src, dst, MEAN[:C], STD[:C], 0, 0, rec, ratio=(0.0, 1.0))
    with pytest.raises(trfn.TrError):
        trfn.tr_fused_norm_sampled(src, dst, MEAN[:C], STD[:C], 0, 0, rec, scale=(0.5, 0.1))
    # records placed over the output
    with pytest.raises(trfn.TrError):
        trfn.tr_fused_norm_sampled(src, dst, MEAN[:C], STD[:C], 0, 0,
                                   dst.view(-1).view(torch.int32)[:N * 5].view(N, 5))
    assert trfn.tr_launch_count() == before

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


@pytest.mark.parametrize("shape,dt,layout", [((64, 224, 224, 3), trfn.OUT_F16, trfn.LAYOUT_NHWC),
                                             ((32, 224, 224, 3), trfn.OUT_F32, trfn.LAYOUT_NCHW),
                                             ((24, 299, 299, 3), trfn.OUT_F16, trfn.LAYOUT_NHWC)])   # odd-row form
@pytest.mark.parametrize("first_records", ["made_in_kernel", "first_S_made_in_kernel", "read_from_sampler"])
def test_overlapped_sampled_launches(shape, dt, layout, first_records):
    """tr_fused_norm_sampled_ex with TR_LAUNCH_OVERLAP_PREVIOUS: a large
    launch, then consecutive sampled batches with their own source, output
    and records, workspaces alternating.  Each sampler writes while the
    kernel before it drains, each fused kernel requests its first bands
    before its sampler is done; by default its consumer warps make the
    records of a CTA's first 2S bands (S where there are fewer than 2S
    consumer warps: 4-stage plans) with the sampler's steps (tr_tune_tiled
    flags bit 25 keeps S, bit 21 reads them all from the sampler's output
    instead).  Records and outputs equal the oracle's every way."""
    import torch
    if first_records == "read_from_sampler":
        trfn.tr_tune_tiled(flags=1 << 21)
    elif first_records == "first_S_made_in_kernel":
        trfn.tr_tune_tiled(flags=1 << 25)
    try:
        _overlapped_sampled_chain(shape, dt, layout)
    finally:
        trfn.tr_tune_tiled()


def _overlapped_sampled_chain(shape, dt, layout):
    import torch
    N, H, W, C = shape
    K = 6
    tdt = torch.float16 if dt == trfn.OUT_F16 else torch.float32
    srcs = [synth.pixels_uniform(900 + k, N, H, W, C) for k in range(K)]
    d_src = [torch.from_numpy(x).cuda() for x in srcs]
    dsts = [torch.full(trfn.out_shape(N, H, W, C, layout), 3.0, dtype=tdt, device="cuda") for _ in range(K)]
    recs = [torch.full((N, 5), -7, dtype=torch.int32, device="cuda") for _ in range(K)]
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    big = synth.pixels_uniform(950, 256, 224, 224, 3)
    d_big = torch.from_numpy(big).cuda()
    d_big_out = torch.empty((256, 224, 224, 3), dtype=torch.float16, device="cuda")
    st = torch.cuda.Stream()
    for rep in range(2):
        for d in dsts:
            d.fill_(3.0)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            trfn.tr_fused_norm(d_big, d_big_out, MEAN[:3], STD[:3], None, stream=st, workspace=wss[1])
            for k in range(K):
                trfn.tr_fused_norm_sampled(d_src[k], dsts[k], MEAN[:C], STD[:C], 70 + k, 24 * k, recs[k],
                                           out_dtype=dt, layout=layout, stream=st, workspace=wss[k % 2],
                                           overlap_previous=True)
        torch.cuda.synchronize()
        for k in range(K):
            ref_rec, _ = oracle.sample_aug_params_blocked(70 + k, 24 * k, N, H, W)
            assert np.array_equal(recs[k].cpu().numpy(), ref_rec)
            ref = oracle.fused_norm(srcs[k], MEAN[:C], STD[:C], ref_rec, out_dtype=dt, layout=layout)
            assert_parity(_bits(dsts[k], dt), ref, dt, "overlapped sampled batch %d" % k)
        for ws in wss:
            assert int(ws.count_nonzero()) == 0
    ref_big = oracle.fused_norm(big, MEAN[:3], STD[:3], None, out_dtype=trfn.OUT_F16)
    assert_parity(_bits(d_big_out, trfn.OUT_F16), ref_big, trfn.OUT_F16, "launch before the chain")
    assert trfn.tr_device_status() == 0

"""Seeded random cases, each compared with the oracle element by element with
guard bytes around the output: shapes with ragged edges (odd rows, one-row
and one-pixel images, rows shorter than a group), every channel count,
output type and layout, offset source and output pointers, the three kernel
choices, tile geometries (band height, stages, CTAs per SM) and
tr_tune_tiled flags, all drawn from one seed.  The tiled cases run once more
through the checked build (libtrfn_bounds.so), which tests every range the
tiled kernel copies, loads or stores and must leave its status word clear;
that test comes first, so a range the planner got wrong shows up there as a
status bit rather than as an access outside a buffer.
(Integration tests as layers of determinism and correctness: "(25)
integration tests" article, §一-§二.)"""
import ctypes

import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import _native, synth
from parity_util import assert_parity, check_case

pytestmark = pytest.mark.gpu

F32, F16 = trfn.OUT_F32, trfn.OUT_F16
NHWC, NCHW, NHWC4 = trfn.LAYOUT_NHWC, trfn.LAYOUT_NCHW, trfn.LAYOUT_NHWC4
AUTO, TILED, GENERIC = trfn.VARIANT_AUTO, trfn.VARIANT_TILED, trfn.VARIANT_GENERIC

SEED = 20261202
CASES = 300
# tr_tune_tiled flag bits that change how the kernels work, not what they
# compute (bit 6, the bounded-wait test hook, is left out)
FLAG_BITS = (0, 1, 2, 3, 4, 5, 7, 10, 11, 16, 17, 18, 19, 20, 23)


def _case(i):
    rng = np.random.default_rng(SEED + i)
    N = int(rng.integers(1, 9))
    H = int(rng.integers(1, 72))
    W = int(rng.integers(1, 140))
    C = int(rng.integers(1, 5))
    dt = F16 if rng.random() < 0.5 else F32
    layout = (NHWC, NCHW, NHWC4)[int(rng.integers(0, 3))]
    variant = (AUTO, TILED, GENERIC)[int(rng.integers(0, 3))]
    ob = 2 if dt == F16 else 4
    flags = 0
    for b in rng.choice(FLAG_BITS, size=int(rng.integers(0, 4)), replace=False):
        flags |= 1 << int(b)
    if rng.random() < 0.3:
        flags |= int(rng.integers(0, 16)) << 12   # erased-span threshold
    return dict(
        src=synth.pixels_uniform(SEED + i, N, H, W, C),
        aug=synth.random_records(SEED + i, N, H, W, allow_outside=True) if rng.random() < 0.8 else None,
        mean=rng.uniform(0.0, 1.0, C).astype(np.float32),
        # |v| <= 5: the binary32 bar (2e-6 absolute) is then above 3 ulps
        std=rng.uniform(0.2, 0.6, C).astype(np.float32),
        dt=dt, layout=layout, variant=variant,
        src_offset=0 if variant == TILED else int(rng.choice([0, 0, 1, 3, 16])),
        dst_offset=int(rng.choice([0, 0, ob, 3 * ob, 16])),
        tune=(int(rng.choice([0, 0, 16, 48, 200, 1000, 4096])), int(rng.choice([0, 0, 2, 3, 4, 8])),
              int(rng.choice([0, 0, 1, 2, 3])), flags),
        workspace=bool(rng.random() < 0.5))


def _checked_status(L):
    v = ctypes.c_int(0)
    assert L.tr_device_status(ctypes.byref(v), 1) == 0
    return v.value


def test_random_tiled_cases_pass_the_checked_build():
    import torch
    L = _native.checked_lib()
    _checked_status(L)
    guard = 64
    for i in range(CASES):
        c = _case(i)
        src = c["src"]
        N, H, W, C = src.shape
        shape = trfn.out_shape(N, H, W, C, c["layout"])
        ob = 2 if c["dt"] == F16 else 4
        nbytes = int(np.prod(shape)) * ob
        s_buf = torch.from_numpy(np.ascontiguousarray(src).reshape(-1)).cuda()
        d_buf = torch.full((nbytes + 2 * guard + c["dst_offset"],), 0xAB, dtype=torch.uint8, device="cuda")
        a = torch.from_numpy(c["aug"]).cuda() if c["aug"] is not None else None
        ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") if c["workspace"] else None
        assert L.tr_tune_tiled(*c["tune"]) == 0
        try:
            rc = L.tr_fused_norm_ws(s_buf.data_ptr(), d_buf.data_ptr() + guard + c["dst_offset"], N, H, W, C,
                                    _native.float_array(c["mean"]), _native.float_array(c["std"]),
                                    a.data_ptr() if a is not None else None, c["dt"], c["layout"], None, TILED,
                                    ws.data_ptr() if ws is not None else None)
            assert rc == 0, L.tr_last_error_message()
            torch.cuda.synchronize()
        finally:
            L.tr_tune_tiled(0, 0, 0, 0)
        host = d_buf.cpu().numpy()
        body = host[guard + c["dst_offset"]:guard + c["dst_offset"] + nbytes]
        got = body.view(np.uint16 if c["dt"] == F16 else np.float32).reshape(shape)
        ref = oracle.fused_norm(src, c["mean"], c["std"], c["aug"], out_dtype=c["dt"], layout=c["layout"])
        assert_parity(got, ref, c["dt"], "checked build, case %d" % i)
        rest = np.concatenate([host[:guard + c["dst_offset"]], host[guard + c["dst_offset"] + nbytes:]])
        assert np.all(rest == 0xAB), "case %d wrote outside its output" % i
        assert _checked_status(L) == 0, "case %d: a bounds check failed" % i


@pytest.mark.parametrize("i", range(CASES))
def test_random_case_matches_the_oracle(i):
    import torch
    c = _case(i)
    ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") if c["workspace"] else None
    trfn.tr_tune_tiled(*c["tune"])
    try:
        check_case(c["src"], c["mean"], c["std"], c["aug"], c["dt"], c["layout"], variant=c["variant"],
                   src_offset=c["src_offset"], dst_offset=c["dst_offset"], workspace=ws)
    finally:
        trfn.tr_tune_tiled()
    if ws is not None:
        assert int(ws.count_nonzero()) == 0, "the scheduling workspace was not returned to zero"
    assert trfn.tr_device_status() == 0


SAMPLED_CASES = 32
# tr_tune_tiled flag bits of the one-call sampled form: first records read
# from the sampler (21), made by the producer warp (22), only the first S
# made (25)
SAMPLED_BITS = (21, 22, 25)


@pytest.mark.parametrize("i", range(SAMPLED_CASES))
def test_random_overlapped_sampled_chains_match_the_oracle(i):
    """Chains of three one-call sampled launches (records drawn on the GPU
    in the same call), each overlapping the one before, on random shapes
    (rows mostly 16-byte multiples, where the fused kernel makes a CTA's
    first records itself), stage counts and flags: every batch's records
    equal the oracle's sampler bit for bit and its output the oracle's."""
    import torch
    rng = np.random.default_rng(SEED + 7000 + i)
    C = int(rng.integers(1, 5))
    W = int(rng.integers(1, 12)) * (16 // np.gcd(16, C)) if rng.random() < 0.8 else int(rng.integers(1, 140))
    H = int(rng.integers(1, 90))
    N = int(rng.integers(1, 70))
    dt = F16 if rng.random() < 0.5 else F32
    layout = (NHWC, NCHW, NHWC4)[int(rng.integers(0, 3))]
    flags = 0
    for b in rng.choice(SAMPLED_BITS, size=int(rng.integers(0, 2)), replace=False):
        flags |= 1 << int(b)
    stages = int(rng.choice([0, 0, 2, 3, 4]))
    mean = rng.uniform(0.0, 1.0, C).astype(np.float32)
    std = rng.uniform(0.2, 0.6, C).astype(np.float32)
    K = 3
    srcs = [synth.pixels_uniform(SEED + 100 * i + k, N, H, W, C) for k in range(K)]
    tdt = torch.float16 if dt == F16 else torch.float32
    dsts = [torch.full(trfn.out_shape(N, H, W, C, layout), 3.0, dtype=tdt, device="cuda") for _ in range(K)]
    recs = [torch.full((N, 5), -7, dtype=torch.int32, device="cuda") for _ in range(K)]
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    d_src = [torch.from_numpy(x).cuda() for x in srcs]
    st = torch.cuda.Stream()
    trfn.tr_tune_tiled(0, stages, 0, flags)
    try:
        with torch.cuda.stream(st):
            for k in range(K):
                trfn.tr_fused_norm_sampled(d_src[k], dsts[k], mean, std, 900 + i, 24 * N * k, recs[k],
                                           out_dtype=dt, layout=layout, stream=st, workspace=wss[k % 2],
                                           overlap_previous=True)
        torch.cuda.synchronize()
    finally:
        trfn.tr_tune_tiled()
    for k in range(K):
        ref_rec, _ = oracle.sample_aug_params_blocked(900 + i, 24 * N * k, N, H, W)
        assert np.array_equal(recs[k].cpu().numpy(), ref_rec), "case %d batch %d records" % (i, k)
        got = dsts[k].cpu()
        got = got.view(torch.int16).numpy().view(np.uint16) if dt == F16 else got.numpy()
        ref = oracle.fused_norm(srcs[k], mean, std, ref_rec, out_dtype=dt, layout=layout)
        assert_parity(got, ref, dt, "case %d batch %d" % (i, k))
    for ws in wss:
        assert int(ws.count_nonzero()) == 0
    assert trfn.tr_device_status() == 0


BATCHES_CASES = 24


@pytest.mark.parametrize("i", range(BATCHES_CASES))
def test_random_batches_per_launch_match_the_oracle(i):
    """tr_fused_norm_batches on random K (1..16), shapes (odd rows
    included), types, layouts, records and schedules, waiting or overlapping
    the launch before: every batch against the oracle."""
    import torch
    rng = np.random.default_rng(SEED + 9000 + i)
    K = int(rng.integers(1, 17))
    C = int(rng.integers(1, 5))
    N, H, W = int(rng.integers(1, 40)), int(rng.integers(1, 60)), int(rng.integers(1, 100))
    dt = F16 if rng.random() < 0.5 else F32
    layout = (NHWC, NCHW, NHWC4)[int(rng.integers(0, 3))]
    mean = rng.uniform(0.0, 1.0, C).astype(np.float32)
    std = rng.uniform(0.2, 0.6, C).astype(np.float32)
    tdt = torch.float16 if dt == F16 else torch.float32
    host, batches = [], []
    for k in range(K):
        src = synth.pixels_uniform(SEED + 50 * i + k, N, H, W, C)
        aug = synth.random_records(SEED + 50 * i + k, N, H, W, allow_outside=True) if rng.random() < 0.8 else None
        host.append((src, aug))
        batches.append((torch.from_numpy(src).cuda(),
                        torch.full(trfn.out_shape(N, H, W, C, layout), 3.0, dtype=tdt, device="cuda"),
                        torch.from_numpy(aug).cuda() if aug is not None else None))
    ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") if rng.random() < 0.5 else None
    trfn.tr_fused_norm_batches(batches, mean, std, out_dtype=dt, layout=layout, workspace=ws,
                               overlap_previous=bool(ws is not None and rng.random() < 0.5))
    torch.cuda.synchronize()
    for k, ((src, aug), (_, dst, _)) in enumerate(zip(host, batches)):
        got = dst.cpu()
        got = got.view(torch.int16).numpy().view(np.uint16) if dt == F16 else got.numpy()
        ref = oracle.fused_norm(src, mean, std, aug, out_dtype=dt, layout=layout)
        assert_parity(got, ref, dt, "case %d batch %d" % (i, k))
    if ws is not None:
        assert int(ws.count_nonzero()) == 0
    assert trfn.tr_device_status() == 0


CROP_CASES = 32


@pytest.mark.parametrize("i", range(CROP_CASES))
def test_random_crop_windows_match_the_oracle(i):
    """tr_fused_norm_crop on random windows of random strided sources: row
    and image strides padded by multiples of 16 bytes half the time (the
    tensor-copy path where the shape allows it) and by any count otherwise,
    origins anywhere (clamped into the source), random records, types,
    layouts, kernel choices and schedules: against the oracle's crop form."""
    import torch
    rng = np.random.default_rng(SEED + 11000 + i)
    C = int(rng.integers(1, 5))
    N = int(rng.integers(1, 9))
    H, W = int(rng.integers(1, 48)), int(rng.integers(1, 80))
    SH, SW = H + int(rng.integers(0, 24)), W + int(rng.integers(0, 40))
    if rng.random() < 0.5:
        SW = -(-SW * C // 16) * 16 // C if (-(-SW * C // 16) * 16) % C == 0 else SW
        row_pad, image_pad = 16 * int(rng.integers(0, 3)), 16 * int(rng.integers(0, 3))
    else:
        row_pad, image_pad = int(rng.integers(0, 20)), int(rng.integers(0, 40))
    dt = F16 if rng.random() < 0.5 else F32
    layout = (NHWC, NCHW, NHWC4)[int(rng.integers(0, 3))]
    variant = (AUTO, GENERIC)[int(rng.integers(0, 2))]
    mean = rng.uniform(0.0, 1.0, C).astype(np.float32)
    std = rng.uniform(0.2, 0.6, C).astype(np.float32)
    src = synth.pixels_uniform(SEED + i, N, SH, SW, C)
    row_stride = SW * C + row_pad
    image_stride = SH * row_stride + image_pad
    buf = np.full(N * image_stride, 0xEE, np.uint8)
    for n in range(N):
        for y in range(SH):
            o = n * image_stride + y * row_stride
            buf[o:o + SW * C] = src[n, y].reshape(-1)
    crop = np.stack([rng.integers(-4, SH - H + 5, N), rng.integers(-4, SW - W + 5, N)], axis=1).astype(np.int32)
    clamped = np.stack([np.clip(crop[:, 0], 0, SH - H), np.clip(crop[:, 1], 0, SW - W)], axis=1).astype(np.int32)
    aug = synth.random_records(SEED + 11000 + i, N, H, W, allow_outside=True) if rng.random() < 0.8 else None
    ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") if rng.random() < 0.5 else None
    d_buf = torch.zeros(buf.size + 64, dtype=torch.uint8, device="cuda")
    d_buf[:buf.size].copy_(torch.from_numpy(buf))
    tdt = torch.float16 if dt == F16 else torch.float32
    out = torch.empty(trfn.out_shape(N, H, W, C, layout), dtype=tdt, device="cuda")
    trfn.tr_fused_norm_crop(d_buf.data_ptr(), SH, SW, row_stride, image_stride, out, N, H, W, C, mean, std,
                            crop=torch.from_numpy(crop).cuda(),
                            aug=torch.from_numpy(aug).cuda() if aug is not None else None,
                            out_dtype=dt, layout=layout, variant=variant, workspace=ws)
    torch.cuda.synchronize()
    got = out.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if dt == F16 else got.numpy()
    ref = oracle.fused_norm_crop(buf, image_stride, row_stride, SH, SW, N, H, W, C, mean, std, clamped, aug,
                                 out_dtype=dt, layout=layout)
    assert_parity(got, ref, dt, "case %d" % i)
    if ws is not None:
        assert int(ws.count_nonzero()) == 0
    assert trfn.tr_device_status() == 0

"""The checked build (libtrfn_bounds.so, compiled with -DTRFN_BOUNDS=1): the
tiled kernel tests every shared-memory and global range it copies, loads or
stores against its buffer, and the 16-byte rules of bulk copies, before the
access; a failed check sets bit 1 of its device status word and skips the
access.  Here the tiled kernel's forms -- aligned and odd rows, every layout
and type, crop windows, the dynamic schedule, several batches per launch,
the realigned odd-row stores -- run under it on small shapes with ragged
edges, and must leave the status word clear and match the oracle.  This is
the stand-in for a memory checker, which is not available on this GPU pool.
(Integration tests as layers of determinism and correctness: "(25)
integration tests" article, §一-§二.)"""
import ctypes

import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import _native, synth
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

F32, F16 = trfn.OUT_F32, trfn.OUT_F16
NHWC, NCHW, NHWC4 = trfn.LAYOUT_NHWC, trfn.LAYOUT_NCHW, trfn.LAYOUT_NHWC4
TILED = trfn.VARIANT_TILED
STREAMS = 1 << 17   # tr_tune_tiled flags: realigned odd-row stores at any size


def _status(L):
    v = ctypes.c_int(0)
    assert L.tr_device_status(ctypes.byref(v), 1) == 0
    return v.value


def _consts(C):
    mean = np.array([0.485, 0.456, 0.406, 0.5], np.float32)[:C]
    std = np.array([0.229, 0.224, 0.225, 0.25], np.float32)[:C]
    return mean, std


def _run(L, src, aug, dt, layout, ws=None, dst_offset=0):
    import torch
    N, H, W, C = src.shape
    mean, std = _consts(C)
    shape = trfn.out_shape(N, H, W, C, layout)
    ob = 2 if dt == F16 else 4
    nbytes = int(np.prod(shape)) * ob
    guard = 64
    s_buf = torch.from_numpy(np.ascontiguousarray(src).reshape(-1)).cuda()
    d_buf = torch.full((nbytes + 2 * guard + dst_offset,), 0xAB, dtype=torch.uint8, device="cuda")
    a = torch.from_numpy(aug).cuda() if aug is not None else None
    rc = L.tr_fused_norm_ws(s_buf.data_ptr(), d_buf.data_ptr() + guard + dst_offset, N, H, W, C,
                            _native.float_array(mean), _native.float_array(std),
                            a.data_ptr() if a is not None else None, dt, layout, None, TILED,
                            ws.data_ptr() if ws is not None else None)
    assert rc == 0, L.tr_last_error_message()
    torch.cuda.synchronize()
    host = d_buf.cpu().numpy()
    body = host[guard + dst_offset:guard + dst_offset + nbytes].view(np.uint16 if dt == F16 else np.float32)
    guards = np.concatenate([host[:guard + dst_offset], host[guard + dst_offset + nbytes:]])
    assert np.all(guards == 0xAB), "bytes outside the output were written"
    ref = oracle.fused_norm(src, mean, std, aug, out_dtype=dt, layout=layout)
    return body.reshape(shape), ref


SHAPES = [(3, 37, 64, 3), (2, 70, 128, 3), (4, 20, 40, 2), (2, 13, 12, 4), (5, 64, 32, 1),   # aligned rows
          (3, 37, 61, 3), (2, 29, 227, 3), (4, 28, 28, 1), (2, 13, 99, 2), (2, 11, 75, 4),   # odd rows
          (1, 45, 299, 3),
          # odd rows whose planes' 16-byte frames stay 0 or 1 element apart
          # (H*W mod 8 of 0 or 1): binary16 NCHW takes the plane-aligned windows
          (2, 8, 75, 3), (2, 9, 89, 2), (1, 45, 301, 3)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dt", [F32, F16])
@pytest.mark.parametrize("layout", [NHWC, NCHW, NHWC4])
def test_tiled_forms_pass_the_checks(shape, dt, layout):
    import torch
    L = _native.checked_lib()
    _status(L)
    N, H, W, C = shape
    src = synth.pixels_uniform(N * 1000 + H + W, N, H, W, C)
    aug = synth.random_records(H + W, N, H, W, allow_outside=True)
    ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda")
    for kw in ({}, {"ws": ws}, {"dst_offset": 2 * (1 + (dt == F32))}):
        got, ref = _run(L, src, aug, dt, layout, **kw)
        assert_parity(got, ref, dt, "%s %s" % (shape, kw.keys()))
    assert L.tr_tune_tiled(0, 0, 0, STREAMS) == 0
    try:
        for kw in ({}, {"dst_offset": 2 * (1 + (dt == F32))}):
            got, ref = _run(L, src, aug, dt, layout, **kw)
            assert_parity(got, ref, dt, "realigned stores %s %s" % (shape, kw.keys()))
    finally:
        L.tr_tune_tiled(0, 0, 0, 0)
    assert _status(L) == 0, "a bounds check failed (status word %#x)" % _status(L)


@pytest.mark.parametrize("dt", [F32, F16])
def test_crop_windows_pass_the_checks(dt):
    import torch
    L = _native.checked_lib()
    _status(L)
    N, C, S, H, W = 6, 3, 80, 45, 64   # TMA windows need W*C and NCHW rows in 16-byte units
    src = synth.pixels_uniform(77, N, S, S, C)
    crop = np.stack([np.arange(N) * 7 % (S - H + 1), np.arange(N) * 5 % (S - W + 1)], axis=1).astype(np.int32)
    aug = synth.random_records(78, N, H, W, allow_outside=True)
    mean, std = _consts(C)
    for layout in (NHWC, NCHW, NHWC4):
        shape = trfn.out_shape(N, H, W, C, layout)
        dst = torch.zeros(shape, dtype=torch.float16 if dt == F16 else torch.float32, device="cuda")
        d_src = torch.from_numpy(src).cuda()
        d_crop = torch.from_numpy(crop).cuda()
        d_aug = torch.from_numpy(aug).cuda()
        rc = L.tr_fused_norm_crop(d_src.data_ptr(), S, S, S * C, S * S * C, d_crop.data_ptr(), dst.data_ptr(), N, H,
                                  W, C, _native.float_array(mean), _native.float_array(std), d_aug.data_ptr(), dt,
                                  layout, None, TILED, None)
        assert rc == 0, L.tr_last_error_message()
        torch.cuda.synchronize()
        got = dst.cpu()
        got = got.view(torch.int16).numpy().view(np.uint16) if dt == F16 else got.numpy()
        ref = oracle.fused_norm_crop(src.reshape(-1), S * S * C, S * C, S, S, N, H, W, C, mean, std, crop, aug, dt,
                                     layout)
        assert_parity(got, ref, dt, "crop layout %d" % layout)
    assert _status(L) == 0


def test_several_batches_pass_the_checks():
    import torch
    L = _native.checked_lib()
    _status(L)
    for (N, H, W, C) in [(12, 37, 64, 3), (5, 29, 227, 3)]:   # K*N images reach the tiled kernel
        K = 4
        mean, std = _consts(C)
        srcs = [synth.pixels_uniform(300 + k, N, H, W, C) for k in range(K)]
        recs = [synth.random_records(400 + k, N, H, W, allow_outside=True) for k in range(K)]
        d_src = [torch.from_numpy(x).cuda() for x in srcs]
        d_aug = [torch.from_numpy(r).cuda() for r in recs]
        d_dst = [torch.zeros((N, H, W, C), dtype=torch.float16, device="cuda") for _ in range(K)]
        arr = (_native.Batch * K)(*[_native.Batch(d_src[k].data_ptr(), d_dst[k].data_ptr(), d_aug[k].data_ptr())
                                    for k in range(K)])
        rc = L.tr_fused_norm_batches(arr, K, N, H, W, C, _native.float_array(mean), _native.float_array(std), F16,
                                     NHWC, None, None, 0)
        assert rc == 0, L.tr_last_error_message()
        torch.cuda.synchronize()
        for k in range(K):
            ref = oracle.fused_norm(srcs[k], mean, std, recs[k], out_dtype=F16)
            assert_parity(d_dst[k].cpu().view(torch.int16).numpy().view(np.uint16), ref, F16, "batch %d" % k)
    assert _status(L) == 0

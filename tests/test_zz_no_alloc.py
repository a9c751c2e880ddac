"""tr_fused_norm_noalloc: the dynamically scheduled kernel for callers that
cannot allocate device memory (a fixed start-up memory plan, loader threads
that must not wait on cudaFree's device-wide synchronisation, plug-ins with
no access to the host's allocator).  Its scheduling scratch lives in the
library's module memory instead of a caller's buffer.

The test calls it through the C ABI twice in a row, on two different
batches, and compares each output with tr_fused_norm's within the parity
tolerances (binary16: 1 ulp, exact +0 for erased elements).  The file is
collected last so that a failure here leaves every other test run."""
import ctypes

import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import _native, synth

pytestmark = pytest.mark.gpu


def _f16_ulps(a, b):
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return np.abs(ordered(a) - ordered(b))


def test_noalloc_matches_tr_fused_norm_on_two_calls_in_a_row():
    import torch
    L = _native.lib()
    N, H, W, C = 64, 224, 224, 3
    mean = _native.float_array(synth.IMAGENET_MEAN)
    std = _native.float_array(synth.IMAGENET_STD)
    stream = torch.cuda.Stream()
    for call in range(2):
        src = torch.from_numpy(synth.pixels_uniform(700 + call, N, H, W, C)).cuda()
        recs, _ = oracle.sample_aug_params(800 + call, 0, N, H, W)
        aug = torch.from_numpy(recs).cuda()
        want = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
        got = torch.full((N, H, W, C), float("nan"), dtype=torch.float16, device="cuda")
        rc = L.tr_fused_norm(src.data_ptr(), want.data_ptr(), N, H, W, C, mean, std, aug.data_ptr(),
                             trfn.OUT_F16, trfn.LAYOUT_NHWC, stream.cuda_stream)
        assert rc == 0
        rc = L.tr_fused_norm_noalloc(src.data_ptr(), got.data_ptr(), N, H, W, C, mean, std, aug.data_ptr(),
                                     trfn.OUT_F16, trfn.LAYOUT_NHWC, stream.cuda_stream)
        assert rc == 0, L.tr_last_error_message()
        stream.synchronize()
        a = want.cpu().view(torch.int16).numpy().view(np.uint16)
        b = got.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.all(b[a == 0] == 0)
        assert int(_f16_ulps(a, b).max()) <= 1
    assert trfn.tr_device_status() == 0


def test_noalloc_rejects_bad_arguments_before_the_gpu():
    L = _native.lib()
    mean = _native.float_array(synth.IMAGENET_MEAN)
    std = _native.float_array(synth.IMAGENET_STD)
    assert L.tr_fused_norm_noalloc(None, None, 1, 4, 16, 3, mean, std, None, 1, 0, None) == 1
    assert L.tr_fused_norm_noalloc(0x1000, 0x100000, 1, 4, 16, 5, mean, std, None, 1, 0, None) == 2
    assert L.tr_fused_norm_noalloc(None, None, 0, 4, 16, 3, mean, std, None, 1, 0, None) == 0

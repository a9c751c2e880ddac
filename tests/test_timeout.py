"""Failure detection on the GPU without a fault: a launch whose first band
waits for bytes that never arrive (tr_tune_tiled's test hook) must end on
its own after the kernels' bounded waits run out, report it through the
device status word, and leave the context usable for the next launch."""
import time

import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import synth
from parity_util import assert_parity

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_survives():
    import torch
    N, H, W, C = 8, 32, 64, 3
    mean = np.array(synth.IMAGENET_MEAN, np.float32)
    std = np.array(synth.IMAGENET_STD, np.float32)
    src = synth.pixels_uniform(17, N, H, W, C)
    d_src = torch.from_numpy(src).cuda()
    out = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
    trfn.tr_device_status(clear=True)
    try:
        trfn.tr_tune_tiled(0, 0, 0, 64)
        t0 = time.perf_counter()
        trfn.tr_fused_norm(d_src, out, mean, std, None, out_dtype=trfn.OUT_F16, variant=trfn.VARIANT_TILED)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        trfn.tr_tune_tiled(0, 0, 0, 0)
    assert 0.5 < elapsed < 30.0          # the waits ran out (about a second each) and the kernel ended
    assert trfn.tr_device_status(clear=True) & 1
    assert trfn.tr_device_status() == 0
    # the context is still usable: a normal launch is correct
    trfn.tr_fused_norm(d_src, out, mean, std, None, out_dtype=trfn.OUT_F16)
    torch.cuda.synchronize()
    ref = oracle.fused_norm(src, mean, std, None, out_dtype=trfn.OUT_F16)
    assert_parity(out.cpu().view(torch.int16).numpy().view(np.uint16), ref, trfn.OUT_F16)
    assert trfn.tr_device_status() == 0

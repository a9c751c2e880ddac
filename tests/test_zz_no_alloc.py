"""tr_fused_norm_noalloc: the dynamically scheduled kernel for callers that
cannot allocate device memory (a fixed start-up memory plan, loader threads
that must not wait on cudaFree's device-wide synchronisation, plug-ins with
no access to the host's allocator).  Its scheduling scratch lives in the
library's module memory instead of a caller's buffer.

The tests call it through the C ABI twice in a row, on two different batches,
for three output forms (binary16 NHWC, binary32 NCHW, binary16 NHWC4), and
check each output element by element against the oracle (binary32 max-abs
2e-6, binary16 1 ulp, exact +0 where the oracle has +0) and bit for bit
against tr_fused_norm and tr_fused_norm_ws with a caller's workspace: all
three run the same kernel, and static and dynamic band schedules give the
same bytes.  The shapes are ones the planner sends to the tiled kernel, the
only one that reads the scratch; a small batch checks the per-element route,
which needs no scratch.  The file is collected last so that a failure here
leaves every other test run."""
import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import _native, synth
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

CASES = [
    (64, 224, 224, 3, trfn.OUT_F16, trfn.LAYOUT_NHWC),
    (32, 224, 224, 3, trfn.OUT_F32, trfn.LAYOUT_NCHW),
    (32, 160, 192, 3, trfn.OUT_F16, trfn.LAYOUT_NHWC4),
]


def _host(t, dt):
    import torch
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if dt == trfn.OUT_F16 else t.numpy()


def _run_three_ways(L, N, H, W, C, dt, layout, seed, stream, ws):
    """The same batch through tr_fused_norm, tr_fused_norm_ws (caller's
    workspace) and tr_fused_norm_noalloc; returns the three outputs, the
    pixels and the records."""
    import torch
    mean = _native.float_array(synth.IMAGENET_MEAN)
    std = _native.float_array(synth.IMAGENET_STD)
    pixels = synth.pixels_uniform(seed, N, H, W, C)
    recs, _ = oracle.sample_aug_params(seed + 100, 0, N, H, W)
    src = torch.from_numpy(pixels).cuda()
    aug = torch.from_numpy(recs).cuda()
    shape = trfn.out_shape(N, H, W, C, layout)
    tdt = torch.float16 if dt == trfn.OUT_F16 else torch.float32
    outs = [torch.full(shape, float("nan"), dtype=tdt, device="cuda") for _ in range(3)]
    args = (N, H, W, C, mean, std, aug.data_ptr(), dt, layout, stream.cuda_stream)
    assert L.tr_fused_norm(src.data_ptr(), outs[0].data_ptr(), *args) == 0
    assert L.tr_fused_norm_ws(src.data_ptr(), outs[1].data_ptr(), *args, trfn.VARIANT_AUTO, ws.data_ptr()) == 0
    rc = L.tr_fused_norm_noalloc(src.data_ptr(), outs[2].data_ptr(), *args)
    assert rc == 0, L.tr_last_error_message()
    stream.synchronize()
    return [_host(o, dt) for o in outs], pixels, recs


@pytest.mark.parametrize("case", CASES, ids=["f16_nhwc", "f32_nchw", "f16_nhwc4"])
def test_noalloc_matches_the_oracle_and_tr_fused_norm_on_two_calls_in_a_row(case):
    import torch
    L = _native.lib()
    N, H, W, C, dt, layout = case
    # the planner sends this shape to the tiled kernel, the one that reads the scratch
    assert trfn.tr_fused_norm_plan(0x1000, 0x1000000, N, H, W, C, dt, layout) == trfn.VARIANT_TILED
    stream = torch.cuda.Stream()
    ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda")
    mean = np.array(synth.IMAGENET_MEAN, np.float32)
    std = np.array(synth.IMAGENET_STD, np.float32)
    for call in range(2):
        (plain, with_ws, noalloc), pixels, recs = _run_three_ways(L, N, H, W, C, dt, layout, 700 + call,
                                                                  stream, ws)
        assert np.array_equal(noalloc.view(np.uint8), plain.view(np.uint8)), "call %d" % call
        assert np.array_equal(noalloc.view(np.uint8), with_ws.view(np.uint8)), "call %d" % call
        ref = oracle.fused_norm(pixels, mean, std, recs, out_dtype=dt, layout=layout)
        assert_parity(noalloc, ref, dt, "call %d" % call)
    assert not torch.any(ws), "the caller's workspace is zero again after its launch"
    assert trfn.tr_device_status() == 0


def test_noalloc_small_batch_takes_the_per_element_kernel():
    """16 x 32x32x3 is below the tiled kernel's threshold: the call runs the
    per-element kernel, which uses no scratch; output as the oracle's."""
    import torch
    L = _native.lib()
    N, H, W, C = 16, 32, 32, 3
    assert trfn.tr_fused_norm_plan(0x1000, 0x1000000, N, H, W, C, trfn.OUT_F32,
                                   trfn.LAYOUT_NHWC) == trfn.VARIANT_GENERIC
    stream = torch.cuda.Stream()
    ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda")
    mean = np.array(synth.IMAGENET_MEAN, np.float32)
    std = np.array(synth.IMAGENET_STD, np.float32)
    for call in range(2):
        (plain, _, noalloc), pixels, recs = _run_three_ways(L, N, H, W, C, trfn.OUT_F32, trfn.LAYOUT_NHWC,
                                                            710 + call, stream, ws)
        assert np.array_equal(noalloc.view(np.uint8), plain.view(np.uint8))
        ref = oracle.fused_norm(pixels, mean, std, recs, out_dtype=trfn.OUT_F32)
        assert_parity(noalloc, ref, trfn.OUT_F32, "call %d" % call)


def test_noalloc_rejects_bad_arguments_before_the_gpu():
    L = _native.lib()
    mean = _native.float_array(synth.IMAGENET_MEAN)
    std = _native.float_array(synth.IMAGENET_STD)
    assert L.tr_fused_norm_noalloc(None, None, 1, 4, 16, 3, mean, std, None, 1, 0, None) == 1
    assert L.tr_fused_norm_noalloc(0x1000, 0x100000, 1, 4, 16, 5, mean, std, None, 1, 0, None) == 2
    assert L.tr_fused_norm_noalloc(None, None, 0, 4, 16, 3, mean, std, None, 1, 0, None) == 0

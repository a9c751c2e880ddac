"""The GPU record sampler (one thread per image, per-image counter blocks)
against the oracle's per-image sampler, bit for bit, and feeding the fused
kernel directly."""
import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import synth
from parity_util import assert_parity

pytestmark = pytest.mark.gpu


def _device_records(seed, offset, N, H, W, **kw):
    import torch
    out = torch.full((max(N, 1), 5), -7, dtype=torch.int32, device="cuda")
    nxt = trfn.tr_sample_aug_params_device(seed, offset, N, H, W, out, **kw)
    torch.cuda.synchronize()
    return out[:N].cpu().numpy(), nxt


@pytest.mark.parametrize("kw", [
    dict(seed=2003, offset=0, N=4096, H=224, W=224),
    dict(seed=1, offset=12345, N=3000, H=32, W=32, erase_p=0.9),
    dict(seed=7, offset=0, N=2000, H=28, W=28, flip=False),
    dict(seed=9, offset=5, N=5000, H=5, W=3, erase_p=1.0),
    dict(seed=2 ** 40 + 3, offset=2 ** 33, N=1024, H=224, W=224, scale=(0.1, 0.5), ratio=(0.5, 2.0)),
    dict(seed=3, offset=0, N=500, H=224, W=224, erase=False),
    dict(seed=3, offset=0, N=777, H=224, W=224, flip_p=0.25, erase_p=0.3),
    dict(seed=11, offset=99, N=200000, H=224, W=224, erase_p=1.0),
])
def test_device_records_match_the_oracle(kw):
    kw = dict(kw)
    seed, offset, N, H, W = kw.pop("seed"), kw.pop("offset"), kw.pop("N"), kw.pop("H"), kw.pop("W")
    got, nxt = _device_records(seed, offset, N, H, W, **kw)
    ref, rnxt = oracle.sample_aug_params_blocked(seed, offset, N, H, W, **kw)
    assert nxt == rnxt == offset + 24 * N
    assert np.array_equal(got, ref)


def test_empty_batch_and_bad_arguments():
    import torch
    out = torch.zeros((1, 5), dtype=torch.int32, device="cuda")
    assert trfn.tr_sample_aug_params_device(0, 10, 0, 4, 4, out) == 10
    with pytest.raises(trfn.TrError):
        trfn.tr_sample_aug_params_device(0, 0, 4, 4, 4, out, ratio=(0.0, 1.0))
    with pytest.raises(trfn.TrError):
        trfn.tr_sample_aug_params_device(0, 0, -1, 4, 4, out)


def test_device_sampled_records_feed_the_kernel():
    import torch
    N, H, W, C = 64, 224, 224, 3
    mean = np.array(synth.IMAGENET_MEAN, np.float32)
    std = np.array(synth.IMAGENET_STD, np.float32)
    src = synth.pixels_uniform(3, N, H, W, C)
    d_src = torch.from_numpy(src).cuda()
    rec = torch.empty((N, 5), dtype=torch.int32, device="cuda")
    out = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
    stream = torch.cuda.Stream()
    trfn.tr_sample_aug_params_device(42, 0, N, H, W, rec, stream=stream)
    trfn.tr_fused_norm(d_src, out, mean, std, rec, out_dtype=trfn.OUT_F16, stream=stream)
    stream.synchronize()
    recs, _ = oracle.sample_aug_params_blocked(42, 0, N, H, W)
    ref = oracle.fused_norm(src, mean, std, recs, out_dtype=trfn.OUT_F16)
    assert_parity(out.cpu().view(torch.int16).numpy().view(np.uint16), ref, trfn.OUT_F16)

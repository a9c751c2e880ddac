"""Seeded synthetic inputs shared by the tests and the benchmark.

This module only draws pixels and per-image parameter records; it holds none
of the fused step's arithmetic.  The pixel recipes stand in for the datasets
the FusedNormalization article trains on (MNIST, ImageNet), whose images are
not used anywhere here: uniform bytes for ImageNet-like crops, a clipped
Gaussian for a validation-like batch, and mostly-zero strokes for MNIST-like
digits.  Everything is drawn with numpy's PCG64 from an explicit seed.
"""
import numpy as np

IMAGENET_MEAN = (0.485, 0.456, 0.406)
IMAGENET_STD = (0.229, 0.224, 0.225)
MNIST_MEAN = (0.1307,)
MNIST_STD = (0.3081,)


def pixels_uniform(seed, N, H, W, C):
    """uint8 NHWC, every byte uniform on [0, 255]."""
    return np.random.default_rng(seed).integers(0, 256, size=(N, H, W, C), dtype=np.uint8)


def pixels_sparse(seed, N, H, W, C, p_zero=0.8):
    """uint8 NHWC, zero with probability p_zero, else uniform on [1, 255]."""
    g = np.random.default_rng(seed)
    v = g.integers(1, 256, size=(N, H, W, C), dtype=np.uint8)
    v[g.random((N, H, W, C)) < p_zero] = 0
    return v


def pixels_gaussian(seed, N, H, W, C, mean=110.0, sd=60.0):
    """uint8 NHWC, rint(Normal(mean, sd)) clipped to [0, 255]."""
    g = np.random.default_rng(seed)
    return np.clip(np.rint(g.normal(mean, sd, size=(N, H, W, C))), 0, 255).astype(np.uint8)


def pixels_gaussian_into(seed, out, mean=110.0, sd=60.0):
    """The bytes of pixels_gaussian(seed, *out.shape) written into the uint8
    array `out` (for instance a pinned host buffer), with one float64
    temporary instead of three.  numpy releases the GIL while it draws and
    converts, so several threads can fill several batches at once."""
    g = np.random.default_rng(seed)
    v = g.normal(mean, sd, size=out.shape)
    np.rint(v, out=v)
    np.clip(v, 0, 255, out=v)
    out[...] = v.astype(np.uint8)
    return out


def coordinate_image(N, H, W, C):
    """Channel 0 holds x mod 256, channel 1 y mod 256, channel 2 n mod 256,
    channel 3 (x + 2y) mod 256: any misplaced or mirrored element changes value."""
    n = np.arange(N)[:, None, None]
    y = np.arange(H)[None, :, None]
    x = np.arange(W)[None, None, :]
    planes = [x + 0 * (n + y), y + 0 * (n + x), n + 0 * (x + y), x + 2 * y + 0 * n]
    return np.stack([p % 256 for p in planes[:C]], axis=-1).astype(np.uint8)


def random_records(seed, N, H, W, p_flip=0.5, p_erase=0.5, allow_outside=False):
    """Per-image int32 records {flip, y0, x0, h, w} drawn uniformly: a flip bit
    and, with probability p_erase, a rectangle with uniform corners.  With
    allow_outside the rectangle may stick out of the image (it must then be
    clipped by the consumer).  Not the article's RandomErasing rule: a plain
    stress generator for positions and sizes."""
    g = np.random.default_rng(seed)
    rec = np.zeros((N, 5), np.int32)
    rec[:, 0] = g.random(N) < p_flip
    on = g.random(N) < p_erase
    if allow_outside:
        y0 = g.integers(-H // 2, H, N)
        x0 = g.integers(-W // 2, W, N)
        h = g.integers(1, H + 2, N)
        w = g.integers(1, W + 2, N)
    else:
        y0 = g.integers(0, H, N)
        x0 = g.integers(0, W, N)
        h = np.array([g.integers(1, H - a + 1) for a in y0]) if N else np.zeros(0, int)
        w = np.array([g.integers(1, W - a + 1) for a in x0]) if N else np.zeros(0, int)
    rec[on, 1] = y0[on]
    rec[on, 2] = x0[on]
    rec[on, 3] = h[on]
    rec[on, 4] = w[on]
    return rec


# The five workloads: shapes, pixel recipe, normalisation and augmentation
# settings, output type and layout.  Seeds: pixels 1000+k, records 2000+k.
CONFIGS = {
    1: dict(name="n16_32x32x3_f32_nhwc_flip_erase", N=16, H=32, W=32, C=3, pixels="uniform",
            mean=IMAGENET_MEAN, std=IMAGENET_STD, flip=True, erase=True, erase_p=0.5,
            out_dtype="f32", layouts=("nhwc",)),
    2: dict(name="n200_28x28x1_f32_nhwc_plain", N=200, H=28, W=28, C=1, pixels="sparse",
            mean=MNIST_MEAN, std=MNIST_STD, flip=False, erase=False, erase_p=0.0,
            out_dtype="f32", layouts=("nhwc",)),
    3: dict(name="n256_224x224x3_f16_nhwc_flip_erase", N=256, H=224, W=224, C=3, pixels="uniform",
            mean=IMAGENET_MEAN, std=IMAGENET_STD, flip=True, erase=True, erase_p=0.5,
            out_dtype="f16", layouts=("nhwc",)),
    4: dict(name="n256_224x224x3_f32_nhwc_nchw_val", N=256, H=224, W=224, C=3, pixels="gaussian",
            mean=IMAGENET_MEAN, std=IMAGENET_STD, flip=False, erase=False, erase_p=0.0,
            out_dtype="f32", layouts=("nhwc", "nchw")),
    5: dict(name="stream64_n256_224x224x3_f16_nhwc_pinned", N=256, H=224, W=224, C=3, pixels="gaussian",
            mean=IMAGENET_MEAN, std=IMAGENET_STD, flip=True, erase=True, erase_p=0.5,
            out_dtype="f16", layouts=("nhwc",), batches=64),
}


def config_pixels(k, seed=None, N=None):
    cfg = CONFIGS[k]
    seed = 1000 + k if seed is None else seed
    N = cfg["N"] if N is None else N
    shape = (N, cfg["H"], cfg["W"], cfg["C"])
    if cfg["pixels"] == "uniform":
        return pixels_uniform(seed, *shape)
    if cfg["pixels"] == "sparse":
        return pixels_sparse(seed, *shape)
    return pixels_gaussian(seed, *shape)

"""Pins for the CPU oracle: each test checks it against something other than
itself — hand-derived closed forms, exact rational arithmetic, an independent
binary16 conversion, published Philox vectors, invariants and brute force.

Source of the method: the Tech-Renaissance FusedNormalization article
(tech-renaissance.cn/blog/?p=487): §五 (the fused steps), §六/§八 (FP32, FP16
and the 4-channel FP16 layout), §九 (presets), §十 (random decisions),
§十二 (random erasing), §十三 (the article's own FP32-vs-FP16 check).
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from image_preprocessing_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


# ---------------------------------------------------------------- helpers --

def _round_fraction_to_f32(q):
    """Correctly rounded binary32 of an exact rational (ties to even)."""
    x = np.float32(float(q))  # within one binary32 ulp of the answer
    best = None
    for cand in (np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))):
        d = abs(Fraction(float(cand)) - q)
        key = (d, int(np.array(cand, np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def _f16_from_bits(b):
    return np.asarray(b, np.uint16).view(np.float16)


# ------------------------------------------------------ binary16 rounding --

def test_f16_rounding_cases():
    for val, bits in _rows("f16_rounding_cases.txt"):
        f = np.float32(float.fromhex(val))
        assert float(f) == float.fromhex(val), val  # representable exactly
        got = int(oracle.f32_to_f16_bits(np.array([f]))[0])
        assert got == int(bits, 16), (val, hex(got), bits)


def _exponent_chunks():
    # every binary32 exponent field that reaches a distinct binary16 regime:
    # zero/subnormal, the whole binary16 subnormal range and its edges, the
    # normal range edges, overflow, and inf/NaN; both signs, all mantissas.
    exps = [0, 1, 90, 101, 102] + list(range(103, 114)) + [114, 120, 127, 128, 141, 142, 143, 144, 200, 254, 255]
    for sign in (0, 1):
        for e in exps:
            yield (sign << 31) | (e << 23)


def _check_f16_chunk(first, count):
    o = oracle.f32_bits_range_to_f16(first, count)
    f = (np.arange(count, dtype=np.uint32) + np.uint32(first)).view(np.float32)
    with np.errstate(all="ignore"):
        ref = f.astype(np.float16).view(np.uint16)  # numpy's own RNE conversion
    nan = np.isnan(f)
    bad = (o != ref) & ~nan
    assert not bad.any(), hex(first + int(np.argmax(bad)))
    if nan.any():
        on = o[nan]
        assert np.all((on & 0x7C00) == 0x7C00) and np.all((on & 0x3FF) != 0), hex(first)


def test_f16_conversion_matches_numpy_per_exponent():
    for first in _exponent_chunks():
        _check_f16_chunk(first, 1 << 23)


def test_f16_conversion_exhaustive():
    """All 2^32 binary32 patterns through the oracle's own binary16 rounding
    against numpy's conversion (NaNs: any quiet binary16 NaN), in chunks on
    the host's threads (the oracle's C code and numpy release the GIL)."""
    import concurrent.futures as cf
    import threading
    step = 1 << 22
    local = threading.local()

    def check(first):
        if not hasattr(local, "base"):   # per-thread buffers, reused chunk after chunk
            local.base = np.arange(step, dtype=np.uint32)
            local.bits = np.empty(step, np.uint32)
        np.add(local.base, np.uint32(first), out=local.bits)
        f = local.bits.view(np.float32)
        o = oracle.f32_bits_range_to_f16(first, step)
        with np.errstate(all="ignore"):
            ref = f.astype(np.float16).view(np.uint16)
        nan = np.isnan(f)
        bad = (o != ref) & ~nan
        assert not bad.any(), hex(first + int(np.argmax(bad)))
        if nan.any():
            on = o[nan]
            assert np.all((on & 0x7C00) == 0x7C00) and np.all((on & 0x3FF) != 0), hex(first)

    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(check, range(0, 1 << 32, step)))


# ------------------------------------------------------------- presets ----

def test_presets_match_the_article_table():
    cases = {
        "NO_NORM": ([0, 0, 0], [1, 1, 1], 3),
        "MNIST": ([0.1307], [0.3081], 1),
        "CIFAR": ([0.4914, 0.4822, 0.4465], [0.2470, 0.2435, 0.2616], 3),
        "IMAGENET": ([0.485, 0.456, 0.406], [0.229, 0.224, 0.225], 3),
        "MLPERF": ([123.68 / 255, 116.78 / 255, 103.94 / 255], [1 / 255] * 3, 3),
    }
    for name, (m, s, ch) in cases.items():
        mean, std, c = oracle.norm_preset(name)
        assert c == ch
        np.testing.assert_allclose(mean, m, rtol=1e-6)
        np.testing.assert_allclose(std, s, rtol=1e-6)


# ------------------------------------------------------------ value map ---

def test_closed_form_imagenet_golden():
    mean, std, _ = oracle.norm_preset("IMAGENET")
    for u, c, expected in _rows("imagenet_closed_form.txt"):
        img = np.zeros((1, 1, 1, 3), np.uint8)
        img[0, 0, 0, int(c)] = int(u)
        got = oracle.fused_norm(img, mean, std)[0, 0, 0, int(c)]
        assert abs(float(got) - float(expected)) <= 1e-6 * abs(float(expected)) + 1e-7, (u, c, got, expected)


def test_closed_form_endpoints():
    # u = 0 gives -mean/std, u = 255 gives (1-mean)/std (exact rationals of the binary32 constants)
    for name in ("IMAGENET", "CIFAR", "MNIST"):
        mean, std, C = oracle.norm_preset(name)
        for u in (0, 255):
            img = np.full((1, 1, 1, C), u, np.uint8)
            got = oracle.fused_norm(img, mean, std)[0, 0, 0]
            for c in range(C):
                q = (Fraction(u, 255) - Fraction(float(mean[c]))) / Fraction(float(std[c]))
                assert got[c] == _round_fraction_to_f32(q)


@pytest.mark.parametrize("name", list(oracle.PRESETS))
def test_exhaustive_domain_exact_rational(name):
    """A 1x256 image whose pixel x holds x in every channel covers every input
    value of every channel; each output must be the correctly rounded binary32
    of the exact rational (x/255 - mean)/std."""
    mean, std, C = oracle.norm_preset(name)
    img = np.repeat(np.arange(256, dtype=np.uint8)[None, None, :, None], C, axis=3)
    out = oracle.fused_norm(img, mean, std)[0, 0]
    out16 = oracle.fused_norm(img, mean, std, out_dtype=oracle.OUT_F16)[0, 0]
    for x in range(256):
        for c in range(C):
            q = (Fraction(x, 255) - Fraction(float(mean[c]))) / Fraction(float(std[c]))
            assert out[x, c] == _round_fraction_to_f32(q), (name, x, c)
    # the FP16 output is the binary16 rounding of the FP32 output (numpy's converter)
    assert np.array_equal(out16, out.astype(np.float16).view(np.uint16))


def test_no_norm_is_division_by_255():
    mean, std, _ = oracle.norm_preset("NO_NORM")
    img = np.arange(256, dtype=np.uint8).reshape(1, 1, 256, 1).repeat(3, axis=3)
    out = oracle.fused_norm(img, mean, std)
    ref = np.arange(256, dtype=np.float32)[:, None] / np.float32(255.0)  # IEEE division, correctly rounded
    assert np.array_equal(out[0, 0], np.repeat(ref, 3, axis=1))


def test_mlperf_is_shift_by_mean():
    mean, std, _ = oracle.norm_preset("MLPERF")
    img = np.arange(256, dtype=np.uint8).reshape(1, 1, 256, 1).repeat(3, axis=3)
    out = oracle.fused_norm(img, mean, std)[0, 0].astype(np.float64)
    x = np.arange(256, dtype=np.float64)[:, None]
    ref = x - np.array([123.68, 116.78, 103.94])[None, :]
    # std = 1/255 in binary32 makes this x*(1+e) - shift: within a few ulp at |v| <= 152
    assert np.max(np.abs(out - ref)) < 1e-4


# --------------------------------------------------------- flip / erase ---

def _coord_batch(N, H, W, C, seed=0):
    return synth.coordinate_image(N, H, W, C)


def test_flip_of_mirror_is_identity():
    mean, std, _ = oracle.norm_preset("IMAGENET")
    src = synth.pixels_uniform(11, 3, 7, 9, 3)
    mirrored = np.ascontiguousarray(src[:, :, ::-1, :])
    flip = np.zeros((3, 5), np.int32)
    flip[:, 0] = 1
    for dt in (oracle.OUT_F32, oracle.OUT_F16):
        a = oracle.fused_norm(mirrored, mean, std, flip, out_dtype=dt)
        b = oracle.fused_norm(src, mean, std, None, out_dtype=dt)
        assert np.array_equal(a, b)


def test_flip_positions_on_coordinate_images():
    N, H, W, C = 2, 5, 13, 3
    src = synth.coordinate_image(N, H, W, C)
    mean, std = np.zeros(3, np.float32), np.full(3, 1.0 / 255.0, np.float32)  # near-identity map
    aug = np.array([[1, 0, 0, 0, 0], [0, 0, 0, 0, 0]], np.int32)
    out = oracle.fused_norm(src, mean, std, aug)
    # channel 0 of the coordinate image encodes x: flipped image n=0 shows W-1-x
    assert np.array_equal(np.rint(out[0, :, :, 0]).astype(int), np.broadcast_to(W - 1 - np.arange(W), (H, W)))
    assert np.array_equal(np.rint(out[1, :, :, 0]).astype(int), np.broadcast_to(np.arange(W), (H, W)))
    # channel 1 encodes y and is untouched by the flip; channel order is kept
    assert np.array_equal(np.rint(out[0, :, :, 1]).astype(int), np.broadcast_to(np.arange(H)[:, None], (H, W)))


def test_erase_is_exact_zero_inside_and_identity_outside():
    mean, std, _ = oracle.norm_preset("IMAGENET")
    src = synth.pixels_uniform(5, 2, 16, 12, 3)
    aug = np.array([[0, 3, 2, 5, 4], [1, 0, 7, 16, 5]], np.int32)
    for dt in (oracle.OUT_F32, oracle.OUT_F16):
        noerase = aug.copy()
        noerase[:, 3:] = 0
        full = oracle.fused_norm(src, mean, std, noerase, out_dtype=dt)
        er = oracle.fused_norm(src, mean, std, aug, out_dtype=dt)
        mask = np.zeros((2, 16, 12), bool)
        mask[0, 3:8, 2:6] = True
        mask[1, 0:16, 7:12] = True
        bits = er.view(np.uint32) if dt == oracle.OUT_F32 else er
        assert np.all(bits[mask] == 0)  # +0, not -0
        assert np.array_equal(er[~mask], full[~mask])
        # the zero mask recovers the rectangle exactly (IMAGENET has no other zeros)
        assert np.array_equal(np.all(bits == 0, axis=-1), mask)


def test_erase_rectangle_is_clipped_to_the_image():
    mean, std, _ = oracle.norm_preset("IMAGENET")
    src = synth.pixels_uniform(6, 1, 6, 6, 3)
    aug = np.array([[0, 4, -2, 10, 4]], np.int32)  # rows 4..13, cols -2..1
    out = oracle.fused_norm(src, mean, std, aug)
    zero = np.all(out.view(np.uint32) == 0, axis=-1)[0]
    expect = np.zeros((6, 6), bool)
    expect[4:6, 0:2] = True
    assert np.array_equal(zero, expect)


def _direct(src, mean, std, flip, rect):
    """Separately written direct formula with numpy array operations."""
    img = src[:, ::-1, :] if flip else src
    v = (img.astype(np.float64) / 255.0 - mean.astype(np.float64)) / std.astype(np.float64)
    v = v.astype(np.float32)
    if rect is not None:
        y0, x0, h, w = rect
        v[y0:y0 + h, x0:x0 + w, :] = 0.0
    return v


def test_brute_force_every_rect_4x4x3():
    mean, std, _ = oracle.norm_preset("CIFAR")
    src = synth.pixels_uniform(77, 1, 4, 4, 3)
    rects = [None] + [(y0, x0, h, w) for y0 in range(4) for x0 in range(4)
                      for h in range(1, 5 - y0) for w in range(1, 5 - x0)]
    for flip in (0, 1):
        for r in rects:
            aug = np.zeros((1, 5), np.int32)
            aug[0, 0] = flip
            if r is not None:
                aug[0, 1:] = r
            got = oracle.fused_norm(src, mean, std, aug)[0]
            assert np.array_equal(got, _direct(src[0], mean, std, flip, r)), (flip, r)
            got16 = oracle.fused_norm(src, mean, std, aug, out_dtype=oracle.OUT_F16)[0]
            assert np.array_equal(got16, got.astype(np.float16).view(np.uint16))


def test_layouts_are_permutations_of_nhwc():
    mean, std, _ = oracle.norm_preset("IMAGENET")
    src = synth.pixels_uniform(9, 3, 5, 7, 3)
    aug = np.array([[1, 1, 1, 2, 3], [0, 0, 0, 0, 0], [1, 4, 6, 1, 1]], np.int32)
    for dt in (oracle.OUT_F32, oracle.OUT_F16):
        nhwc = oracle.fused_norm(src, mean, std, aug, out_dtype=dt)
        nchw = oracle.fused_norm(src, mean, std, aug, out_dtype=dt, layout=oracle.LAYOUT_NCHW)
        nhwc4 = oracle.fused_norm(src, mean, std, aug, out_dtype=dt, layout=oracle.LAYOUT_NHWC4)
        assert np.array_equal(nchw, np.transpose(nhwc, (0, 3, 1, 2)))
        assert np.array_equal(nhwc4[..., :3], nhwc)
        assert np.all(nhwc4[..., 3:].view(np.uint16 if dt else np.uint32) == 0)


def test_articles_fp32_vs_fp16_check():
    """The article's own check (§十三): 28x28 gray, FP32 vs FP16 output,
    MSE < 1e-5 and max relative error < 1e-3 over |v| > 1e-6."""
    mean, std, _ = oracle.norm_preset("MNIST")
    src = synth.pixels_sparse(3, 4, 28, 28, 1)
    f32 = oracle.fused_norm(src, mean, std).astype(np.float64)
    f16 = _f16_from_bits(oracle.fused_norm(src, mean, std, out_dtype=oracle.OUT_F16)).astype(np.float64)
    mse = np.mean((f32 - f16) ** 2)
    sel = np.abs(f32) > 1e-6
    rel = np.max(np.abs(f32[sel] - f16[sel]) / np.abs(f32[sel]))
    assert mse < 1e-5 and rel < 1e-3


def test_rejects_bad_arguments():
    src = np.zeros((1, 2, 2, 3), np.uint8)
    with pytest.raises(ValueError):
        oracle.fused_norm(src, np.zeros(3), np.ones(3), out_dtype=7)


# ----------------------------------------------------------- Philox / RNG --

def test_philox_known_answer_vectors():
    for row in _rows("philox4x32_10_kat.txt"):
        v = [int(t, 16) for t in row]
        assert oracle.philox4x32_10(v[0:4], v[4:6]).tolist() == v[6:10]


def test_uniform_is_in_unit_interval_and_uniform():
    u = np.array([oracle.uniform01(12345, k) for k in range(40000)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 4 * np.sqrt(1 / 12 / u.size)
    hist = np.histogram(u, bins=16, range=(0, 1))[0]
    exp = u.size / 16
    assert np.sum((hist - exp) ** 2 / exp) < 45  # chi-square, 15 dof, far tail
    # 24-bit grid
    assert np.all(np.floor(u * 2 ** 24) == u * 2 ** 24)


def test_sampler_is_deterministic_and_resumable():
    a, nxt = oracle.sample_aug_params(7, 100, 64, 224, 224)
    b, nxt2 = oracle.sample_aug_params(7, 100, 64, 224, 224)
    assert np.array_equal(a, b) and nxt == nxt2
    # sampling in two halves, resuming from the returned offset, gives the same stream
    h1, mid = oracle.sample_aug_params(7, 100, 30, 224, 224)
    h2, end = oracle.sample_aug_params(7, mid, 34, 224, 224)
    assert np.array_equal(np.concatenate([h1, h2]), a) and end == nxt


def test_sampler_consumes_no_draw_when_disabled():
    a, nxt = oracle.sample_aug_params(1, 50, 10, 32, 32, flip=False, erase=False)
    assert nxt == 50 and not a.any()
    a, nxt = oracle.sample_aug_params(1, 50, 10, 32, 32, flip=True, erase=False)
    assert nxt == 60 and not a[:, 1:].any()
    a, nxt = oracle.sample_aug_params(1, 50, 10, 32, 32, flip=False, erase=True, erase_p=0.0)
    assert nxt == 50 and not a.any()


def test_sampler_draw_count_per_image():
    # flip draw + gate draw, then 2 per attempt, then 2 on acceptance
    for seed in range(40):
        a, nxt = oracle.sample_aug_params(seed, 0, 1, 224, 224, erase_p=1.0)
        if a[0, 3] > 0:
            assert nxt in [2 + 2 * k + 2 for k in range(1, 11)]
        else:
            assert nxt == 2 + 20  # ten rejected attempts
        a, nxt = oracle.sample_aug_params(seed, 0, 1, 224, 224, erase_p=1e-9)
        assert nxt == 2  # the gate failed: flip draw + gate draw only


def test_sampler_rects_are_valid_and_strictly_inside():
    for (H, W) in ((224, 224), (32, 32), (7, 5), (2, 2)):
        a, _ = oracle.sample_aug_params(11, 0, 3000, H, W, erase_p=0.9)
        e = a[a[:, 3] > 0]
        assert np.all((a[:, 3] > 0) == (a[:, 4] > 0))
        assert np.all(e[:, 3] < H) and np.all(e[:, 4] < W)
        assert np.all(e[:, 1] >= 0) and np.all(e[:, 2] >= 0)
        assert np.all(e[:, 1] + e[:, 3] <= H) and np.all(e[:, 2] + e[:, 4] <= W)


def test_sampler_randint_is_inclusive():
    # at 4x4 the rectangle is small; the last start row H-h must be reachable
    a, _ = oracle.sample_aug_params(5, 0, 20000, 4, 4, flip=False, erase_p=1.0)
    e = a[a[:, 3] > 0]
    assert np.any(e[:, 1] == 4 - e[:, 3]) and np.any(e[:, 1] == 0)
    assert np.any(e[:, 2] == 4 - e[:, 4]) and np.any(e[:, 2] == 0)


def test_sampler_moments_at_224():
    N = 20000
    a, _ = oracle.sample_aug_params(2003, 0, N, 224, 224)
    sigma = np.sqrt(0.25 / N)
    assert abs(a[:, 0].mean() - 0.5) < 4 * sigma  # flip rate
    erased = a[:, 3] > 0
    assert abs(erased.mean() - 0.5) < 4 * sigma  # gate p = 0.5, attempts practically never all fail
    area = (a[erased, 3] * a[erased, 4]) / (224.0 * 224.0)
    # area fraction ~ U[0.02, 0.33] truncated by validity: mean near 0.175
    assert 0.16 < area.mean() < 0.19
    assert area.min() > 0.015 and area.max() < 0.345
    ar = a[erased, 3] / a[erased, 4]
    # log aspect ratio ~ U[log 0.3, log 3.3]: median near 1, both sides populated
    assert 0.8 < np.median(ar) < 1.25
    assert np.mean(ar > 1) > 0.4 and np.mean(ar < 1) > 0.4
    # erased pixel fraction per image ~ 0.5 * 0.175
    frac = (a[:, 3] * a[:, 4]).sum() / (N * 224.0 * 224.0)
    assert 0.08 < frac < 0.095


@pytest.mark.parametrize("blocked", [False, True])
def test_sampler_rates_follow_p(blocked):
    """Flip iff u < flip_p (§五) and erase iff u < p (§十二): away from 1/2 the
    rates tell a reversed comparison from the right one."""
    N = 20000
    sample = oracle.sample_aug_params_blocked if blocked else oracle.sample_aug_params
    a, _ = sample(31, 0, N, 224, 224, flip_p=0.2, erase_p=0.3)
    for rate, p in ((a[:, 0].mean(), 0.2), ((a[:, 3] > 0).mean(), 0.3)):
        assert abs(rate - p) < 4 * np.sqrt(p * (1 - p) / N), (rate, p)


# ------------------------------------------------------------- crop -------

def _strided(src, row_pad, image_pad):
    """Lay a compact (N, SH, SW, C) batch out with padded rows and images."""
    N, SH, SW, C = src.shape
    row_stride = SW * C + row_pad
    image_stride = SH * row_stride + image_pad
    buf = np.full(N * image_stride, 0xEE, np.uint8)
    for n in range(N):
        for y in range(SH):
            o = n * image_stride + y * row_stride
            buf[o:o + SW * C] = src[n, y].reshape(-1)
    return buf, image_stride, row_stride


@pytest.mark.parametrize("pads", [(0, 0), (16, 0), (5, 96), (48, 7)])
def test_crop_equals_slicing_then_the_plain_step(pads):
    """A window of a strided source equals numpy slicing followed by the
    compact oracle: the crop only moves indices."""
    mean, std, _ = oracle.norm_preset("IMAGENET")
    N, SH, SW, C, H, W = 4, 12, 20, 3, 7, 9
    src = synth.pixels_uniform(21, N, SH, SW, C)
    buf, istr, rstr = _strided(src, *pads)
    crop = np.array([[0, 0], [5, 11], [2, 3], [SH - H, SW - W]], np.int32)
    aug = np.array([[1, 1, 2, 3, 4], [0, 0, 0, 0, 0], [1, 6, 8, 1, 1], [0, 2, 0, 5, 9]], np.int32)
    for dt in (oracle.OUT_F32, oracle.OUT_F16):
        for lay in (oracle.LAYOUT_NHWC, oracle.LAYOUT_NCHW, oracle.LAYOUT_NHWC4):
            got = oracle.fused_norm_crop(buf, istr, rstr, SH, SW, N, H, W, C, mean, std, crop, aug, dt, lay)
            windows = np.stack([src[n, cy:cy + H, cx:cx + W] for n, (cy, cx) in enumerate(crop)])
            assert np.array_equal(got, oracle.fused_norm(windows, mean, std, aug, out_dtype=dt, layout=lay))


def test_crop_rejects_windows_outside_the_source():
    mean, std, _ = oracle.norm_preset("IMAGENET")
    src = synth.pixels_uniform(1, 1, 8, 8, 3)
    with pytest.raises(ValueError):
        oracle.fused_norm_crop(src.reshape(-1), 192, 24, 8, 8, 1, 4, 4, 3, mean, std, np.array([[5, 0]]))
    with pytest.raises(ValueError):
        oracle.fused_norm_crop(src.reshape(-1), 192, 24, 8, 8, 1, 4, 4, 3, mean, std, np.array([[0, -1]]))


# ------------------------------------------ per-image counter blocks ------

def test_own_exp_is_within_two_ulp_of_the_exact_exp():
    x = np.linspace(-20.0, 20.0, 400001, dtype=np.float32)
    x = np.concatenate([x, np.log(np.float32([0.3, 3.3])), np.float32([0.0, -1e-8, 1e-8, 0.34657359])])
    got = oracle.exp_f32(x).astype(np.float64)
    exact = np.exp(x.astype(np.float64))
    ulp = np.spacing(exact.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got - exact) / ulp) <= 2.0
    assert oracle.exp_f32(np.float32([0.0]))[0] == 1.0


def test_blocked_sampler_is_per_image():
    """Image n's record depends only on (seed, offset + 24n): sampling a
    suffix from its block offset gives the same records."""
    a, nxt = oracle.sample_aug_params_blocked(5, 1000, 64, 224, 224, erase_p=0.7)
    assert nxt == 1000 + 24 * 64
    b, _ = oracle.sample_aug_params_blocked(5, 1000 + 24 * 40, 24, 224, 224, erase_p=0.7)
    assert np.array_equal(a[40:], b)
    c, _ = oracle.sample_aug_params_blocked(5, 1000, 64, 224, 224, erase_p=0.7)
    assert np.array_equal(a, c)


def test_blocked_sampler_distribution():
    N = 20000
    a, _ = oracle.sample_aug_params_blocked(2003, 0, N, 224, 224)
    sigma = np.sqrt(0.25 / N)
    assert abs(a[:, 0].mean() - 0.5) < 4 * sigma
    erased = a[:, 3] > 0
    assert abs(erased.mean() - 0.5) < 4 * sigma
    area = (a[erased, 3] * a[erased, 4]) / (224.0 * 224.0)
    assert 0.16 < area.mean() < 0.19
    e = a[erased]
    assert np.all(e[:, 1] + e[:, 3] <= 224) and np.all(e[:, 2] + e[:, 4] <= 224)
    assert np.all(e[:, 3] < 224) and np.all(e[:, 4] < 224) and np.all(e[:, 1:3] >= 0)
    ar = a[erased, 3] / a[erased, 4]
    assert 0.8 < np.median(ar) < 1.25


def test_blocked_and_sequential_samplers_agree_on_the_first_image():
    # image 0 draws from offset, offset+1, ... in both forms
    a, _ = oracle.sample_aug_params(9, 77, 1, 224, 224, erase_p=1.0)
    b, _ = oracle.sample_aug_params_blocked(9, 77, 1, 224, 224, erase_p=1.0)
    # the rectangle sizes may differ only through exp's last place; the flip and the gate agree
    assert a[0, 0] == b[0, 0] and (a[0, 3] > 0) == (b[0, 3] > 0)

"""Planted mistakes: each case copies the oracle's C source, plants one
plausible mistake in it (a dropped term, a wrong sign, index or bound, a
transposed operand, a lost rounding rule), builds the copy on the CPU and runs
the pins of test_oracle.py against it.  Every planted mistake must fail at
least one pin, and the unmodified source must pass them all, so the pins are
shown to reach every part of the oracle the parity tests lean on.

Each mutation is a plain text substitution that keeps every memory access of
the oracle inside its buffers (indices are permuted or mirrored within the
same ranges, never shifted out of them).

Source of the method: the Tech-Renaissance FusedNormalization article
(tech-renaissance.cn/blog/?p=487): §五 (the fused steps), §六/§八 (FP32, FP16,
the 4-channel layout), §十 (random decisions), §十二 (random erasing).
"""
import hashlib
import os
import re

import numpy as np
import pytest

import oracle
from oracle.build import SRC, compile_oracle

import test_oracle as pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

NORM = "((double)u / 255.0 - (double)mean[c]) / (double)stdv[c]"
ERASE_TEST = ("const int erased = has_erase && y >= ey0 && y < ey0 + eh &&\n"
              "                                   x >= ex0 && x < ex0 + ew;\n"
              "                const int xs = flip ? (W - 1 - x) : x;   /* mirrored read */")

# name -> list of (text in the oracle source, replacement); every occurrence
# of the text is replaced
MUTANTS = {
    # value map (§五: x/255, then (x - mean)/std)
    "mean dropped": [(NORM, "((double)u / 255.0) / (double)stdv[c]")],
    "mean added": [(NORM, "((double)u / 255.0 + (double)mean[c]) / (double)stdv[c]")],
    "std multiplies": [(NORM, "((double)u / 255.0 - (double)mean[c]) * (double)stdv[c]")],
    "divides by 256": [(NORM, "((double)u / 256.0 - (double)mean[c]) / (double)stdv[c]")],
    "first channel's constants": [(NORM, "((double)u / 255.0 - (double)mean[0]) / (double)stdv[0]")],
    "binary32 arithmetic": [(NORM, "(double)(((float)u / 255.0f - mean[c]) / stdv[c])")],
    # flip (§五: the mirrored column)
    "flip dropped": [("const int xs = flip ? (W - 1 - x) : x;", "const int xs = x; (void)flip;")],
    "flip inverted": [("const int xs = flip ? (W - 1 - x) : x;", "const int xs = flip ? x : (W - 1 - x);")],
    # erase (§十二: [y0, y0+h) x [x0, x0+w) in output coordinates, +0)
    "erase rows end inclusive": [("y < ey0 + eh", "y <= ey0 + eh")],
    "erase columns end inclusive": [("x < ex0 + ew", "x <= ex0 + ew")],
    "erase axes swapped": [("y >= ey0 && y < ey0 + eh &&\n                                   x >= ex0 && x < ex0 + ew",
                            "y >= ex0 && y < ex0 + ew &&\n                                   x >= ey0 && x < ey0 + eh")],
    "erase in source coordinates": [(ERASE_TEST,
                                     "const int xs = flip ? (W - 1 - x) : x;\n"
                                     "                const int erased = has_erase && y >= ey0 && y < ey0 + eh &&\n"
                                     "                                   xs >= ex0 && xs < ex0 + ew;")],
    "erase writes -0": [("v32 = 0.0f;", "v32 = -0.0f;")],
    # layouts (§六/§八)
    "NCHW index transposed": [("o = (((size_t)n * C + c) * H + y) * W + x;",
                               "o = (((size_t)n * C + c) * W + x) * H + y;")],
    "NHWC4 pixel stride of C": [("o = (((size_t)n * H + y) * W + x) * out_ch + c;",
                                 "o = (((size_t)n * H + y) * W + x) * C + c;")],
    # binary16 rounding (§六: round to nearest, ties to even)
    "ties away from zero": [("(rem == half && (q & 1))", "(rem == half)")],
    "truncation": [("q += 1;\n    return q;", "q += 0;\n    return q;")],
    "no carry into the exponent": [("if (q == 2048) { q = 1024; E += 1; }", "")],
    "subnormal shift off by one": [("unsigned s = (unsigned)(-(E + 1));", "unsigned s = (unsigned)(-E);")],
    "overflow one binade late": [("if (he >= 31)", "if (he > 31)")],
    "sign dropped": [("uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);", "uint16_t sign = 0;")],
    "NaN made infinity": [("return (uint16_t)(sign | 0x7C00u | 0x0200u | (frac >> 13));",
                           "return (uint16_t)(sign | 0x7C00u);")],
    # presets (§九)
    "a preset constant": [("stdv[1] = 0.224f", "stdv[1] = 0.225f")],
    # Philox4x32-10
    "key bump dropped": [("key[1] += 0xBB67AE85u;", "key[1] += 0u;")],
    "round output words swapped": [("out[0] = hi1 ^ ctr[1] ^ key[0];", "out[0] = hi0 ^ ctr[1] ^ key[0];")],
    "nine rounds": [("for (int r = 0; r < 10; ++r)", "for (int r = 0; r < 9; ++r)")],
    "uniform on 23 bits": [("return out[0] >> 8;", "return out[0] >> 9;")],
    # sampler (§十, §十二)
    "randint exclusive": [("(int64_t)hi - (int64_t)lo + 1", "(int64_t)hi - (int64_t)lo")],
    "flip comparison reversed": [("(rng_uniform(&g, 0.0f, 1.0f) < flip_p)", "(rng_uniform(&g, 0.0f, 1.0f) >= flip_p)")],
    "erase gate reversed": [("if (rng_uniform(&g, 0.0f, 1.0f) >= erase_p) continue;",
                             "if (rng_uniform(&g, 0.0f, 1.0f) < erase_p) continue;")],
    "aspect applied to both sides": [("int eh = (int)roundf(sqrtf(area * ar));", "int eh = (int)roundf(sqrtf(area / ar));")],
    "blocked: flip comparison reversed": [("(block_uniform(seed, base, &k) < flip_p)",
                                           "(block_uniform(seed, base, &k) >= flip_p)")],
    "blocked: block of 23 draws": [("const uint64_t base = offset + (uint64_t)n * ORACLE_DRAWS_PER_IMAGE;",
                                    "const uint64_t base = offset + (uint64_t)n * 23u;")],
    "exp: a Taylor term dropped": [("p = fmaf(p, r, 1.0f / 24.0f);", "p = fmaf(p, r, 0.0f);")],
    "exp: 2^k one binade low": [("(uint32_t)((int)k + 127) << 23", "(uint32_t)((int)k + 126) << 23")],
    # crop (a window of a strided source, then the step)
    "crop ignores the flip": [("(size_t)(cx + xs) * C + c", "(size_t)(cx + x) * C + c")],
    "crop rows mirrored": [("(size_t)(cy + y) * row_stride", "(size_t)(cy + H - 1 - y) * row_stride")],
}


def _f16_sampled():
    """The per-exponent binary16 pin on a random sample of each exponent's
    mantissas (the full pin covers all of them and takes tens of seconds)."""
    rng = np.random.default_rng(3)
    for first in pins._exponent_chunks():
        bits = (np.uint32(first) + rng.integers(0, 1 << 23, 4096, dtype=np.uint32)).astype(np.uint32)
        bits = np.concatenate([bits, np.uint32(first) + np.arange(0, 1 << 23, 1 << 13, dtype=np.uint32)])
        f = bits.view(np.float32)
        got = oracle.f32_to_f16_bits(f)
        with np.errstate(all="ignore"):
            ref = f.astype(np.float16).view(np.uint16)
        nan = np.isnan(f)
        assert np.array_equal(got[~nan], ref[~nan]), hex(int(first))
        gn = got[nan]
        assert np.all((gn & 0x7C00) == 0x7C00) and np.all((gn & 0x3FF) != 0)   # NaN stays NaN


def _battery():
    yield "presets", pins.test_presets_match_the_article_table
    yield "f16 rounding cases", pins.test_f16_rounding_cases
    yield "f16 per exponent (sampled)", _f16_sampled
    yield "closed form golden", pins.test_closed_form_imagenet_golden
    yield "closed form endpoints", pins.test_closed_form_endpoints
    for name in oracle.PRESETS:
        yield "exact rational " + name, lambda name=name: pins.test_exhaustive_domain_exact_rational(name)
    yield "no_norm", pins.test_no_norm_is_division_by_255
    yield "mlperf", pins.test_mlperf_is_shift_by_mean
    yield "flip of mirror", pins.test_flip_of_mirror_is_identity
    yield "flip positions", pins.test_flip_positions_on_coordinate_images
    yield "erase zero inside", pins.test_erase_is_exact_zero_inside_and_identity_outside
    yield "erase clipped", pins.test_erase_rectangle_is_clipped_to_the_image
    yield "brute force 4x4x3", pins.test_brute_force_every_rect_4x4x3
    yield "layouts", pins.test_layouts_are_permutations_of_nhwc
    yield "article fp32 vs fp16", pins.test_articles_fp32_vs_fp16_check
    yield "philox KAT", pins.test_philox_known_answer_vectors
    yield "uniform", pins.test_uniform_is_in_unit_interval_and_uniform
    yield "sampler deterministic", pins.test_sampler_is_deterministic_and_resumable
    yield "sampler no draw", pins.test_sampler_consumes_no_draw_when_disabled
    yield "sampler draw count", pins.test_sampler_draw_count_per_image
    yield "sampler rects valid", pins.test_sampler_rects_are_valid_and_strictly_inside
    yield "sampler randint inclusive", pins.test_sampler_randint_is_inclusive
    yield "sampler moments", pins.test_sampler_moments_at_224
    for blocked in (False, True):
        yield "sampler rates %d" % blocked, lambda b=blocked: pins.test_sampler_rates_follow_p(b)
    for pads in ((0, 0), (5, 96)):
        yield "crop %s" % (pads,), lambda p=pads: pins.test_crop_equals_slicing_then_the_plain_step(p)
    yield "own exp", pins.test_own_exp_is_within_two_ulp_of_the_exact_exp
    yield "blocked per image", pins.test_blocked_sampler_is_per_image
    yield "blocked distribution", pins.test_blocked_sampler_distribution
    yield "blocked vs sequential", pins.test_blocked_and_sequential_samplers_agree_on_the_first_image


def _failing_pins(lib, stop_at_first):
    saved = oracle._lib
    oracle._lib = lib
    failed = []
    try:
        for name, pin in _battery():
            try:
                pin()
            except (AssertionError, ValueError) as e:
                failed.append((name, type(e).__name__))
                if stop_at_first:
                    break
    finally:
        oracle._lib = saved
    return failed


def _build(tmp_path, name, text):
    # a file name of its own for every build: the dynamic loader hands back
    # the library already loaded from a path instead of reading it again
    stem = "%s_%s" % (re.sub(r"[^A-Za-z0-9]+", "_", name), hashlib.sha256(text.encode()).hexdigest()[:12])
    src = os.path.join(str(tmp_path), stem + ".c")
    with open(src, "w") as f:
        f.write(text)
    return oracle.bind(compile_oracle(src, os.path.join(str(tmp_path), stem + ".so")))


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_unmodified_source_passes_every_pin(source, tmp_path):
    assert _failing_pins(_build(tmp_path, "control", source), stop_at_first=False) == []


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(name, source, tmp_path):
    text = source
    for old, new in MUTANTS[name]:
        assert old in text, "the oracle no longer contains %r" % old
        text = text.replace(old, new)
    assert text != source
    failed = _failing_pins(_build(tmp_path, name, text), stop_at_first=True)
    assert failed, "no pin fails when the oracle has the mistake %r" % name

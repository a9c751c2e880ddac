/*
 * Oracle for FusedNormalization — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of what the fused
 * preprocessing step computes, written from the Tech-Renaissance article
 * "(11) FusedNormalization: fuse the last step of data augmentation into one
 * memory traversal" (tech-renaissance.cn/blog/?p=487).  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark may load this
 * file; the product library never links, calls or includes it, and it shares
 * no code, header, table or helper with the CUDA path.
 *
 * Arithmetic: every normalised value is formed in binary64 from its plain
 * definition and rounded once to binary32; the binary16 output is the
 * round-to-nearest-even conversion of that binary32 value, done by this
 * file's own bit-level routine.  Build with -O2 and -ffp-contract=off, no
 * fast-math.
 *
 * Pins (all in tests/test_oracle.py, none of which re-types these formulas):
 *   - value map: hand-derived closed forms, exact rational arithmetic over the
 *     whole 256-value input domain of every channel;
 *   - flip: flip(mirror(img)) == no-flip(img), coordinate-encoding images;
 *   - erase: exact +0 inside the rectangle, unchanged elsewhere;
 *   - brute force over every rectangle of 4x4x3 images;
 *   - binary16 conversion: exhaustive over all 2^32 binary32 patterns against
 *     an independent library conversion;
 *   - Philox4x32-10: the published known-answer vectors of its authors.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_OUT_F32 0
#define ORACLE_OUT_F16 1
#define ORACLE_LAYOUT_NHWC 0
#define ORACLE_LAYOUT_NCHW 1
#define ORACLE_LAYOUT_NHWC4 2

/* ------------------------------------------------------------------------ */
/* binary32 -> binary16, round to nearest, ties to even (IEEE 754-2008 §4.3.1).
 * The F16C instruction the article uses for its FP16 output rounds this way
 * (article §六 "FP32 and FP16 output": rounding-mode immediate 0).          */

/* Shift m right by s bits (1 <= s <= 40), rounding to nearest, ties to even. */
static uint64_t shift_right_rne(uint64_t m, unsigned s) {
    uint64_t q = m >> s;
    uint64_t rem = m & ((((uint64_t)1) << s) - 1);
    uint64_t half = ((uint64_t)1) << (s - 1);
    if (rem > half || (rem == half && (q & 1))) q += 1;
    return q;
}

uint16_t oracle_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t bexp = (x >> 23) & 0xFFu;
    uint32_t frac = x & 0x7FFFFFu;

    if (bexp == 0xFFu) {                       /* infinity or NaN */
        if (frac == 0) return (uint16_t)(sign | 0x7C00u);
        /* NaN stays NaN: keep the top payload bits and force the quiet bit. */
        return (uint16_t)(sign | 0x7C00u | 0x0200u | (frac >> 13));
    }
    if (bexp == 0) {
        /* zero or binary32 subnormal: magnitude < 2^-126, far below half of
         * the smallest binary16 subnormal (2^-25), so it rounds to zero.   */
        return sign;
    }
    /* value = M * 2^(E-23) with a 24-bit significand M */
    uint64_t M = (uint64_t)(frac | 0x800000u);
    int E = (int)bexp - 127;

    if (E >= -14) {
        /* binary16 normal range: keep 11 significant bits */
        uint64_t q = shift_right_rne(M, 13);   /* in [1024, 2048] */
        if (q == 2048) { q = 1024; E += 1; }
        int he = E + 15;
        if (he >= 31) return (uint16_t)(sign | 0x7C00u);   /* overflow */
        return (uint16_t)(sign | ((uint32_t)he << 10) | (uint32_t)(q & 0x3FFu));
    }
    /* binary16 subnormal range: count units of 2^-24.
     * value / 2^-24 = M * 2^(E+1), and E+1 <= -14 here.                    */
    unsigned s = (unsigned)(-(E + 1));
    if (s > 40) return sign;                   /* far below 2^-25 */
    uint64_t q = shift_right_rne(M, s);        /* q == 1024 is the smallest normal */
    return (uint16_t)(sign | (uint32_t)q);
}

void oracle_f32_to_f16_array(const float* in, uint16_t* out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(in[i]);
}

/* Exhaustive self-check helper: converts the 2^k consecutive bit patterns
 * starting at `first` (as binary32) into `out`.                             */
void oracle_f32_to_f16_bits_range(uint32_t first, uint32_t count, uint16_t* out) {
    for (uint32_t i = 0; i < count; ++i) {
        uint32_t b = first + i;
        float f;
        memcpy(&f, &b, sizeof f);
        out[i] = oracle_f32_to_f16(f);
    }
}

/* ------------------------------------------------------------------------ */
/* Normalisation presets (article §九 "Five normalisation presets").
 * mean/std are the binary32 constants the article's table holds; MLPERF's are
 * the binary32 quotients of its printed values by 255.                      */
int oracle_norm_preset(int preset, float mean[3], float stdv[3], int* channels) {
    switch (preset) {
    case 0: /* NO_NORM */
        mean[0] = 0.0f; mean[1] = 0.0f; mean[2] = 0.0f;
        stdv[0] = 1.0f; stdv[1] = 1.0f; stdv[2] = 1.0f;
        *channels = 3; return 0;
    case 1: /* MNIST */
        mean[0] = 0.1307f; mean[1] = 0.0f; mean[2] = 0.0f;
        stdv[0] = 0.3081f; stdv[1] = 1.0f; stdv[2] = 1.0f;
        *channels = 1; return 0;
    case 2: /* CIFAR */
        mean[0] = 0.4914f; mean[1] = 0.4822f; mean[2] = 0.4465f;
        stdv[0] = 0.2470f; stdv[1] = 0.2435f; stdv[2] = 0.2616f;
        *channels = 3; return 0;
    case 3: /* IMAGENET */
        mean[0] = 0.485f; mean[1] = 0.456f; mean[2] = 0.406f;
        stdv[0] = 0.229f; stdv[1] = 0.224f; stdv[2] = 0.225f;
        *channels = 3; return 0;
    case 4: /* MLPERF */
        mean[0] = 123.68f / 255.0f; mean[1] = 116.78f / 255.0f; mean[2] = 103.94f / 255.0f;
        stdv[0] = 1.0f / 255.0f; stdv[1] = 1.0f / 255.0f; stdv[2] = 1.0f / 255.0f;
        *channels = 3; return 0;
    default:
        return -1;
    }
}

/* ------------------------------------------------------------------------ */
/* The fused step itself (article §五 "What FusedNormalization fuses", §十二
 * "Random erasing"): per image, an optional horizontal flip and an optional
 * erase rectangle; per element, ToTensor (x/255) then Normalize
 * ((x - mean)/std); erased output elements are +0 for every channel.
 *
 * Readings of points the article leaves open:
 *   - the erase rectangle is applied to the output buffer after the flipped
 *     main pass, so it is in output (post-flip) coordinates;
 *   - the erased value is +0.0 (a memset of the normalised output);
 *   - a rectangle with h <= 0 or w <= 0 means "no erase"; parts of a
 *     rectangle outside the image erase nothing;
 *   - any non-zero flip word means "flip".
 *
 * src   : uint8, compact NHWC, N*H*W*C bytes.
 * dst   : binary32 or binary16 (as uint16 bits), compact, in the layout asked:
 *           NHWC  ((n*H + y)*W + x)*C + c
 *           NCHW  ((n*C + c)*H + y)*W + x
 *           NHWC4 ((n*H + y)*W + x)*4 + c, channels C..3 set to +0
 *             (the article's AMP layout, §六 and §八).
 * aug   : N records of five int32 {flip, y0, x0, h, w}, or NULL (no flip, no
 *         erase for every image).
 * Only images n_begin <= n < n_end are written (to split work over threads).
 * Returns 0, or -1 for arguments the article's contract rejects.            */
int oracle_fused_norm(const uint8_t* src, void* dst, int N, int H, int W, int C,
                      const float* mean, const float* stdv, const int32_t* aug,
                      int out_dtype, int out_layout, int n_begin, int n_end) {
    if (N < 0 || H < 1 || W < 1 || C < 1 || C > 4) return -1;
    if (out_dtype != ORACLE_OUT_F32 && out_dtype != ORACLE_OUT_F16) return -1;
    if (out_layout != ORACLE_LAYOUT_NHWC && out_layout != ORACLE_LAYOUT_NCHW &&
        out_layout != ORACLE_LAYOUT_NHWC4) return -1;
    if (n_begin < 0) n_begin = 0;
    if (n_end > N) n_end = N;

    float* d32 = (float*)dst;
    uint16_t* d16 = (uint16_t*)dst;
    const int out_ch = (out_layout == ORACLE_LAYOUT_NHWC4) ? 4 : C;

    for (int n = n_begin; n < n_end; ++n) {
        int flip = 0;
        long long ey0 = 0, ex0 = 0, eh = 0, ew = 0;
        if (aug != NULL) {
            const int32_t* a = aug + (size_t)n * 5;
            flip = (a[0] != 0);
            ey0 = a[1]; ex0 = a[2]; eh = a[3]; ew = a[4];
        }
        const int has_erase = (eh > 0 && ew > 0);
        for (int y = 0; y < H; ++y) {
            for (int x = 0; x < W; ++x) {
                const int erased = has_erase && y >= ey0 && y < ey0 + eh &&
                                   x >= ex0 && x < ex0 + ew;
                const int xs = flip ? (W - 1 - x) : x;   /* mirrored read */
                for (int c = 0; c < out_ch; ++c) {
                    float v32;
                    if (c >= C || erased) {
                        v32 = 0.0f;
                    } else {
                        uint8_t u = src[(((size_t)n * H + y) * W + xs) * C + c];
                        double r = ((double)u / 255.0 - (double)mean[c]) / (double)stdv[c];
                        v32 = (float)r;
                    }
                    size_t o;
                    if (out_layout == ORACLE_LAYOUT_NCHW)
                        o = (((size_t)n * C + c) * H + y) * W + x;
                    else
                        o = (((size_t)n * H + y) * W + x) * out_ch + c;
                    if (out_dtype == ORACLE_OUT_F32) d32[o] = v32;
                    else d16[o] = oracle_f32_to_f16(v32);
                }
            }
        }
    }
    return 0;
}

/* The same step on windows of a larger, possibly strided, source: output
 * pixel (n, y, x) reads source pixel (n, cy_n + y, cx_n + x') with x' the
 * (possibly mirrored) column inside the H x W window, i.e. a crop followed by
 * the fused step (the article's execute() takes an input stride, §五; the
 * crop is the one upstream of it, §一).  Source byte (n, sy, sx, c) is at
 * src[n*image_stride + sy*row_stride + sx*C + c].  crop: N pairs {cy, cx}
 * (NULL = all zero); a window must lie inside the src_H x src_W image.
 * Returns -1 for windows outside the source or bad strides.                */
int oracle_fused_norm_crop(const uint8_t* src, size_t image_stride, size_t row_stride, int src_H, int src_W,
                           const int32_t* crop, void* dst, int N, int H, int W, int C,
                           const float* mean, const float* stdv, const int32_t* aug,
                           int out_dtype, int out_layout, int n_begin, int n_end) {
    if (N < 0 || H < 1 || W < 1 || C < 1 || C > 4 || src_H < H || src_W < W) return -1;
    if (row_stride < (size_t)src_W * C || image_stride < (size_t)(src_H - 1) * row_stride + (size_t)src_W * C)
        return -1;
    if (out_dtype != ORACLE_OUT_F32 && out_dtype != ORACLE_OUT_F16) return -1;
    if (out_layout != ORACLE_LAYOUT_NHWC && out_layout != ORACLE_LAYOUT_NCHW &&
        out_layout != ORACLE_LAYOUT_NHWC4) return -1;
    if (n_begin < 0) n_begin = 0;
    if (n_end > N) n_end = N;
    float* d32 = (float*)dst;
    uint16_t* d16 = (uint16_t*)dst;
    const int out_ch = (out_layout == ORACLE_LAYOUT_NHWC4) ? 4 : C;
    for (int n = n_begin; n < n_end; ++n) {
        const long long cy = crop ? crop[2 * (size_t)n] : 0;
        const long long cx = crop ? crop[2 * (size_t)n + 1] : 0;
        if (cy < 0 || cx < 0 || cy + H > src_H || cx + W > src_W) return -1;
        int flip = 0;
        long long ey0 = 0, ex0 = 0, eh = 0, ew = 0;
        if (aug != NULL) {
            const int32_t* a = aug + (size_t)n * 5;
            flip = (a[0] != 0);
            ey0 = a[1]; ex0 = a[2]; eh = a[3]; ew = a[4];
        }
        const int has_erase = (eh > 0 && ew > 0);
        for (int y = 0; y < H; ++y) {
            for (int x = 0; x < W; ++x) {
                const int erased = has_erase && y >= ey0 && y < ey0 + eh && x >= ex0 && x < ex0 + ew;
                const int xs = flip ? (W - 1 - x) : x;
                for (int c = 0; c < out_ch; ++c) {
                    float v32;
                    if (c >= C || erased) {
                        v32 = 0.0f;
                    } else {
                        const uint8_t u = src[(size_t)n * image_stride + (size_t)(cy + y) * row_stride +
                                              (size_t)(cx + xs) * C + c];
                        double r = ((double)u / 255.0 - (double)mean[c]) / (double)stdv[c];
                        v32 = (float)r;
                    }
                    size_t o;
                    if (out_layout == ORACLE_LAYOUT_NCHW)
                        o = (((size_t)n * C + c) * H + y) * W + x;
                    else
                        o = (((size_t)n * H + y) * W + x) * out_ch + c;
                    if (out_dtype == ORACLE_OUT_F32) d32[o] = v32;
                    else d16[o] = oracle_f32_to_f16(v32);
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with the
 * round key bumped by the Weyl constants between rounds.                    */
static void philox_round(uint32_t ctr[4], const uint32_t key[2]) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * ctr[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * ctr[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t out[4];
    out[0] = hi1 ^ ctr[1] ^ key[0];
    out[1] = lo1;
    out[2] = hi0 ^ ctr[3] ^ key[1];
    out[3] = lo0;
    memcpy(ctr, out, sizeof out);
}

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t ctr[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint32_t key[2] = {key_in[0], key_in[1]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            key[0] += 0x9E3779B9u;
            key[1] += 0xBB67AE85u;
        }
        philox_round(ctr, key);
    }
    memcpy(out, ctr, sizeof ctr);
}

/* The generator behind the article's uniform()/randint() (§十
 * "Reproducible random decisions"): one Philox value per (seed, offset).
 * Reading (the article defers the mapping to a later post that is not
 * available): key = the 64-bit seed split into two 32-bit words (low first),
 * counter = the 64-bit offset in words 0-1, words 2-3 zero; the first output
 * word w gives k = w >> 8, a 24-bit integer.                                */
static uint32_t philox_bits24(uint64_t seed, uint64_t offset) {
    uint32_t ctr[4] = {(uint32_t)offset, (uint32_t)(offset >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[0] >> 8;
}

/* u in [0,1): k * 2^-24, exact in binary32 */
float oracle_uniform01(uint64_t seed, uint64_t offset) {
    return (float)philox_bits24(seed, offset) * (1.0f / 16777216.0f);
}

/* Sampler state: a seed and the next unused offset (one offset per draw). */
typedef struct { uint64_t seed; uint64_t offset; } oracle_rng;

static float rng_uniform(oracle_rng* g, float lo, float hi) {
    float u = oracle_uniform01(g->seed, g->offset);
    g->offset += 1;
    return lo + u * (hi - lo);
}

/* Integer draw in [lo, hi] inclusive.  Reading: lo + floor(u * (hi-lo+1))
 * with u the 24-bit fraction above, computed exactly in integers.           */
static int rng_randint(oracle_rng* g, int lo, int hi) {
    uint32_t k = philox_bits24(g->seed, g->offset);
    g->offset += 1;
    uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
    return (int)((int64_t)lo + (int64_t)(((uint64_t)k * span) >> 24));
}

/* Per-image augmentation decisions (article §五 execute() and §十二
 * generate_erase_rect): a flip draw when flipping is enabled (flip iff
 * u < flip_p; the article hard-codes 0.5), then, when erasing is enabled and
 * p > 0, a gate draw (skip unless u < p) and up to ten attempts of
 *   area   = (scale_lo + u*(scale_hi - scale_lo)) * H * W
 *   aspect = exp(log(ratio_lo) + u*(log(ratio_hi) - log(ratio_lo)))
 *   eh = round(sqrt(area*aspect)), ew = round(sqrt(area/aspect))
 * accepted when 0 < eh < H and 0 < ew < W, followed by y0 = randint(0, H-eh)
 * and x0 = randint(0, W-ew).  All of it in binary32 as the article writes it.
 * out: N records {flip, y0, x0, h, w}; h = w = 0 when there is no erase.
 * Returns the next unused offset through *next_offset.                      */
int oracle_sample_aug_params(uint64_t seed, uint64_t offset, int N, int H, int W,
                             int flip_enabled, float flip_p,
                             int erase_enabled, float erase_p,
                             float scale_lo, float scale_hi,
                             float ratio_lo, float ratio_hi,
                             int32_t* out, uint64_t* next_offset) {
    if (N < 0 || H < 1 || W < 1) return -1;
    oracle_rng g = {seed, offset};
    const float log_lo = logf(ratio_lo);
    const float log_hi = logf(ratio_hi);
    const float img_area = (float)H * (float)W;
    for (int n = 0; n < N; ++n) {
        int32_t* a = out + (size_t)n * 5;
        a[0] = 0; a[1] = 0; a[2] = 0; a[3] = 0; a[4] = 0;
        if (flip_enabled) a[0] = (rng_uniform(&g, 0.0f, 1.0f) < flip_p) ? 1 : 0;
        if (!erase_enabled || erase_p <= 0.0f) continue;
        if (rng_uniform(&g, 0.0f, 1.0f) >= erase_p) continue;
        for (int attempt = 0; attempt < 10; ++attempt) {
            float ratio = scale_lo + rng_uniform(&g, 0.0f, 1.0f) * (scale_hi - scale_lo);
            float area = ratio * img_area;
            float log_ar = log_lo + rng_uniform(&g, 0.0f, 1.0f) * (log_hi - log_lo);
            float ar = expf(log_ar);
            int eh = (int)roundf(sqrtf(area * ar));
            int ew = (int)roundf(sqrtf(area / ar));
            if (eh > 0 && ew > 0 && eh < H && ew < W) {
                a[1] = rng_randint(&g, 0, H - eh);
                a[2] = rng_randint(&g, 0, W - ew);
                a[3] = eh;
                a[4] = ew;
                break;
            }
        }
    }
    if (next_offset) *next_offset = g.offset;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Record sampling with one counter block per image, the form a GPU thread
 * per image can produce: image n's draws use offsets offset + 24n + k,
 * k < 24 (a flip draw, a gate draw, ten attempts of two draws, two origin
 * draws: at most 24).  The decisions are those of oracle_sample_aug_params;
 * only the offset of each draw differs.
 *
 * exp of the log-aspect draw uses this file's own exp (below), written so that
 * every step is a correctly rounded IEEE operation (multiply, add, fma, rint,
 * exact scaling by 2^k): any implementation that takes the same steps gets
 * the same bits, so the integer rectangle sizes cannot differ by a libm's
 * last-place choice.                                                        */

/* e^x for |x| < 80: Cody–Waite reduction x = k ln2 + r with ln2 split into a
 * 24-bit head whose products with |k| < 2^9 are exact and a tail, |r| <= ln2/2,
 * then the degree-7 Taylor polynomial of e^r (truncation below 5e-9 relative)
 * in Horner form with fused multiply-adds, then multiplication by 2^k.     */
float oracle_exp_f32(float x) {
    const float inv_ln2 = 1.44269504088896341f;
    const float ln2_hi = 0.693145751953125f;      /* 0x3f317200 */
    const float ln2_lo = 1.42860682030941723212e-6f;
    const float k = rintf(x * inv_ln2);
    float r = fmaf(-k, ln2_hi, x);
    r = fmaf(-k, ln2_lo, r);
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    uint32_t bits = (uint32_t)((int)k + 127) << 23;   /* 2^k, a normal number for |k| < 126 */
    float two_k;
    memcpy(&two_k, &bits, sizeof two_k);
    return p * two_k;
}

void oracle_exp_f32_array(const float* in, float* out, size_t n) {
    for (size_t i = 0; i < n; ++i) out[i] = oracle_exp_f32(in[i]);
}

#define ORACLE_DRAWS_PER_IMAGE 24

static float block_uniform(uint64_t seed, uint64_t base, int* k) {
    float u = oracle_uniform01(seed, base + (uint64_t)(*k));
    *k += 1;
    return u;
}

int oracle_sample_aug_params_blocked(uint64_t seed, uint64_t offset, int N, int H, int W,
                                     int flip_enabled, float flip_p,
                                     int erase_enabled, float erase_p,
                                     float scale_lo, float scale_hi,
                                     float ratio_lo, float ratio_hi,
                                     int32_t* out, uint64_t* next_offset) {
    if (N < 0 || H < 1 || W < 1) return -1;
    const float log_lo = logf(ratio_lo);
    const float log_hi = logf(ratio_hi);
    const float img_area = (float)H * (float)W;
    for (int n = 0; n < N; ++n) {
        const uint64_t base = offset + (uint64_t)n * ORACLE_DRAWS_PER_IMAGE;
        int k = 0;
        int32_t* a = out + (size_t)n * 5;
        a[0] = 0; a[1] = 0; a[2] = 0; a[3] = 0; a[4] = 0;
        if (flip_enabled) a[0] = (block_uniform(seed, base, &k) < flip_p) ? 1 : 0;
        if (!erase_enabled || erase_p <= 0.0f) continue;
        if (block_uniform(seed, base, &k) >= erase_p) continue;
        for (int attempt = 0; attempt < 10; ++attempt) {
            float ratio = scale_lo + block_uniform(seed, base, &k) * (scale_hi - scale_lo);
            float area = ratio * img_area;
            float log_ar = log_lo + block_uniform(seed, base, &k) * (log_hi - log_lo);
            float ar = oracle_exp_f32(log_ar);
            int eh = (int)roundf(sqrtf(area * ar));
            int ew = (int)roundf(sqrtf(area / ar));
            if (eh > 0 && ew > 0 && eh < H && ew < W) {
                /* integer draw in [lo, hi]: lo + floor(u * (hi - lo + 1)), exact */
                uint32_t ky = philox_bits24(seed, base + (uint64_t)k); k += 1;
                uint32_t kx = philox_bits24(seed, base + (uint64_t)k); k += 1;
                a[1] = (int32_t)(((uint64_t)ky * (uint64_t)(H - eh + 1)) >> 24);
                a[2] = (int32_t)(((uint64_t)kx * (uint64_t)(W - ew + 1)) >> 24);
                a[3] = eh;
                a[4] = ew;
                break;
            }
        }
    }
    if (next_offset) *next_offset = offset + (uint64_t)N * ORACLE_DRAWS_PER_IMAGE;
    return 0;
}

// Per-image augmentation decisions on the GPU, from one thread or from one
// warp (the 24 counter words computed in parallel).
//
// The decisions are those of the FusedNormalization article
// (tech-renaissance.cn/blog/?p=487): the flip draw of execute() (§五),
// uniform() and randint() over a counter-based Philox generator (§十) and
// generate_erase_rect() (§十二).  Image n draws from its own counter block,
// offsets offset + 24n + k (a flip draw, a gate draw, ten attempts of two
// draws and two origin draws are at most 24).  Every floating-point step is a
// correctly rounded IEEE operation written out with an intrinsic (no
// contraction), and exp is computed by the steps below rather than by a math
// library, so a CPU that takes the same steps makes the same records bit for
// bit.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace trfn {

constexpr int kDrawsPerImage = 24;

// Philox4x32-10 (Salmon et al., SC'11): first output word for (seed, counter).
__device__ __forceinline__ uint32_t philox_word0(uint64_t seed, uint64_t ctr) {
    uint32_t x0 = (uint32_t)ctr, x1 = (uint32_t)(ctr >> 32), x2 = 0u, x3 = 0u;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, x0), lo0 = 0xD2511F53u * x0;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, x2), lo1 = 0xCD9E8D57u * x2;
        const uint32_t y0 = hi1 ^ x1 ^ k0, y2 = hi0 ^ x3 ^ k1;
        x0 = y0; x1 = lo1; x2 = y2; x3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return x0;
}

// e^x: Cody–Waite reduction x = k ln2 + r (ln2 as a 24-bit head, exact in
// products with |k| < 2^9, plus a tail), the degree-7 Taylor polynomial of
// e^r in Horner form with fused multiply-adds, then scaling by 2^k.
__device__ __forceinline__ float exp_steps(float x) {
    const float k = rintf(__fmul_rn(x, 1.44269504088896341f));
    float r = __fmaf_rn(-k, 0.693145751953125f, x);
    r = __fmaf_rn(-k, 1.42860682030941723212e-6f, r);
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float(((int)k + 127) << 23));
}

// One image's record from its draws; draw24() returns the next draw's 24-bit
// value (first Philox word >> 8), in counter order.
template <class Draw>
__device__ __forceinline__ tr_aug_param decide_record(const SampleSpec& sp, Draw&& draw24) {
    auto uniform = [&]() { return __fmul_rn((float)draw24(), 5.9604644775390625e-8f); };   // k * 2^-24
    tr_aug_param a = {0, 0, 0, 0, 0};
    if (sp.flip_enabled) a.flip = (uniform() < sp.flip_p) ? 1 : 0;
    if (sp.erase && uniform() < sp.erase_p) {
        const float area_img = __fmul_rn((float)sp.H, (float)sp.W);
        const float scale_span = __fsub_rn(sp.scale_hi, sp.scale_lo);
        const float log_span = __fsub_rn(sp.log_hi, sp.log_lo);
        for (int attempt = 0; attempt < 10; ++attempt) {
            const float frac = __fadd_rn(sp.scale_lo, __fmul_rn(uniform(), scale_span));
            const float area = __fmul_rn(frac, area_img);
            const float ar = exp_steps(__fadd_rn(sp.log_lo, __fmul_rn(uniform(), log_span)));
            const int h = (int)roundf(__fsqrt_rn(__fmul_rn(area, ar)));
            const int w = (int)roundf(__fsqrt_rn(__fdiv_rn(area, ar)));
            if (h > 0 && w > 0 && h < sp.H && w < sp.W) {
                const uint64_t ky = draw24(), kx = draw24();
                a.y0 = (int)((ky * (uint64_t)(sp.H - h + 1)) >> 24);
                a.x0 = (int)((kx * (uint64_t)(sp.W - w + 1)) >> 24);
                a.h = h;
                a.w = w;
                break;
            }
        }
    }
    return a;
}

// Image n's record from one thread: draws computed one at a time, in order.
__device__ __forceinline__ tr_aug_param sample_record(const SampleSpec& sp, int n) {
    const uint64_t base = sp.offset + (uint64_t)n * kDrawsPerImage;
    int k = 0;
    return decide_record(sp, [&]() { return philox_word0(sp.seed, base + (uint64_t)(k++)) >> 8; });
}

// Image n's record from a whole warp (every lane calls it, lane = lane index):
// lane k computes draw k, and the decisions run on every lane alike with the
// draws taken by shuffles, so the warp stays converged.  Same result as
// sample_record.
__device__ __forceinline__ tr_aug_param sample_record_warp(const SampleSpec& sp, int n, int lane) {
    const uint64_t base = sp.offset + (uint64_t)n * kDrawsPerImage;
    const uint32_t mine = lane < kDrawsPerImage ? philox_word0(sp.seed, base + (uint64_t)lane) >> 8 : 0u;
    int k = 0;
    return decide_record(sp, [&]() { return __shfl_sync(0xffffffffu, mine, k++); });
}

}  // namespace trfn

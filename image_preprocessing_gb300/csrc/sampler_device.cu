// On-device sampling of the per-image augmentation records: one thread per
// image, so the records of a batch are made where the fused kernel reads them
// and need no upload.
//
// The decisions are those of the host sampler (FusedNormalization article,
// tech-renaissance.cn/blog/?p=487: the flip draw of execute(), §五; uniform()
// and randint() over a counter-based Philox generator, §十;
// generate_erase_rect(), §十二), but image n draws from its own counter block,
// offsets offset + 24n + k (a flip draw, a gate draw, ten attempts of two
// draws and two origin draws are at most 24).  Every floating-point step is a
// correctly rounded IEEE operation written out with an intrinsic (no
// contraction), and exp is computed by the steps below rather than by a math
// library, so a CPU that takes the same steps makes the same records bit for
// bit.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace trfn {
namespace {

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

struct SampleParams {
    uint64_t seed, offset;
    int N, H, W;
    int flip_enabled, erase;
    float flip_p, erase_p, scale_lo, scale_hi, log_lo, log_hi;
    tr_aug_param* out;
};

__global__ void __launch_bounds__(128) sample_kernel(const __grid_constant__ SampleParams p) {
    // launched with programmatic stream serialization: the records buffer may
    // still be read by the previous kernel in the stream, so wait for it
    // before writing, and let the next kernel start its prologue right away
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= p.N) return;
    const uint64_t base = p.offset + (uint64_t)n * kDrawsPerImage;
    int k = 0;
    auto draw24 = [&]() { return philox_word0(p.seed, base + (uint64_t)(k++)) >> 8; };
    auto uniform = [&]() { return __fmul_rn((float)draw24(), 5.9604644775390625e-8f); };   // k * 2^-24
    tr_aug_param a = {0, 0, 0, 0, 0};
    if (p.flip_enabled) a.flip = (uniform() < p.flip_p) ? 1 : 0;
    if (p.erase && uniform() < p.erase_p) {
        const float area_img = __fmul_rn((float)p.H, (float)p.W);
        const float scale_span = __fsub_rn(p.scale_hi, p.scale_lo);
        const float log_span = __fsub_rn(p.log_hi, p.log_lo);
        for (int attempt = 0; attempt < 10; ++attempt) {
            const float frac = __fadd_rn(p.scale_lo, __fmul_rn(uniform(), scale_span));
            const float area = __fmul_rn(frac, area_img);
            const float ar = exp_steps(__fadd_rn(p.log_lo, __fmul_rn(uniform(), log_span)));
            const int h = (int)roundf(__fsqrt_rn(__fmul_rn(area, ar)));
            const int w = (int)roundf(__fsqrt_rn(__fdiv_rn(area, ar)));
            if (h > 0 && w > 0 && h < p.H && w < p.W) {
                const uint64_t ky = draw24(), kx = draw24();
                a.y0 = (int)((ky * (uint64_t)(p.H - h + 1)) >> 24);
                a.x0 = (int)((kx * (uint64_t)(p.W - w + 1)) >> 24);
                a.h = h;
                a.w = w;
                break;
            }
        }
    }
    p.out[n] = a;
}

}  // namespace
}  // namespace trfn

extern "C" int tr_sample_aug_params_device(uint64_t seed, uint64_t offset, int N, int H, int W,
                                           int flip_enabled, float flip_p, int erase_enabled, float erase_p,
                                           float scale_lo, float scale_hi, float ratio_lo, float ratio_hi,
                                           tr_aug_param* d_out, uint64_t* next_offset, void* stream) {
    using namespace trfn;
    if (N < 0 || H < 1 || W < 1) return TR_ERR_INVALID_ARGUMENT;
    if (N > 0 && (d_out == nullptr || ((uintptr_t)d_out % 4u) != 0)) return TR_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(flip_p) || !std::isfinite(erase_p)) return TR_ERR_INVALID_ARGUMENT;
    const bool erase = erase_enabled && erase_p > 0.0f;
    if (erase && (!std::isfinite(scale_lo) || !std::isfinite(scale_hi) || !std::isfinite(ratio_lo) ||
                  !std::isfinite(ratio_hi) || scale_lo > scale_hi || ratio_lo <= 0.0f || ratio_lo > ratio_hi))
        return TR_ERR_INVALID_ARGUMENT;
    if (next_offset) *next_offset = offset + (uint64_t)N * kDrawsPerImage;
    if (N == 0) return TR_OK;
    SampleParams p;
    p.seed = seed;
    p.offset = offset;
    p.N = N; p.H = H; p.W = W;
    p.flip_enabled = flip_enabled ? 1 : 0;
    p.erase = erase ? 1 : 0;
    p.flip_p = flip_p;
    p.erase_p = erase_p;
    p.scale_lo = scale_lo;
    p.scale_hi = scale_hi;
    // the bounds' logarithms are taken once, on the host
    p.log_lo = erase ? std::log(ratio_lo) : 0.0f;
    p.log_hi = erase ? std::log(ratio_hi) : 0.0f;
    p.out = d_out;
    const int threads = 128;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((N + threads - 1) / threads));
    cfg.blockDim = dim3(threads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, sample_kernel, p);
    if (e != cudaSuccess) {
        set_last_error("sample kernel launch", (int)e);
        return TR_ERR_CUDA;
    }
    count_launch();
    return TR_OK;
}

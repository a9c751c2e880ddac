// On-device sampling of the per-image augmentation records (a warp or a
// thread per image), so the records of a batch are made where the fused
// kernel reads them and need no upload.  The decisions and their bit-exact
// arithmetic are in aug_sampling.cuh.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "aug_sampling.cuh"
#include "internal.h"

namespace trfn {
namespace {

// Launched with programmatic stream serialization.  Normally the records
// buffer may still be read by the previous kernel in the stream, so the
// kernel waits for it before writing and then lets the next kernel start.
// With `overlap` the caller has promised that the previous kernel does not
// use the records buffer: the kernel lets the next one start and writes at
// once, and waits for the previous kernel only before it exits, so it still
// completes after it (the fused kernel that reads these records waits for
// this one, hence for both).
__device__ __forceinline__ void sampler_enter(int overlap) {
    if (!overlap) asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void sampler_leave(int overlap) {
    if (overlap) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// One thread per image: for batches too large for a warp each in one wave.
__global__ void __launch_bounds__(128) sample_kernel(const __grid_constant__ SampleSpec sp, int N,
                                                     tr_aug_param* out, int overlap) {
    sampler_enter(overlap);
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n < N) out[n] = sample_record(sp, n);
    sampler_leave(overlap);
}

// One warp per image: lane k computes the image's draw k, so a record costs
// one Philox evaluation of latency instead of one per draw.
__global__ void __launch_bounds__(128) sample_kernel_warp(const __grid_constant__ SampleSpec sp, int N,
                                                          tr_aug_param* out, int overlap) {
    sampler_enter(overlap);
    const int n = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (n < N) {   // whole warps take the same branch
        const tr_aug_param a = sample_record_warp(sp, n, lane);
        if (lane == 0) out[n] = a;
    }
    sampler_leave(overlap);
}

}  // namespace

int make_sample_spec(uint64_t seed, uint64_t offset, int H, int W, int flip_enabled, float flip_p,
                     int erase_enabled, float erase_p, float scale_lo, float scale_hi, float ratio_lo,
                     float ratio_hi, SampleSpec* sp) {
    if (H < 1 || W < 1) return TR_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(flip_p) || !std::isfinite(erase_p)) return TR_ERR_INVALID_ARGUMENT;
    const bool erase = erase_enabled && erase_p > 0.0f;
    if (erase && (!std::isfinite(scale_lo) || !std::isfinite(scale_hi) || !std::isfinite(ratio_lo) ||
                  !std::isfinite(ratio_hi) || scale_lo > scale_hi || ratio_lo <= 0.0f || ratio_lo > ratio_hi))
        return TR_ERR_INVALID_ARGUMENT;
    sp->seed = seed;
    sp->offset = offset;
    sp->H = H;
    sp->W = W;
    sp->flip_enabled = flip_enabled ? 1 : 0;
    sp->erase = erase ? 1 : 0;
    sp->flip_p = flip_p;
    sp->erase_p = erase_p;
    sp->scale_lo = scale_lo;
    sp->scale_hi = scale_hi;
    // the bounds' logarithms are taken once, on the host
    sp->log_lo = erase ? std::log(ratio_lo) : 0.0f;
    sp->log_hi = erase ? std::log(ratio_hi) : 0.0f;
    return TR_OK;
}

int launch_sampler(const SampleSpec& sp, int N, tr_aug_param* d_out, void* stream, bool overlap) {
    if (N == 0) return TR_OK;
    // A warp per image for small batches (shortest latency: 1.3 us for 256
    // images against 1.6 us), a thread per image beyond (a warp per image
    // repeats the decisions on 32 lanes: 2.0 us for 4,096 images, 16.8 us
    // for 65,536, against 1.9 and 2.7 us).  Measured on GB300.
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        set_last_error("cudaDeviceGetAttribute", (int)cudaGetLastError());
        return TR_ERR_CUDA;
    }
    const bool per_warp = (long long)N <= (long long)sms * 8;
    const int threads = 128;
    cudaLaunchConfig_t cfg = {};
    const long long total_threads = per_warp ? (long long)N * 32 : (long long)N;
    cfg.gridDim = dim3((unsigned)((total_threads + threads - 1) / threads));
    cfg.blockDim = dim3(threads);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int ov = overlap ? 1 : 0;
    const cudaError_t e = per_warp ? cudaLaunchKernelEx(&cfg, sample_kernel_warp, sp, N, d_out, ov)
                                   : cudaLaunchKernelEx(&cfg, sample_kernel, sp, N, d_out, ov);
    if (e != cudaSuccess) {
        set_last_error("sample kernel launch", (int)e);
        return TR_ERR_CUDA;
    }
    count_launch();
    return TR_OK;
}

}  // namespace trfn

extern "C" int tr_sample_aug_params_device(uint64_t seed, uint64_t offset, int N, int H, int W,
                                           int flip_enabled, float flip_p, int erase_enabled, float erase_p,
                                           float scale_lo, float scale_hi, float ratio_lo, float ratio_hi,
                                           tr_aug_param* d_out, uint64_t* next_offset, void* stream) {
    using namespace trfn;
    if (N < 0) return TR_ERR_INVALID_ARGUMENT;
    if (N > 0 && (d_out == nullptr || ((uintptr_t)d_out % 4u) != 0)) return TR_ERR_INVALID_ARGUMENT;
    SampleSpec sp;
    const int rc = make_sample_spec(seed, offset, H, W, flip_enabled, flip_p, erase_enabled, erase_p, scale_lo,
                                    scale_hi, ratio_lo, ratio_hi, &sp);
    if (rc != TR_OK) return rc;
    if (next_offset) *next_offset = offset + (uint64_t)N * kDrawsPerImage;
    return launch_sampler(sp, N, d_out, stream);
}

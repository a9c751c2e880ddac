// tr_fused_norm_noalloc: the dynamically scheduled fused normalisation for
// callers that cannot allocate device memory.
//
// tr_fused_norm_ws needs a small zeroed scratch buffer (its band-scheduling
// counters) that the caller allocates.  Some callers cannot do that: a
// program whose device memory is laid out once by a fixed memory plan and
// may not allocate afterwards, a data-loader thread that must never wait on
// the device-wide synchronisation cudaFree implies, or a plug-in that runs
// inside a host application and has no access to its allocator.  This entry
// point serves them with scratch that lives in this library's own module
// memory instead: a file-scope __device__ array that every GPU loading the
// library holds until the process exits.  The call itself allocates nothing
// (no cudaMalloc, no cudaFree, no allocating library routine).
//
// All calls on a device share that one array.  Each call clears the part it
// uses on its stream before the kernel runs, and the kernel leaves it zero
// when it finishes; calls that overlap on the GPU (other streams, other
// threads) would share the counters and race, so they must be ordered.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace {

// Capacity of the module scratch: one scheduling workspace.  Every shape the
// tiled kernel accepts needs exactly tr_workspace_bytes() of it.
constexpr size_t kNoAllocScratchBytes = 2048;

static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoAllocScratchBytes / sizeof(unsigned int)];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on `dev` (made current by the caller).
// In host code the array's name is only a host-side stand-in, so the address
// is looked up once per device with cudaGetSymbolAddress and cached.  The
// cache is never refreshed: a device reset (cudaDeviceReset) or a teardown of
// the primary context while the process keeps running is not supported.
int scratch_address(int dev, void** out) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return TR_ERR_NOT_SUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            trfn::set_last_error("cudaGetSymbolAddress(no-alloc scratch)", (int)e);
            return TR_ERR_CUDA;
        }
        addr[dev] = p;
    }
    *out = addr[dev];
    return TR_OK;
}

}  // namespace

extern "C" int tr_fused_norm_noalloc(const uint8_t* src_u8, void* dst, int N, int H, int W, int C,
                                     const float* mean, const float* std,
                                     const tr_aug_param* aug_params, int out_dtype, int out_layout,
                                     void* stream) {
    // Host checks first (shape, type, layout, constants; then pointers), so
    // that a rejected call touches neither the GPU nor the shared scratch.
    int rc = tr_fused_norm_ws(src_u8, dst, 0, H, W, C, mean, std, nullptr, out_dtype, out_layout,
                              stream, TR_VARIANT_AUTO, nullptr);
    if (rc != TR_OK) return rc;
    if (N < 0) return TR_ERR_INVALID_ARGUMENT;
    if (N == 0) return TR_OK;
    if (src_u8 == nullptr || dst == nullptr) return TR_ERR_INVALID_ARGUMENT;
    const size_t ob = (out_dtype == TR_OUT_F16) ? 2 : 4;
    if (((uintptr_t)dst % ob) != 0) return TR_ERR_INVALID_ARGUMENT;
    if (aug_params != nullptr && ((uintptr_t)aug_params % 4u) != 0) return TR_ERR_INVALID_ARGUMENT;
    const size_t out_ch = (out_layout == TR_LAYOUT_NHWC4) ? 4 : (size_t)C;
    const uintptr_t s0 = (uintptr_t)src_u8, d0 = (uintptr_t)dst;
    const size_t in_bytes = (size_t)N * H * W * C, out_bytes = (size_t)N * H * W * out_ch * ob;
    if (s0 < d0 + out_bytes && d0 < s0 + in_bytes) return TR_ERR_INVALID_ARGUMENT;
    const size_t need = tr_workspace_bytes();
    if (need > kNoAllocScratchBytes) {
        // the kernel's scheduling state would not fit the module scratch
        trfn::set_last_error("tr_fused_norm_noalloc: scratch needed exceeds its 2048-byte capacity",
                             (int)cudaErrorInvalidValue);
        return TR_ERR_NOT_SUPPORTED;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        trfn::set_last_error("cudaGetDevice", (int)e);
        return TR_ERR_CUDA;
    }
    void* scratch = nullptr;
    rc = scratch_address(dev, &scratch);
    if (rc != TR_OK) return rc;
    // only the tiled kernel reads the counters; the per-element kernel (small
    // batches, unaligned buffers) ignores them, so it needs no clearing
    int variant = TR_VARIANT_TILED;
    rc = tr_fused_norm_plan(src_u8, dst, N, H, W, C, out_dtype, out_layout, &variant);
    if (rc != TR_OK) return rc;
    if (variant != TR_VARIANT_TILED)
        return tr_fused_norm_ws(src_u8, dst, N, H, W, C, mean, std, aug_params, out_dtype, out_layout,
                                stream, TR_VARIANT_GENERIC, nullptr);
    // the counters must start at zero: clear them in stream order
    e = cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        trfn::set_last_error("cudaMemsetAsync(no-alloc scratch)", (int)e);
        return TR_ERR_CUDA;
    }
    return tr_fused_norm_ws(src_u8, dst, N, H, W, C, mean, std, aug_params, out_dtype, out_layout,
                            stream, TR_VARIANT_TILED, scratch);
}

// Internal declarations shared by the library's translation units (not part
// of the C ABI; see include/tr_fused_norm.h for that).
#pragma once

#include <cstddef>
#include <cstdint>

#include "tr_fused_norm.h"

namespace trfn {

// Settings of the per-image record sampler (tr_sample_aug_params_device and
// the sampled fused kernel); log_lo/log_hi are log(ratio_lo)/log(ratio_hi),
// taken once on the host.
struct SampleSpec {
    uint64_t seed = 0, offset = 0;
    int H = 0, W = 0;
    int flip_enabled = 0, erase = 0;
    float flip_p = 0.0f, erase_p = 0.0f, scale_lo = 0.0f, scale_hi = 0.0f, log_lo = 0.0f, log_hi = 0.0f;
};

// Arguments of one fused-normalisation launch after host validation.
struct LaunchArgs {
    const uint8_t* src;
    void* dst;
    int N, H, W, C;
    // value = (x - 255*mean_c) / (255*std_c), evaluated as
    // fma(x - shift_c, scale_c, bias_c): shift_c is 255*mean_c rounded to an
    // integer (0 when that is beyond 2^20), so x - shift_c is exact, and
    // bias_c carries only the remainder; the map's terms then stay near the
    // value itself instead of cancelling (255*mean_c = 123.68 would otherwise
    // leave binary32 rounding errors of ulp(124) on values near 0)
    float shift[4];   // integer-valued
    float scale[4];   // 1/(255*std_c), formed in binary64, rounded to binary32
    float bias[4];    // -(255*mean_c - shift_c)*scale_c, formed in binary64, rounded once
    const tr_aug_param* aug;
    int out_dtype;
    int out_layout;
    void* stream;
    void* workspace;  // scheduling workspace (tr_workspace_bytes(), zeroed), or null
    // the launch shares no buffer with the kernel before it in the stream:
    // the tiled kernel may start its copies while that kernel drains
    bool overlap_prev = false;
    // the records were just written by the previous kernel in the stream (the
    // device sampler): with overlap_prev the tiled kernel requests its first
    // bands before that kernel has completed and reads the records after
    bool records_from_prev = false;
    // records to be made on the GPU (tr_fused_norm_sampled): the sampler's
    // settings and the N records' destination; launch() runs the sampler
    // first and the kernel on its output (records_from_prev), an overlapped
    // tiled launch making its CTAs' first records itself (sample_in_kernel)
    const SampleSpec* spec = nullptr;
    tr_aug_param* records_out = nullptr;
    bool sample_in_kernel = false;
    // windows of a strided source (tr_fused_norm_crop); otherwise a compact
    // NHWC source of H x W images
    bool crop_src = false;
    const int32_t* crop = nullptr;
    int src_H = 0, src_W = 0;
    size_t src_row_stride = 0, src_image_stride = 0;
    // several batches in one tiled launch (tr_fused_norm_batches): N counts
    // the images of all batches, batch_images those of one, and image n is
    // image n % batch_images of batch n / batch_images (src, dst and aug are
    // then batch 0's); 0 = one batch
    int batch_images = 0;
    const uint8_t* bsrc[TR_MAX_BATCHES] = {};
    void* bdst[TR_MAX_BATCHES] = {};
    const tr_aug_param* baug[TR_MAX_BATCHES] = {};
};

constexpr size_t kWorkspaceBytes = 2048;

// Fills a.shift/scale/bias for channels 0..C-1 (zeros above C); false when
// a constant is not finite or std_c is 0.
bool fold_constants(const float* mean, const float* stdv, int C, LaunchArgs& a);

// Whether the tiled kernel's aligned form applies (16-byte aligned pointers,
// rows and NCHW output rows a multiple of 16 bytes); otherwise a supported
// compact source takes its odd-row form.
bool tiled_aligned(const uint8_t* src, const void* dst, int W, int C, int f16, int out_layout);

// Whether the tiled kernel's preconditions hold for these arguments.
bool tiled_supported(const uint8_t* src, const void* dst, int N, int H, int W, int C,
                     int out_dtype, int out_layout);

// Whether the tiled kernel can read crop windows of this strided source
// through TMA tensor copies.
bool tiled_crop_supported(const uint8_t* src, const void* dst, int N, int H, int W, int C, int out_dtype,
                          int out_layout, int src_H, int src_W, size_t row_stride, size_t image_stride);

// Launches the chosen kernel (TR_VARIANT_TILED or TR_VARIANT_GENERIC) on
// a.stream.  Returns a tr_status.
int launch(const LaunchArgs& a, int variant);

// What a tiled launch with these arguments would take (host only; occupancy
// queries need the device): rows per band, shared-memory stages, threads per
// CTA, CTAs per SM, grid size, and whether the odd-row form applies.
struct TiledGeometry {
    int rows, stages, threads, ctas_per_sm, grid, odd_form;
};
int tiled_geometry(const LaunchArgs& a, TiledGeometry* g);

// Reads (and optionally clears) the device status word of the current device.
int read_device_status(int* flags, bool clear);

// Per-thread last CUDA error text.
void set_last_error(const char* what, int cuda_error);
const char* last_error();

// Tiled-kernel geometry knobs (0 = default).
void tune_tiled(int band_bytes, int stages, int ctas_per_sm, int flags);

// Record sampler (sampler_device.cu): validates the sampling settings into
// a SampleSpec (TR_ERR_INVALID_ARGUMENT as tr_sample_aug_params), and
// launches the one-thread-per-image sampler writing N records to d_out.
int make_sample_spec(uint64_t seed, uint64_t offset, int H, int W, int flip_enabled, float flip_p,
                     int erase_enabled, float erase_p, float scale_lo, float scale_hi, float ratio_lo,
                     float ratio_hi, SampleSpec* sp);
// overlap: the previous kernel in the stream does not use d_out (see
// sample_kernel); the sampler then writes at once and waits for that kernel
// only before it exits.
int launch_sampler(const SampleSpec& sp, int N, tr_aug_param* d_out, void* stream, bool overlap = false);

// Count of kernels launched by this library.
void count_launch();
uint64_t launch_count();

// Staging-area hooks for the station (staging.cpp): checks that b is a batch
// of st handed out for N images of H*W*C bytes; counts a release queued on a
// stream; and performs it (from a stream host function: no CUDA call).
int stage_batch_ok(const tr_staging* st, const tr_stage_batch* b, int N, int H, int W, int C);
void stage_release_queued(tr_staging* st);
void stage_release_from_stream(tr_staging* st, long long batch);

}  // namespace trfn

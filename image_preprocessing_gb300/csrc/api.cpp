// C ABI entry points of libtrfn.so: argument checks, folding of mean/std into
// scale/bias, kernel choice, presets and diagnostics.  Every check here runs
// on the host before anything touches the GPU.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "stream_guard.h"

namespace trfn {

namespace {
thread_local char t_last_error[256] = "";
}

void set_last_error(const char* what, int cuda_error) {
    std::snprintf(t_last_error, sizeof t_last_error, "%s: %s (%d)", what,
                  cudaGetErrorString(static_cast<cudaError_t>(cuda_error)), cuda_error);
}

const char* last_error() { return t_last_error; }

namespace {

constexpr long long kMaxElements = 1LL << 40;

// Below this many output elements the tiled kernel's fixed latency (record
// load, TMA round trip, TMA store) exceeds the per-element kernel's whole
// run: a 16 x 32x32x3 batch takes 4.5 us tiled and 2.5 us generic on GB300.
constexpr long long kSmallBatchElements = 1LL << 18;

bool small_batch(int N, int H, int W, int C, int out_layout) {
    const long long out_ch = (out_layout == TR_LAYOUT_NHWC4) ? 4 : C;
    return (long long)N * H * W * out_ch < kSmallBatchElements;
}

// Shape/type checks shared by the launch and plan entry points.
int check_shape(int N, int H, int W, int C, int out_dtype, int out_layout) {
    if (N < 0 || H < 1 || W < 1 || C < 1) return TR_ERR_INVALID_ARGUMENT;
    if (C > 4) return TR_ERR_NOT_SUPPORTED;
    if (out_dtype != TR_OUT_F32 && out_dtype != TR_OUT_F16) return TR_ERR_INVALID_ARGUMENT;
    if (out_layout != TR_LAYOUT_NHWC && out_layout != TR_LAYOUT_NCHW && out_layout != TR_LAYOUT_NHWC4)
        return TR_ERR_INVALID_ARGUMENT;
    const long long per_image = (long long)H * W;
    if (per_image > kMaxElements) return TR_ERR_INVALID_ARGUMENT;
    if (per_image * 4 * N > kMaxElements) return TR_ERR_INVALID_ARGUMENT;
    return TR_OK;
}

// A strided source read through per-image windows (tr_fused_norm_crop).
struct CropSource {
    bool on = false;
    const int32_t* crop = nullptr;
    int src_H = 0, src_W = 0;
    size_t row_stride = 0, image_stride = 0;
};

// Records drawn on the GPU as part of the launch (tr_fused_norm_sampled).
struct Sampling {
    bool on = false;
    SampleSpec spec;
    tr_aug_param* out = nullptr;   // device, N records
};

}  // namespace

// (x/255 - m)/s == (x - 255 m) * (1/(255 s)).  With A = 255 m rounded to an
// integer, x - A is an exact small integer and the rest, -(255 m - A)/(255 s),
// is at most half a scale step: every constant is formed in binary64 (255 m
// is exact there) and rounded once to binary32.  The kernels' one FMA then
// adds terms of the value's own size, so the result is within 3 binary32
// ulps of the exact value whatever the mean (the product's relative error
// is 2^-24 and |x - A| * scale <= 2 |value| when x != A), where x * scale +
// (-m/s) would cancel two terms of up to 255 * scale.
bool fold_constants(const float* mean, const float* stdv, int C, LaunchArgs& a) {
    for (int c = 0; c < 4; ++c) { a.shift[c] = 0.0f; a.scale[c] = 0.0f; a.bias[c] = 0.0f; }
    for (int c = 0; c < C; ++c) {
        const double m = mean[c], s = stdv[c];
        if (!std::isfinite(m) || !std::isfinite(s) || s == 0.0) return false;
        const double am = 255.0 * m;
        const double A = (std::fabs(am) <= 1048576.0) ? std::nearbyint(am) : 0.0;
        a.shift[c] = (float)A;
        a.scale[c] = (float)(1.0 / (255.0 * s));
        a.bias[c] = (float)(-(am - A) / (255.0 * s));
        if (!std::isfinite(a.scale[c]) || !std::isfinite(a.bias[c])) return false;
    }
    return true;
}

namespace {

// The workspace of the last launch on each of 256 streams (stream_guard.h).
bool note_stream_workspace(void* stream, void* workspace) {
    static StreamWorkspaceGuard<256> guard;
    return guard.note(stream, workspace);
}

int fused_norm_impl(const uint8_t* src, void* dst, int N, int H, int W, int C, const float* mean,
                    const float* stdv, const tr_aug_param* aug, int out_dtype, int out_layout,
                    void* stream, int variant, void* workspace, const CropSource& cs = CropSource(),
                    const Sampling& smp = Sampling(), unsigned flags = 0) {
    if ((flags & ~(unsigned)TR_LAUNCH_OVERLAP_PREVIOUS) != 0) return TR_ERR_INVALID_ARGUMENT;
    int rc = check_shape(N, H, W, C, out_dtype, out_layout);
    if (rc != TR_OK) return rc;
    // one channel: NCHW and NHWC are the same bytes; the NHWC path's tile
    // stores avoid shared-memory bank conflicts (binary32 256x224x224x1:
    // 0.88 -> 0.94 of the copy peak)
    if (C == 1 && out_layout == TR_LAYOUT_NCHW) out_layout = TR_LAYOUT_NHWC;
    if (variant != TR_VARIANT_AUTO && variant != TR_VARIANT_TILED && variant != TR_VARIANT_GENERIC)
        return TR_ERR_INVALID_ARGUMENT;
    if (mean == nullptr || stdv == nullptr) return TR_ERR_INVALID_ARGUMENT;
    LaunchArgs a;
    if (!fold_constants(mean, stdv, C, a)) return TR_ERR_INVALID_ARGUMENT;
    if (N == 0) return TR_OK;
    if (src == nullptr || dst == nullptr) return TR_ERR_INVALID_ARGUMENT;
    const int ob = (out_dtype == TR_OUT_F16) ? 2 : 4;
    // an output array of binary32/binary16 elements starts on an element
    // boundary; the records are int32 fields
    if (((uintptr_t)dst % (uintptr_t)ob) != 0) return TR_ERR_INVALID_ARGUMENT;
    if (aug != nullptr && ((uintptr_t)aug % 4u) != 0) return TR_ERR_INVALID_ARGUMENT;
    if (workspace != nullptr && ((uintptr_t)workspace % 16u) != 0) return TR_ERR_INVALID_ARGUMENT;
    const int out_ch = (out_layout == TR_LAYOUT_NHWC4) ? 4 : C;
    if (cs.on) {
        if (cs.src_H < H || cs.src_W < W) return TR_ERR_INVALID_ARGUMENT;
        if (cs.row_stride < (size_t)cs.src_W * C ||
            cs.image_stride < (size_t)(cs.src_H - 1) * cs.row_stride + (size_t)cs.src_W * C)
            return TR_ERR_INVALID_ARGUMENT;
        if (cs.crop != nullptr && ((uintptr_t)cs.crop % 4u) != 0) return TR_ERR_INVALID_ARGUMENT;
    }
    const unsigned long long in_bytes =
        cs.on ? (unsigned long long)(N - 1) * cs.image_stride + (unsigned long long)(cs.src_H - 1) * cs.row_stride +
                    (unsigned long long)cs.src_W * C
              : (unsigned long long)N * H * W * C;
    const unsigned long long out_bytes = (unsigned long long)N * H * W * out_ch * ob;
    const uintptr_t s0 = (uintptr_t)src, d0 = (uintptr_t)dst;
    if (s0 < d0 + out_bytes && d0 < s0 + in_bytes) return TR_ERR_INVALID_ARGUMENT;   // overlap
    if (smp.on) {
        // the kernel writes the records while it reads src and writes dst
        const uintptr_t r0 = (uintptr_t)smp.out;
        const unsigned long long rec_bytes = (unsigned long long)N * sizeof(tr_aug_param);
        if (smp.out == nullptr || (r0 % 4u) != 0 || aug != nullptr) return TR_ERR_INVALID_ARGUMENT;
        if ((r0 < s0 + in_bytes && s0 < r0 + rec_bytes) || (r0 < d0 + out_bytes && d0 < r0 + rec_bytes))
            return TR_ERR_INVALID_ARGUMENT;
    }

    const bool tiled_ok = cs.on ? tiled_crop_supported(src, dst, N, H, W, C, out_dtype, out_layout, cs.src_H,
                                                       cs.src_W, cs.row_stride, cs.image_stride)
                                : tiled_supported(src, dst, N, H, W, C, out_dtype, out_layout);
    const bool forced = (variant != TR_VARIANT_AUTO);
    if (variant == TR_VARIANT_TILED && !tiled_ok) return TR_ERR_NOT_SUPPORTED;
    if (variant == TR_VARIANT_AUTO)
        variant = (tiled_ok && !small_batch(N, H, W, C, out_layout)) ? TR_VARIANT_TILED : TR_VARIANT_GENERIC;

    a.src = src;
    a.dst = dst;
    a.N = N; a.H = H; a.W = W; a.C = C;
    a.aug = aug;
    a.out_dtype = out_dtype;
    a.out_layout = out_layout;
    a.stream = stream;
    a.workspace = workspace;
    a.crop_src = cs.on;
    a.crop = cs.crop;
    a.src_H = cs.src_H;
    a.src_W = cs.src_W;
    a.src_row_stride = cs.row_stride;
    a.src_image_stride = cs.image_stride;
    // overlap only what the caller declared independent, never a kernel that
    // used the same workspace; with GPU-made records the sampler overlaps the
    // previous kernel and the fused kernel reads the records once the sampler
    // (hence that kernel too) has completed
    const bool same_ws = note_stream_workspace(stream, workspace);
    a.overlap_prev = (flags & TR_LAUNCH_OVERLAP_PREVIOUS) != 0 && !same_ws;
    if (smp.on) {
        // records made on the GPU: by the tiled kernel itself where it can,
        // else by the sampler first (launch() decides)
        a.aug = nullptr;
        a.spec = &smp.spec;
        a.records_out = smp.out;
    }
    rc = launch(a, variant);
    if (rc == TR_ERR_NOT_SUPPORTED && variant == TR_VARIANT_TILED && !forced) {
        // the tiled geometry does not fit this device's shared memory (rows
        // of hundreds of kilobytes): the generic kernel handles any shape
        rc = launch(a, TR_VARIANT_GENERIC);
    }
    return rc;
}

}  // namespace
}  // namespace trfn

using namespace trfn;

extern "C" {

int tr_fused_norm(const uint8_t* src_u8, void* dst, int N, int H, int W, int C, const float* mean,
                  const float* std, const tr_aug_param* aug_params, int out_dtype, int out_layout,
                  void* stream) {
    return fused_norm_impl(src_u8, dst, N, H, W, C, mean, std, aug_params, out_dtype, out_layout,
                           stream, TR_VARIANT_AUTO, nullptr);
}

int tr_fused_norm_variant(const uint8_t* src_u8, void* dst, int N, int H, int W, int C,
                          const float* mean, const float* std, const tr_aug_param* aug_params,
                          int out_dtype, int out_layout, void* stream, int variant) {
    return fused_norm_impl(src_u8, dst, N, H, W, C, mean, std, aug_params, out_dtype, out_layout,
                           stream, variant, nullptr);
}

int tr_fused_norm_ws(const uint8_t* src_u8, void* dst, int N, int H, int W, int C, const float* mean,
                     const float* std, const tr_aug_param* aug_params, int out_dtype, int out_layout,
                     void* stream, int variant, void* workspace) {
    return fused_norm_impl(src_u8, dst, N, H, W, C, mean, std, aug_params, out_dtype, out_layout,
                           stream, variant, workspace);
}

int tr_fused_norm_ex(const uint8_t* src_u8, void* dst, int N, int H, int W, int C, const float* mean,
                     const float* std, const tr_aug_param* aug_params, int out_dtype, int out_layout,
                     void* stream, int variant, void* workspace, unsigned flags) {
    return fused_norm_impl(src_u8, dst, N, H, W, C, mean, std, aug_params, out_dtype, out_layout,
                           stream, variant, workspace, CropSource(), Sampling(), flags);
}

int tr_fused_norm_batches(const tr_batch* batches, int K, int N, int H, int W, int C, const float* mean,
                          const float* std, int out_dtype, int out_layout, void* stream, void* workspace,
                          unsigned flags) {
    if ((flags & ~(unsigned)TR_LAUNCH_OVERLAP_PREVIOUS) != 0) return TR_ERR_INVALID_ARGUMENT;
    if (K < 0 || K > TR_MAX_BATCHES || (K > 0 && batches == nullptr)) return TR_ERR_INVALID_ARGUMENT;
    int rc = check_shape(N, H, W, C, out_dtype, out_layout);
    if (rc != TR_OK) return rc;
    LaunchArgs a;
    if (mean == nullptr || std == nullptr || !fold_constants(mean, std, C, a)) return TR_ERR_INVALID_ARGUMENT;
    if (K == 0 || N == 0) return TR_OK;
    if (workspace != nullptr && ((uintptr_t)workspace % 16u) != 0) return TR_ERR_INVALID_ARGUMENT;
    if (C == 1 && out_layout == TR_LAYOUT_NCHW) out_layout = TR_LAYOUT_NHWC;   // the same bytes
    const int ob = (out_dtype == TR_OUT_F16) ? 2 : 4;
    const int out_ch = (out_layout == TR_LAYOUT_NHWC4) ? 4 : C;
    const unsigned long long in_bytes = (unsigned long long)N * H * W * C;
    const unsigned long long out_bytes = (unsigned long long)N * H * W * out_ch * ob;
    auto overlaps = [](uintptr_t a0, unsigned long long an, uintptr_t b0, unsigned long long bn) {
        return a0 < b0 + bn && b0 < a0 + an;
    };
    bool one_launch = K > 1 && (long long)K * N * H <= (1LL << 31) - 1 &&
                      (long long)K * N * H * W * 4 <= kMaxElements && !small_batch(K * N, H, W, C, out_layout);
    for (int k = 0; k < K; ++k) {
        const tr_batch& b = batches[k];
        if (b.src_u8 == nullptr || b.dst == nullptr) return TR_ERR_INVALID_ARGUMENT;
        if (((uintptr_t)b.dst % (uintptr_t)ob) != 0) return TR_ERR_INVALID_ARGUMENT;
        if (b.aug_params != nullptr && ((uintptr_t)b.aug_params % 4u) != 0) return TR_ERR_INVALID_ARGUMENT;
        for (int j = 0; j < K; ++j) {
            if (overlaps((uintptr_t)b.dst, out_bytes, (uintptr_t)batches[j].src_u8, in_bytes))
                return TR_ERR_INVALID_ARGUMENT;
            if (j != k && overlaps((uintptr_t)b.dst, out_bytes, (uintptr_t)batches[j].dst, out_bytes))
                return TR_ERR_INVALID_ARGUMENT;
        }
        one_launch = one_launch && ((uintptr_t)b.src_u8 % 16u) == 0 && ((uintptr_t)b.dst % 16u) == 0 &&
                     tiled_supported(b.src_u8, b.dst, N, H, W, C, out_dtype, out_layout);
    }
    if (one_launch) {
        a.src = batches[0].src_u8;
        a.dst = batches[0].dst;
        a.N = K * N; a.H = H; a.W = W; a.C = C;
        a.aug = nullptr;
        a.out_dtype = out_dtype;
        a.out_layout = out_layout;
        a.stream = stream;
        a.workspace = workspace;
        a.batch_images = N;
        for (int k = 0; k < K; ++k) {
            a.bsrc[k] = batches[k].src_u8;
            a.bdst[k] = batches[k].dst;
            a.baug[k] = batches[k].aug_params;
        }
        const bool same_ws = note_stream_workspace(stream, workspace);
        a.overlap_prev = (flags & TR_LAUNCH_OVERLAP_PREVIOUS) != 0 && !same_ws;
        rc = launch(a, TR_VARIANT_TILED);
        if (rc != TR_ERR_NOT_SUPPORTED) return rc;
        // the tiled geometry does not fit this device: one launch per batch
    }
    for (int k = 0; k < K; ++k) {
        rc = fused_norm_impl(batches[k].src_u8, batches[k].dst, N, H, W, C, mean, std, batches[k].aug_params,
                             out_dtype, out_layout, stream, TR_VARIANT_AUTO, workspace, CropSource(), Sampling(),
                             flags);
        if (rc != TR_OK) return rc;
    }
    return TR_OK;
}

size_t tr_workspace_bytes(void) { return kWorkspaceBytes; }

int tr_fused_norm_sampled(const uint8_t* src_u8, void* dst, int N, int H, int W, int C, const float* mean,
                          const float* std, uint64_t seed, uint64_t offset, const tr_aug_sampling* sampling,
                          tr_aug_param* d_records, uint64_t* next_offset, int out_dtype, int out_layout,
                          void* stream, int variant, void* workspace) {
    return tr_fused_norm_sampled_ex(src_u8, dst, N, H, W, C, mean, std, seed, offset, sampling, d_records,
                                    next_offset, out_dtype, out_layout, stream, variant, workspace, 0u);
}

int tr_fused_norm_sampled_ex(const uint8_t* src_u8, void* dst, int N, int H, int W, int C, const float* mean,
                             const float* std, uint64_t seed, uint64_t offset, const tr_aug_sampling* sampling,
                             tr_aug_param* d_records, uint64_t* next_offset, int out_dtype, int out_layout,
                             void* stream, int variant, void* workspace, unsigned flags) {
    if (sampling == nullptr || H < 1 || W < 1) return TR_ERR_INVALID_ARGUMENT;
    Sampling smp;
    smp.on = true;
    smp.out = d_records;
    int rc = make_sample_spec(seed, offset, H, W, sampling->flip_enabled, sampling->flip_p,
                              sampling->erase_enabled, sampling->erase_p, sampling->scale_lo, sampling->scale_hi,
                              sampling->ratio_lo, sampling->ratio_hi, &smp.spec);
    if (rc != TR_OK) return rc;
    if (N > 0 && d_records == nullptr) return TR_ERR_INVALID_ARGUMENT;
    rc = fused_norm_impl(src_u8, dst, N, H, W, C, mean, std, nullptr, out_dtype, out_layout, stream, variant,
                         workspace, CropSource(), smp, flags);
    if (rc == TR_OK && next_offset != nullptr) *next_offset = offset + (uint64_t)N * 24u;
    return rc;
}

int tr_fused_norm_crop(const uint8_t* src_u8, int src_H, int src_W, size_t src_row_stride,
                       size_t src_image_stride, const int32_t* crop_yx, void* dst, int N, int H, int W, int C,
                       const float* mean, const float* std, const tr_aug_param* aug_params, int out_dtype,
                       int out_layout, void* stream, int variant, void* workspace) {
    if (src_H < 1 || src_W < 1) return TR_ERR_INVALID_ARGUMENT;
    CropSource cs;
    cs.on = true;
    cs.crop = crop_yx;
    cs.src_H = src_H;
    cs.src_W = src_W;
    cs.row_stride = src_row_stride;
    cs.image_stride = src_image_stride;
    return fused_norm_impl(src_u8, dst, N, H, W, C, mean, std, aug_params, out_dtype, out_layout, stream,
                           variant, workspace, cs);
}

int tr_fused_norm_crop_ex(const uint8_t* src_u8, int src_H, int src_W, size_t src_row_stride,
                          size_t src_image_stride, const int32_t* crop_yx, void* dst, int N, int H, int W, int C,
                          const float* mean, const float* std, const tr_aug_param* aug_params, int out_dtype,
                          int out_layout, void* stream, int variant, void* workspace, unsigned flags) {
    if (src_H < 1 || src_W < 1) return TR_ERR_INVALID_ARGUMENT;
    CropSource cs;
    cs.on = true;
    cs.crop = crop_yx;
    cs.src_H = src_H;
    cs.src_W = src_W;
    cs.row_stride = src_row_stride;
    cs.image_stride = src_image_stride;
    return fused_norm_impl(src_u8, dst, N, H, W, C, mean, std, aug_params, out_dtype, out_layout, stream,
                           variant, workspace, cs, Sampling(), flags);
}

int tr_fused_norm_plan(const uint8_t* src_u8, const void* dst, int N, int H, int W, int C,
                       int out_dtype, int out_layout, int* variant) {
    const int rc = check_shape(N, H, W, C, out_dtype, out_layout);
    if (rc != TR_OK) return rc;
    if (variant == nullptr) return TR_ERR_INVALID_ARGUMENT;
    if (C == 1 && out_layout == TR_LAYOUT_NCHW) out_layout = TR_LAYOUT_NHWC;   // the same bytes, as in the launch
    *variant = (tiled_supported(src_u8, dst, N, H, W, C, out_dtype, out_layout) &&
                !small_batch(N, H, W, C, out_layout))
                   ? TR_VARIANT_TILED
                   : TR_VARIANT_GENERIC;
    return TR_OK;
}

int tr_fused_norm_geometry(const uint8_t* src_u8, const void* dst, int N, int H, int W, int C, int out_dtype,
                           int out_layout, unsigned flags, int* rows, int* stages, int* ctas_per_sm, int* grid,
                           int* odd_form) {
    if ((flags & ~(unsigned)TR_LAUNCH_OVERLAP_PREVIOUS) != 0) return TR_ERR_INVALID_ARGUMENT;
    const int rc = check_shape(N, H, W, C, out_dtype, out_layout);
    if (rc != TR_OK) return rc;
    if (N < 1 || rows == nullptr || stages == nullptr || ctas_per_sm == nullptr || grid == nullptr ||
        odd_form == nullptr)
        return TR_ERR_INVALID_ARGUMENT;
    if (C == 1 && out_layout == TR_LAYOUT_NCHW) out_layout = TR_LAYOUT_NHWC;   // as in the launch
    if (!tiled_supported(src_u8, dst, N, H, W, C, out_dtype, out_layout)) return TR_ERR_NOT_SUPPORTED;
    LaunchArgs a;
    for (int c = 0; c < 4; ++c) { a.shift[c] = 0.0f; a.scale[c] = 0.0f; a.bias[c] = 0.0f; }
    a.src = src_u8;
    a.dst = const_cast<void*>(dst);
    a.N = N; a.H = H; a.W = W; a.C = C;
    a.aug = nullptr;
    a.out_dtype = out_dtype;
    a.out_layout = out_layout;
    a.stream = nullptr;
    a.workspace = nullptr;
    a.overlap_prev = (flags & TR_LAUNCH_OVERLAP_PREVIOUS) != 0;
    TiledGeometry g;
    const int r2 = tiled_geometry(a, &g);
    if (r2 != TR_OK) return r2;
    *rows = g.rows;
    *stages = g.stages;
    *ctas_per_sm = g.ctas_per_sm;
    *grid = g.grid;
    *odd_form = g.odd_form;
    return TR_OK;
}

int tr_norm_preset(int preset, float mean[3], float std[3], int* channels) {
    if (mean == nullptr || std == nullptr || channels == nullptr) return TR_ERR_INVALID_ARGUMENT;
    // values of the preset table in the FusedNormalization article, §九
    static const struct { float m[3]; float s[3]; int ch; } table[5] = {
        {{0.0f, 0.0f, 0.0f}, {1.0f, 1.0f, 1.0f}, 3},                                  // NO_NORM
        {{0.1307f, 0.0f, 0.0f}, {0.3081f, 1.0f, 1.0f}, 1},                            // MNIST
        {{0.4914f, 0.4822f, 0.4465f}, {0.2470f, 0.2435f, 0.2616f}, 3},                // CIFAR
        {{0.485f, 0.456f, 0.406f}, {0.229f, 0.224f, 0.225f}, 3},                      // IMAGENET
        {{123.68f / 255.0f, 116.78f / 255.0f, 103.94f / 255.0f},
         {1.0f / 255.0f, 1.0f / 255.0f, 1.0f / 255.0f}, 3},                           // MLPERF
    };
    if (preset < 0 || preset > 4) return TR_ERR_INVALID_ARGUMENT;
    for (int c = 0; c < 3; ++c) {
        mean[c] = table[preset].m[c];
        std[c] = table[preset].s[c];
    }
    *channels = table[preset].ch;
    return TR_OK;
}

int tr_validate_aug_params(const tr_aug_param* p, int N, int H, int W, int* bad_index) {
    if (bad_index) *bad_index = -1;
    if (N < 0 || H < 1 || W < 1) return TR_ERR_INVALID_ARGUMENT;
    if (N > 0 && p == nullptr) return TR_ERR_INVALID_ARGUMENT;
    for (int n = 0; n < N; ++n) {
        const tr_aug_param& a = p[n];
        if (a.h <= 0 || a.w <= 0) continue;
        const long long y1 = (long long)a.y0 + a.h, x1 = (long long)a.x0 + a.w;
        if (a.y0 < 0 || a.x0 < 0 || y1 > H || x1 > W) {
            if (bad_index) *bad_index = n;
            return TR_ERR_INVALID_ARGUMENT;
        }
    }
    return TR_OK;
}

int tr_device_status(int* flags, int clear) {
    if (flags == nullptr) return TR_ERR_INVALID_ARGUMENT;
    return read_device_status(flags, clear != 0);
}

uint64_t tr_launch_count(void) { return launch_count(); }

int tr_tune_tiled(int band_bytes, int stages, int max_ctas_per_sm, int flags) {
    if (band_bytes < 0 || stages < 0 || stages > 8 || stages == 1 || max_ctas_per_sm < 0)
        return TR_ERR_INVALID_ARGUMENT;
    tune_tiled(band_bytes, stages, max_ctas_per_sm, flags);
    return TR_OK;
}

const char* tr_status_string(int status) {
    switch (status) {
    case TR_OK: return "ok";
    case TR_ERR_INVALID_ARGUMENT: return "invalid argument";
    case TR_ERR_NOT_SUPPORTED: return "not supported";
    case TR_ERR_CUDA: return "CUDA error";
    case TR_ERR_TIMEOUT: return "timed out";
    case TR_ERR_DEVICE: return "device reported an error";
    case TR_END_OF_DATA: return "end of data";
    default: return "unknown status";
    }
}

const char* tr_last_error_message(void) { return last_error(); }

int tr_version(void) { return 100; }

}  // extern "C"

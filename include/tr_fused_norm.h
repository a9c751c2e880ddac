/*
 * tr_fused_norm.h — C ABI of the GB300 fused normalisation library (libtrfn.so).
 *
 * One memory pass turns a batch of uint8 NHWC images into normalised binary32
 * or binary16 tensors: ToTensor (x/255) and per-channel Normalize
 * ((x - mean)/std) folded into one multiply-add, an optional horizontal flip
 * and an optional erase rectangle per image.  The operation is the one the
 * Tech-Renaissance article "(11) FusedNormalization: fuse the last step of data
 * augmentation into one memory traversal" (tech-renaissance.cn/blog/?p=487)
 * describes as CPU SIMD code; here it runs as hand-written CUDA for sm_103a.
 *
 * Conventions for every entry point:
 *   - Return a tr_status code; nothing throws across this boundary.
 *   - Arguments are checked on the host before anything is launched; a call
 *     that returns TR_ERR_INVALID_ARGUMENT or TR_ERR_NOT_SUPPORTED has not
 *     touched the GPU.
 *   - Every buffer is owned by the caller.  Nothing on the call path
 *     allocates memory.
 *   - "stream" is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued on it; calls do not wait for the GPU.
 *   - Device pointers must stay valid until the enqueued work has finished.
 */
#ifndef TR_FUSED_NORM_H
#define TR_FUSED_NORM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  INVALID_ARGUMENT is the article's ValueError (its execute()
 * rejects an externally set output stride, §五); NOT_SUPPORTED is its
 * TR_NOT_IMPLEMENTED (§七, FP16 on a CPU without the needed extension).     */
typedef enum tr_status {
    TR_OK = 0,
    TR_ERR_INVALID_ARGUMENT = 1,
    TR_ERR_NOT_SUPPORTED = 2,
    TR_ERR_CUDA = 3,          /* a CUDA runtime call failed; see tr_last_error_message() */
    TR_ERR_TIMEOUT = 4,       /* a bounded wait ran out (host event wait or device pipeline wait) */
    TR_ERR_DEVICE = 5,        /* a kernel reported an error through the device status word */
    TR_END_OF_DATA = 6        /* staging: the data set was closed and has no further sample/batch */
} tr_status;

/* Output element type (article §六 "FP32 and FP16 output"). */
typedef enum tr_out_dtype {
    TR_OUT_F32 = 0,           /* binary32 */
    TR_OUT_F16 = 1            /* binary16, round to nearest even of the binary32 value */
} tr_out_dtype;

/* Output layout.  The article writes NHWC; FP16 there is always padded to four
 * channels (§六, §八).  N, H, W, C as in the input.                          */
typedef enum tr_layout {
    TR_LAYOUT_NHWC = 0,       /* out[((n*H + y)*W + x)*C + c]                     */
    TR_LAYOUT_NCHW = 1,       /* out[((n*C + c)*H + y)*W + x]                     */
    TR_LAYOUT_NHWC4 = 2       /* out[((n*H + y)*W + x)*4 + c], channels C..3 = +0 */
} tr_layout;

/* Normalisation presets (article §九 "Five normalisation presets"). */
typedef enum tr_preset {
    TR_PRESET_NO_NORM = 0,    /* mean 0, std 1 (3 channels): x/255 only          */
    TR_PRESET_MNIST = 1,      /* 0.1307 / 0.3081 (1 channel)                     */
    TR_PRESET_CIFAR = 2,
    TR_PRESET_IMAGENET = 3,
    TR_PRESET_MLPERF = 4      /* mean (123.68, 116.78, 103.94)/255, std 1/255    */
} tr_preset;

/* Per-image augmentation record (20 bytes, int32 fields).
 *   flip      non-zero: output pixel (y, x) takes source pixel (y, W-1-x)
 *             (article §五: read from the mirrored or the original position).
 *   y0,x0,h,w erase rectangle in OUTPUT (post-flip) coordinates: every channel
 *             of output pixels y0 <= y < y0+h, x0 <= x < x0+w is +0.0 (article
 *             §十二: a memset of the normalised output after the main pass).
 *             h <= 0 or w <= 0 means no erase.  Parts outside the image are
 *             ignored (the kernels clip), so a bad record cannot write out of
 *             bounds; tr_validate_aug_params() reports such records.          */
typedef struct tr_aug_param {
    int32_t flip;
    int32_t y0;
    int32_t x0;
    int32_t h;
    int32_t w;
} tr_aug_param;

/* Kernel selection, for tests and benchmarks.  AUTO picks TILED whenever its
 * preconditions hold (a 16-byte aligned source, rows of at most 2^24 bytes,
 * fewer than 2^31 image rows) and the batch has at least 2^18 output elements
 * (below that the per-element kernel finishes first), else GENERIC.  TILED
 * runs its aligned form when dst is 16-byte aligned, W*C is a multiple of 16
 * and, for NCHW, W*sizeof(out) is a multiple of 16; otherwise its odd-row
 * form (bands staged from the 16-byte boundary below them, groups realigned
 * in registers, output tiles following the band's global alignment): at
 * 256x299x299x3 about 0.75 of the aligned form's rate for binary16 and the
 * same rate for binary32.  One-channel NCHW output is the same bytes as
 * NHWC and takes that path.  Forcing TILED where its preconditions fail
 * returns TR_ERR_NOT_SUPPORTED.                                             */
typedef enum tr_variant {
    TR_VARIANT_AUTO = 0,
    TR_VARIANT_TILED = 1,     /* persistent CTAs, TMA bulk row-band staging, TMA bulk stores */
    TR_VARIANT_GENERIC = 2    /* one thread per output pixel, any shape, stride and alignment */
} tr_variant;

/* ------------------------------------------------------------------------
 * tr_fused_norm — the fused step on a batch (article §五, §六, §八, §十二).
 *
 *   src_u8      device, N*H*W*C bytes, compact NHWC uint8.
 *   dst         device, N*H*W*C' elements of out_dtype in out_layout, compact
 *               (C' = 4 for TR_LAYOUT_NHWC4, else C), aligned to its element
 *               size (4 or 2 bytes).  There is no stride
 *               argument: like the article's execute(), the output stride is
 *               fixed by the shape, type and layout.  Must not overlap src.
 *   N,H,W,C     N >= 0 (0 = nothing to do), H >= 1, W >= 1, 1 <= C <= 4.
 *   mean, std   host arrays of C floats, read during the call.  std[c] must be
 *               finite and non-zero, mean[c] finite.  The kernels compute
 *               (x - A)*scale + bias in one fused multiply-add, with A =
 *               255*mean rounded to an integer (so x - A is exact), scale =
 *               1/(255*std) and bias = -(255*mean - A)*scale, each formed in
 *               binary64 and rounded to binary32: within 3 binary32 ulps of
 *               the exact value for any mean and std.
 *   aug_params  device array of N tr_aug_param (4-byte aligned), read in
 *               stream order; NULL means no flip and no erase for every image.
 *   out_dtype   tr_out_dtype; out_layout tr_layout.
 *   stream      cudaStream_t as void*.
 * Errors: TR_ERR_INVALID_ARGUMENT (bad shape, type, layout, null pointer,
 * dst or aug_params off their element alignment, non-finite or zero std,
 * overlapping src/dst, sizes beyond 2^40 elements),
 * TR_ERR_NOT_SUPPORTED (C > 4), TR_ERR_CUDA (launch failure).  Pointers off
 * a 16-byte boundary are not an error: a source off 16 bytes takes the
 * GENERIC kernel, an output off 16 bytes the TILED kernel's odd-row form.   */
int tr_fused_norm(const uint8_t* src_u8, void* dst, int N, int H, int W, int C,
                  const float* mean, const float* std, const tr_aug_param* aug_params,
                  int out_dtype, int out_layout, void* stream);

/* tr_fused_norm with an explicit kernel choice (tr_variant). */
int tr_fused_norm_variant(const uint8_t* src_u8, void* dst, int N, int H, int W, int C,
                          const float* mean, const float* std, const tr_aug_param* aug_params,
                          int out_dtype, int out_layout, void* stream, int variant);

/* tr_fused_norm with a scheduling workspace.  The TILED kernel then hands
 * out row bands dynamically (CTAs that run faster take more), so all CTAs
 * finish together; results are identical to tr_fused_norm's.
 *   workspace  device buffer of tr_workspace_bytes() bytes, 16-byte aligned,
 *              all zero before its first use.  Every launch leaves it zero
 *              again, so launches that run one after another (one stream,
 *              or a graph's chain) may share it; launches that can run at the
 *              same time (other streams) need their own.  NULL = the static
 *              schedule of tr_fused_norm.  After a TR_ERR_DEVICE report the
 *              workspace must be zeroed again.  The GENERIC kernel ignores it.
 * Other arguments and errors as tr_fused_norm_variant; a workspace off a
 * 16-byte boundary is TR_ERR_INVALID_ARGUMENT.                              */
int tr_fused_norm_ws(const uint8_t* src_u8, void* dst, int N, int H, int W, int C,
                     const float* mean, const float* std, const tr_aug_param* aug_params,
                     int out_dtype, int out_layout, void* stream, int variant, void* workspace);

/* Launch options of tr_fused_norm_ex (bits of `flags`). */
enum {
    /* This launch reads and writes nothing that the kernel before it in the
     * stream writes, writes nothing that kernel reads, and its workspace (if
     * any) is not that kernel's: consecutive batches of a data loader, each
     * with its own source, output and records, and workspaces alternating
     * between two buffers.  The TILED kernel then starts its copies while the
     * previous kernel drains instead of after it has completed; each CTA still
     * waits for the previous kernel before it exits, so this launch completes
     * after it and later work in the stream sees both results.  Only a
     * preceding kernel that releases its dependents early (this library's)
     * can be overlapped; after a copy, a memset or another library's kernel
     * stream order is unchanged.  A launch whose workspace equals the one of
     * this library's previous launch on the same stream is not overlapped (the
     * flag is dropped); the library remembers the last 256 streams it launched
     * on, and once more have been used, a launch with a workspace on a stream
     * it no longer remembers is not overlapped either.  A launch releases the next kernel in the stream only
     * once the kernel before it has completed, so no launch ever overlaps
     * more than the one kernel before it.  The GENERIC kernel (small batches,
     * strided or unaligned buffers) honours the flag the same way: one thread
     * of each block waits for the previous kernel while the others work.     */
    TR_LAUNCH_OVERLAP_PREVIOUS = 1
};

/* tr_fused_norm_ws with launch options.  Measured at 256x224x224x3 (graph of
 * launches over rotating buffers, static schedule): binary16 20.9 -> 19.4 us
 * a batch, binary32 32.7 -> 30.0 us with TR_LAUNCH_OVERLAP_PREVIOUS.
 *   flags  0 or TR_LAUNCH_OVERLAP_PREVIOUS; other bits are
 *          TR_ERR_INVALID_ARGUMENT.
 * Other arguments, results and errors as tr_fused_norm_ws.                  */
int tr_fused_norm_ex(const uint8_t* src_u8, void* dst, int N, int H, int W, int C,
                     const float* mean, const float* std, const tr_aug_param* aug_params,
                     int out_dtype, int out_layout, void* stream, int variant, void* workspace,
                     unsigned flags);

/* tr_fused_norm_batches — the fused step on K batches of the same shape in
 * one launch (the article's execute() runs once per batch, §五; a data
 * loader hands the step one batch after another).  Each launch that waits
 * for the previous one pays a fixed cost (grid launch, the first copies'
 * round trip, the drain of its last bands: about 2.5 us of 19 at
 * 256x224x224x3 -> binary16); one launch over K batches pays it once.
 *   batches     host array of K descriptors, read during the call: batch k's
 *               source (N*H*W*C bytes, compact NHWC uint8), output (as
 *               tr_fused_norm's dst) and records (N, or NULL: no flip and no
 *               erase), all device pointers.
 *   K           0 <= K <= TR_MAX_BATCHES (0 = nothing to do).
 *   N,H,W,C, mean, std, out_dtype, out_layout: the shape of ONE batch and
 *               the step's settings, as tr_fused_norm.
 *   stream, workspace, flags: as tr_fused_norm_ex (one workspace for the
 *               launch; TR_LAUNCH_OVERLAP_PREVIOUS promises that no batch
 *               shares a buffer with the kernel before the call).
 * Results: batch k's output equals tr_fused_norm's on batch k, bit for bit.
 * Every source and output must be 16-byte aligned and the batches large
 * enough for the TILED kernel (tr_fused_norm_plan on K*N images) for the
 * single launch; otherwise the batches are launched one after another
 * (stream order, same results).
 * Errors as tr_fused_norm for every batch, TR_ERR_INVALID_ARGUMENT for K
 * outside 0..TR_MAX_BATCHES, a NULL batches array with K > 0, or any batch's
 * output overlapping any batch's source or another batch's output.          */
#define TR_MAX_BATCHES 16
typedef struct tr_batch {
    const uint8_t* src_u8;
    void* dst;
    const tr_aug_param* aug_params;
} tr_batch;

int tr_fused_norm_batches(const tr_batch* batches, int K, int N, int H, int W, int C, const float* mean,
                          const float* std, int out_dtype, int out_layout, void* stream, void* workspace,
                          unsigned flags);

/* tr_fused_norm_crop — the fused step on H x W windows of a larger, strided
 * source: the crop just upstream of the step fused into its load (the
 * article's execute() takes an input stride, §五; DALI's crop_mirror_normalize,
 * cited as prior art in §二.2, also fuses the crop).
 *   src_u8       device; image n's byte (sy, sx, c) is at
 *                src_u8[n*src_image_stride + sy*src_row_stride + sx*C + c],
 *                0 <= sy < src_H, 0 <= sx < src_W.
 *   crop_yx      device int32 [N][2]: the window's top row and left column in
 *                its source image (4-byte aligned), or NULL for (0, 0) for all.
 *                Windows are clamped into the source image, so an origin out
 *                of range cannot read out of bounds.
 *   N,H,W,C, dst, mean, std, aug_params (in window coordinates), out_dtype,
 *   out_layout, stream, variant, workspace: as tr_fused_norm_ws.
 * Output pixel (n, y, x) takes source pixel (n, cy + y, cx + x') with x' the
 * column of the window, mirrored when flipping.  The TILED kernel reads the
 * windows with TMA tensor copies when src is 16-byte aligned, src_W*C,
 * src_row_stride and src_image_stride are multiples of 16,
 * src_image_stride >= src_H*src_row_stride and W*C <= 4064 (plus the TILED
 * conditions of tr_fused_norm); otherwise GENERIC.
 * Errors as tr_fused_norm, and TR_ERR_INVALID_ARGUMENT for src_H < H,
 * src_W < W, a row stride below src_W*C or an image stride below
 * (src_H-1)*src_row_stride + src_W*C.                                       */
int tr_fused_norm_crop(const uint8_t* src_u8, int src_H, int src_W, size_t src_row_stride,
                       size_t src_image_stride, const int32_t* crop_yx, void* dst, int N, int H, int W, int C,
                       const float* mean, const float* std, const tr_aug_param* aug_params, int out_dtype,
                       int out_layout, void* stream, int variant, void* workspace);

/* tr_fused_norm_crop with launch options (flags as tr_fused_norm_ex; the
 * crop origins are read like the other inputs, so they too must not be
 * written by the kernel before the launch when TR_LAUNCH_OVERLAP_PREVIOUS is
 * given).  Other arguments, results and errors as tr_fused_norm_crop.       */
int tr_fused_norm_crop_ex(const uint8_t* src_u8, int src_H, int src_W, size_t src_row_stride,
                          size_t src_image_stride, const int32_t* crop_yx, void* dst, int N, int H, int W, int C,
                          const float* mean, const float* std, const tr_aug_param* aug_params, int out_dtype,
                          int out_layout, void* stream, int variant, void* workspace, unsigned flags);

/* Bytes of the scheduling workspace (2048). */
size_t tr_workspace_bytes(void);

/* tr_fused_norm_noalloc — tr_fused_norm_ws for callers that cannot allocate
 * device memory.  No counterpart in the FusedNormalization article: it exists
 * for programs whose device memory is fixed by a memory plan made at start-up,
 * loader threads that must not wait on the device-wide synchronisation of
 * cudaFree, and plug-ins without access to their host's allocator.  Instead
 * of a caller's workspace it uses a 2048-byte scratch array in this
 * library's module memory (a file-scope __device__ array that every GPU which
 * loads the library holds until the process exits), and it allocates nothing.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress, with the device current) and caches it; make that
 *     first call before any stream capture.  The cached address outlives a
 *     device reset, so resetting a device (cudaDeviceReset) or tearing down
 *     its primary context in a process that keeps calling this is not
 *     supported.
 *   - Each call that takes the tiled kernel (tr_fused_norm_plan) clears the
 *     scratch on `stream` (an asynchronous memset) before its kernel, and the
 *     kernel leaves it zero again; a call that takes the per-element kernel
 *     (small batches, unaligned buffers) uses no scratch and clears nothing.  All calls on a device
 *     share the one array: calls that overlap on the GPU (other streams or
 *     threads) race on it and must be ordered by the caller.
 *   - Scratch needs above the 2048-byte capacity are rejected with
 *     TR_ERR_NOT_SUPPORTED (tr_last_error_message() says so); every shape the
 *     kernels accept currently needs exactly tr_workspace_bytes().
 * Other arguments, results and errors as tr_fused_norm.                      */
int tr_fused_norm_noalloc(const uint8_t* src_u8, void* dst, int N, int H, int W, int C,
                          const float* mean, const float* std, const tr_aug_param* aug_params,
                          int out_dtype, int out_layout, void* stream);

/* Which kernel AUTO would pick for these arguments (TR_VARIANT_TILED or
 * TR_VARIANT_GENERIC), through *variant; host only, launches nothing.        */
int tr_fused_norm_plan(const uint8_t* src_u8, const void* dst, int N, int H, int W, int C,
                       int out_dtype, int out_layout, int* variant);

/* The geometry a TILED launch with these arguments would take, through the
 * same planning as the launch (host only, launches nothing; the CTAs-per-SM
 * figure comes from the device's occupancy calculator, so a CUDA device is
 * needed).  For tests and tuning.
 *   src_u8, dst  as for tr_fused_norm; only their alignment is used.
 *   flags        0 or TR_LAUNCH_OVERLAP_PREVIOUS (which changes the planning).
 *   *rows        rows per band; *stages shared-memory input stages;
 *   *ctas_per_sm resident CTAs per SM; *grid CTAs launched by the static
 *                schedule (no workspace: the bands spread evenly over the
 *                fewest CTAs that fit); with a workspace the launch takes
 *                ctas_per_sm times the SM count, or one CTA per band if
 *                there are fewer bands;
 *   *odd_form    1 when the odd-row form applies, else 0.
 * Errors as tr_fused_norm's argument checks; TR_ERR_NOT_SUPPORTED where the
 * TILED kernel does not apply; TR_ERR_INVALID_ARGUMENT for N < 1 or a NULL
 * result pointer.                                                          */
int tr_fused_norm_geometry(const uint8_t* src_u8, const void* dst, int N, int H, int W, int C, int out_dtype,
                           int out_layout, unsigned flags, int* rows, int* stages, int* ctas_per_sm, int* grid,
                           int* odd_form);

/* Preset mean/std (article §九).  Writes 3 floats to mean and std (unused
 * channels get mean 0, std 1) and the channel count to *channels.           */
int tr_norm_preset(int preset, float mean[3], float std[3], int* channels);

/* ------------------------------------------------------------------------
 * tr_sample_aug_params — host-side sampling of the per-image records with
 * the article's random decisions (§五 execute(), §十 uniform()/randint(),
 * §十二 generate_erase_rect()).  Per image, in this order: when
 * flip_enabled, one draw u and flip iff u < flip_p (the article hard-codes
 * 0.5); when erase_enabled and erase_p > 0, one gate draw (no erase unless
 * u < erase_p), then up to ten attempts of two draws each:
 *   area = (scale_lo + u*(scale_hi - scale_lo)) * H * W,
 *   aspect = exp(log(ratio_lo) + u*(log(ratio_hi) - log(ratio_lo))),
 *   h = round(sqrt(area*aspect)), w = round(sqrt(area/aspect)),
 * accepted when 0 < h < H and 0 < w < W, followed by y0 uniform on
 * [0, H-h] and x0 uniform on [0, W-w] (one draw each).  Binary32 arithmetic
 * without contraction, as written in the article.
 * Random numbers: Philox4x32-10 keyed by the 64-bit seed (low word first),
 * counter = the 64-bit offset (low word first) and two zero words; draw k
 * uses offset+k and its first output word w gives u = (w >> 8) * 2^-24 and
 * integer draws lo + floor(u*(hi-lo+1)).
 *   out_host    host array of N records.
 *   next_offset receives the first unused offset (may be NULL): sampling N1
 *               then N2 images from it equals sampling N1+N2 at once.
 * Errors: TR_ERR_INVALID_ARGUMENT for N < 0, H < 1, W < 1, a NULL out_host
 * with N > 0, non-finite or out-of-order scale/ratio bounds, ratio_lo <= 0. */
int tr_sample_aug_params(uint64_t seed, uint64_t offset, int N, int H, int W,
                         int flip_enabled, float flip_p, int erase_enabled, float erase_p,
                         float scale_lo, float scale_hi, float ratio_lo, float ratio_hi,
                         tr_aug_param* out_host, uint64_t* next_offset);

/* tr_sample_aug_params_device — the same decisions made on the GPU (a warp
 * per image for batches up to 8 images per SM, else a thread per image),
 * written to d_out (device, N records, 4-byte aligned) on
 * `stream` in stream order.  Image n draws from its own counter block,
 * offsets offset + 24n + k (24 = the most draws one image can take), so the
 * batch needs no sequential pass; *next_offset (may be NULL) receives
 * offset + 24N.  exp of the log-aspect draw is evaluated by fixed steps
 * (Cody–Waite reduction, degree-7 Taylor polynomial, correctly rounded
 * operations), so a CPU that takes the same steps reproduces the records bit
 * for bit; the records differ from tr_sample_aug_params' (which draws
 * sequentially) but follow the same distribution.  Errors as
 * tr_sample_aug_params, TR_ERR_CUDA on a launch failure.                     */
int tr_sample_aug_params_device(uint64_t seed, uint64_t offset, int N, int H, int W,
                                int flip_enabled, float flip_p, int erase_enabled, float erase_p,
                                float scale_lo, float scale_hi, float ratio_lo, float ratio_hi,
                                tr_aug_param* d_out, uint64_t* next_offset, void* stream);

/* Sampling settings of tr_fused_norm_sampled (meaning as the arguments of
 * tr_sample_aug_params).                                                    */
typedef struct tr_aug_sampling {
    int flip_enabled;
    float flip_p;
    int erase_enabled;
    float erase_p;
    float scale_lo, scale_hi;   /* erased area as a fraction of the image */
    float ratio_lo, ratio_hi;   /* erased aspect ratio h/w               */
} tr_aug_sampling;

/* tr_sample_aug_params_device(seed, offset, ...) into d_records, then
 * tr_fused_norm_ws reading them, as one call: two launches in stream order
 * (the kernel's prologue overlaps the sampler), no record crosses the host
 * link.  d_records: device, N records, 4-byte aligned, not overlapping src or
 * dst.  *next_offset (may be NULL) receives offset + 24N.  Errors as
 * tr_fused_norm_ws and tr_sample_aug_params_device, all checked before
 * either launch; TR_ERR_INVALID_ARGUMENT for a NULL sampling or d_records
 * (N > 0).  There is no such call in the article (its execute() draws on
 * the CPU, §五).  Sampling inside the fused kernel instead (the producer warp
 * drawing each band's record) measured slower: 22.6 against 21.3 us for
 * 256x224x224x3, as a record costs more to sample than to load and sits on
 * the producer's path to its next copy.                                    */
int tr_fused_norm_sampled(const uint8_t* src_u8, void* dst, int N, int H, int W, int C,
                          const float* mean, const float* std, uint64_t seed, uint64_t offset,
                          const tr_aug_sampling* sampling, tr_aug_param* d_records, uint64_t* next_offset,
                          int out_dtype, int out_layout, void* stream, int variant, void* workspace);

/* tr_fused_norm_sampled with launch options (flags as tr_fused_norm_ex).
 * With TR_LAUNCH_OVERLAP_PREVIOUS the caller promises that the kernel before
 * this call in the stream uses none of src, dst, d_records and workspace: the
 * sampler then writes the records while that kernel drains, and the fused
 * kernel requests its first bands at once.  Its records become readable only
 * when the sampler has completed, which is after the previous kernel; so in
 * the TILED kernel's aligned form each CTA makes the records of its first
 * bands itself (consumer warps, in parallel, with the sampler's steps: the
 * same bits) and converts them while the previous kernel drains, and reads
 * the later records from the sampler's output.  The crop and odd-row forms
 * wait for the sampler before they touch memory.                           */
int tr_fused_norm_sampled_ex(const uint8_t* src_u8, void* dst, int N, int H, int W, int C,
                             const float* mean, const float* std, uint64_t seed, uint64_t offset,
                             const tr_aug_sampling* sampling, tr_aug_param* d_records, uint64_t* next_offset,
                             int out_dtype, int out_layout, void* stream, int variant, void* workspace,
                             unsigned flags);

/* Host check of N records: TR_OK when every rectangle is either "no erase"
 * (h <= 0 or w <= 0) or lies inside the H x W image; else
 * TR_ERR_INVALID_ARGUMENT with the first bad index in *bad_index (may be
 * NULL).                                                                    */
int tr_validate_aug_params(const tr_aug_param* host_params, int N, int H, int W, int* bad_index);

/* ------------------------------------------------------------------------
 * tr_transfer_station — double-buffered feeding of the kernel from pinned
 * host memory (the TransferStation of the Tech-Renaissance article
 * "(10) Multi-threaded preprocessing, NUMA awareness, asynchronous double
 * buffering", tech-renaissance.cn/blog/?p=481, §四): two device slots A/B;
 * the host-to-device copy of batch k+1 on the copy stream overlaps the
 * kernel on batch k on the compute stream, with CUDA events handing each
 * slot over.  The station owns only its events; slots, streams and host
 * buffers belong to the caller.
 */
typedef struct tr_transfer_station tr_transfer_station;

/* Bytes one device slot needs for a batch of N images: the slot layout is
 * [N images][N records][filler image][filler record][scheduling workspace],
 * each zone starting on a 256-byte boundary (the article's
 * [labels][padding][image] zones, §四).  Slots without room for the filler
 * zones cannot take short batches or records; slots without room for the
 * workspace run the statically scheduled kernel.                          */
size_t tr_ts_slot_bytes(int N, int H, int W, int C);

/*   device        CUDA device ordinal the slots and streams belong to.
 *   d_slot        two device buffers of slot_bytes each (input slots A/B).
 *   copy_stream   stream for host-to-device copies (cudaStream_t as void*).
 *   compute_stream stream for the kernel.
 *   d2h_stream    stream for optional device-to-host copies of results, or
 *                 NULL when results stay on the device.
 * Errors: TR_ERR_INVALID_ARGUMENT for NULL slots/streams/out or a zero size,
 * TR_ERR_CUDA when events cannot be created.                                */
int tr_ts_create(int device, void* const d_slot[2], size_t slot_bytes,
                 void* copy_stream, void* compute_stream, void* d2h_stream,
                 tr_transfer_station** out);

/* Enqueue batch k: copy h_src (pinned host, N*H*W*C bytes) and, when
 * h_params is not NULL, its N records (pinned host) into slot k%2 on the copy
 * stream once the kernel that last read that slot has finished; run
 * tr_fused_norm from the slot into d_dst (device) on the compute stream after
 * the copy; when h_dst is not NULL, copy d_dst to h_dst (pinned host) on the
 * d2h stream after the kernel.  d_dst must not be reused by the caller before
 * the work it receives has finished (tr_ts_sync, or stream order on the
 * compute stream).  Returns without waiting for the GPU.
 * *batch_index (may be NULL) receives k.                                     */
int tr_ts_submit(tr_transfer_station* ts, const uint8_t* h_src, const tr_aug_param* h_params,
                 void* d_dst, void* h_dst, int N, int H, int W, int C,
                 const float* mean, const float* std, int out_dtype, int out_layout,
                 long long* batch_index);

/* tr_ts_submit for a short batch: h_src holds n_valid images (1 <= n_valid
 * <= N) and h_params, when not NULL, n_valid records; images n_valid..N-1 of
 * the batch repeat the filler, so that every batch has N images (the
 * article's incomplete-batch filling, TransferStation §四.1: the engine sees
 * one batch size and one captured graph).  The filler is the first image and
 * record of the first batch this station received (its record is "no flip,
 * no erase" if that batch had none); both are kept in the slots' filler zones
 * and copied into place on the copy stream.  Errors as tr_ts_submit, and
 * TR_ERR_INVALID_ARGUMENT for n_valid outside 1..N or slots without room for
 * the filler zones (tr_ts_slot_bytes).                                       */
int tr_ts_submit_partial(tr_transfer_station* ts, const uint8_t* h_src, const tr_aug_param* h_params,
                         int n_valid, void* d_dst, void* h_dst, int N, int H, int W, int C,
                         const float* mean, const float* std, int out_dtype, int out_layout,
                         long long* batch_index);

/* Wait until everything submitted so far has finished, polling events; gives
 * up after timeout_ms milliseconds with TR_ERR_TIMEOUT (the work stays
 * queued; a later call may wait again).  timeout_ms < 0 waits without limit. */
int tr_ts_sync(tr_transfer_station* ts, int timeout_ms);

/* Waits (without limit) for submitted work, then destroys the events. */
int tr_ts_destroy(tr_transfer_station* ts);

/* ------------------------------------------------------------------------
 * tr_staging — the host side of the station: preprocessing workers (host
 * threads) write samples into two caller-owned host zones A/B, one batch per
 * zone, while the station uploads the other zone (the TransferStation of
 * "(10) Multi-threaded preprocessing, NUMA awareness, asynchronous double
 * buffering", tech-renaissance.cn/blog/?p=481, §四: a buffer that holds a
 * whole batch, or the last samples once the data has run out, becomes
 * readable, and the workers switch to the other buffer; §四.2: two ways of
 * placing samples).  Batch b lives in zone b % 2; a zone takes samples of one
 * batch at a time and is given back (released) once that batch's upload has
 * finished.  Every wait has a deadline.  Pure host code: no CUDA call except
 * in tr_ts_submit_staged.  All functions are thread-safe; any number of
 * producer threads and one consumer thread.
 */
typedef struct tr_staging tr_staging;

typedef enum tr_stage_mode {
    TR_STAGE_FAST = 0,         /* a shared counter hands out the next free place (§四.2) */
    TR_STAGE_REPRODUCIBLE = 1  /* sample s goes to batch s / N, place s % N, so every run
                                  lays batches out identically (§四.2)                     */
} tr_stage_mode;

/* A place claimed by a producer. */
typedef struct tr_stage_slot {
    uint8_t* image;            /* H*W*C bytes to write the sample's uint8 NHWC image to */
    tr_aug_param* record;      /* its record (read by the station when asked to)        */
    long long sample;          /* sample number = batch * N + index                     */
    long long batch;
    int index;                 /* place within the batch, 0..N-1                        */
    int zone;                  /* 0 = A, 1 = B                                          */
} tr_stage_slot;

/* A readable batch handed to the consumer: places 0..count-1 of one zone. */
typedef struct tr_stage_batch {
    uint8_t* images;           /* count images of H*W*C bytes, back to back             */
    tr_aug_param* records;     /* count records                                         */
    long long batch;
    int count;                 /* N, or 1..N for the last batch of closed data          */
    int zone;
} tr_stage_batch;

/* Bytes one zone needs: [N images][pad][N records], the record array on a
 * 256-byte boundary (the article's aligned zones, §四); 0 for a bad shape.   */
size_t tr_stage_zone_bytes(int N, int H, int W, int C);

/* zone: two non-overlapping host buffers of zone_bytes each (pinned memory,
 * e.g. cudaHostAlloc, for asynchronous uploads; any host memory works, the
 * upload is then synchronous), aligned to 4 bytes.  The staging area never
 * reads or writes the zones itself.  Errors: TR_ERR_INVALID_ARGUMENT.       */
int tr_stage_create(void* const zone[2], size_t zone_bytes, int N, int H, int W, int C, int mode,
                    tr_staging** out);

/* Producer: claim a place.  FAST mode ignores `sample` and takes the next
 * sample number; REPRODUCIBLE mode claims sample `sample` (>= 0).  Waits
 * until the zone of the sample's batch takes that batch (the consumer has
 * released the batch two before it): TR_ERR_TIMEOUT after timeout_ms
 * milliseconds (nothing claimed; timeout_ms < 0 waits without limit).
 * TR_END_OF_DATA once the data is closed and the sample lies beyond it.
 * TR_ERR_INVALID_ARGUMENT for a REPRODUCIBLE sample already claimed or whose
 * batch was already consumed.                                                */
int tr_stage_acquire(tr_staging* st, long long sample, int timeout_ms, tr_stage_slot* slot);

/* Producer: the sample in `slot` is written.  The batch turns readable when
 * its last place is committed.  TR_ERR_INVALID_ARGUMENT for a slot not
 * claimed, or committed twice.                                               */
int tr_stage_commit(tr_staging* st, const tr_stage_slot* slot);

/* End of the data ("every worker reports that samples ran out", §四): the
 * data set has total_samples samples, or, with -1, the ones claimed so far
 * (FAST: handed out; REPRODUCIBLE: up to the highest claimed sample).  Places
 * beyond it are refused (TR_END_OF_DATA); a short last batch becomes readable
 * once its places are committed.  TR_ERR_INVALID_ARGUMENT if already closed
 * or if total_samples is below a sample already claimed (FAST: differs from
 * the number handed out).                                                    */
int tr_stage_close(tr_staging* st, long long total_samples);

/* Consumer: the next batch in order, once readable; TR_ERR_TIMEOUT after
 * timeout_ms milliseconds (< 0: no limit); TR_END_OF_DATA after the last
 * batch of closed data.  The zone stays the consumer's until released.      */
int tr_stage_wait_readable(tr_staging* st, int timeout_ms, tr_stage_batch* batch);

/* Consumer: give the zone of `batch` back to the producers (for batch + 2).
 * TR_ERR_INVALID_ARGUMENT if that batch is not handed out.                   */
int tr_stage_release(tr_staging* st, long long batch);

/* Waits (without limit) for releases queued by tr_ts_submit_staged, then
 * frees the staging area.                                                    */
int tr_stage_destroy(tr_staging* st);

/* tr_ts_submit of a staged batch: uploads b->count images (and, when
 * with_records != 0, their records; else no flip and no erase) from the zone,
 * pads a short batch to N with the station's filler (tr_ts_submit_partial),
 * and releases the zone on the copy stream as soon as its host-to-device
 * copies have finished (a host function queued on the copy stream; it takes
 * the staging area's lock and makes no CUDA call).  Other arguments and
 * errors as tr_ts_submit; TR_ERR_INVALID_ARGUMENT when b is not a batch of
 * st handed out for N images of H*W*C bytes.  After a failed call the zone
 * may still be handed out: tr_ts_sync, then tr_stage_release (which answers
 * TR_ERR_INVALID_ARGUMENT if the queued release already gave it back).      */
int tr_ts_submit_staged(tr_transfer_station* ts, tr_staging* st, const tr_stage_batch* b, int with_records,
                        void* d_dst, void* h_dst, int N, int H, int W, int C, const float* mean,
                        const float* std, int out_dtype, int out_layout, long long* batch_index);

/* ------------------------------------------------------------------------
 * Diagnostics.
 */
/* Reads the device status word the kernels set when a bounded pipeline wait
 * runs out (bit 0); with clear != 0 resets it.  Synchronous (waits for the
 * current device).                                                          */
int tr_device_status(int* flags, int clear);

/* Geometry of the TILED kernel, for tuning on a given device (process-wide;
 * 0 keeps the default for that knob):
 *   band_bytes       source bytes per row band (default: about 32 KB of
 *                    output per band; the band height is the largest divisor
 *                    of H near the target, else the height that splits H into
 *                    as many bands as evenly as a fixed height allows;
 *                    lowered (down to half) where three CTAs would not fit an
 *                    SM — for 4-stage plans only when the launch overlaps the
 *                    previous one or gives each CTA fewer than five bands —
 *                    then lowered where a band's groups
 *                    leave the consumer threads' last stride mostly empty;
 *                    crop sources may lower it so that as many CTAs fit an
 *                    SM as for a compact source; the odd-row form, where each
 *                    CTA streams at least five bands, takes two stages and
 *                    the height that fits the most CTAs, up to four),
 *   stages           shared-memory input stages, 2..8 (default 3 for bands
 *                    above 8 KB of source, else 4; 2 for the odd-row form's
 *                    own planning),
 *   max_ctas_per_sm  cap on resident CTAs per SM (default: occupancy limit),
 *   flags            L2 policies (default: source loads and output stores
 *                    both evict-first): bit 0 normal-priority loads, bit 1
 *                    normal-priority stores, bit 2 evict-last stores (for a
 *                    consumer that reads the output from L2); bit 3 makes a
 *                    CTA release the next kernel in the stream only once its
 *                    copies are all issued (default: as soon as the previous
 *                    kernel has completed); bit 4
 *                    lets a CTA exit once its last store has read shared
 *                    memory instead of once the store has completed (the
 *                    grid's completion still covers the writes); bit 5 makes
 *                    a CTA wait for its first band's record before requesting
 *                    the band (default: the first band of a compact source is
 *                    requested at once, erased span included); bit 7 turns
 *                    off the rotated order of the output tile's 16-byte
 *                    shared-memory stores (a bank-conflict avoidance for
 *                    layouts whose groups span 64 bytes or more); bit 6 is a
 *                    test hook for the kernels' bounded waits: the first band
 *                    of a batch waits for 16 bytes that never arrive, its waits
 *                    run out after about a second, the launch returns with bit 0
 *                    of the device status word set and its output incomplete;
 *                    bit 10 makes the odd-row form write its output tile
 *                    element by element (default, for NHWC pixels of 2, 4, 6
 *                    or 12 bytes and NCHW plane runs of 32 bytes or more
 *                    when the launch gives each CTA at least five bands:
 *                    each group's output bytes moved to the tile's 16-byte
 *                    frame in registers and written with 16-byte stores,
 *                    2/4/8-byte stores only at its ends), bit 17 uses that
 *                    realignment however few bands a CTA gets (for NHWC
 *                    output with 1 or 3 channels the groups are then laid on
 *                    the output tile's 16-byte frame instead, a pixel and a
 *                    chunk boundary at once, so no realignment is needed;
 *                    bit 23 keeps the realigned pixel groups); bit 20 makes
 *                    the odd-row form store 16-byte binary16 NCHW plane runs
 *                    (2 or 3 channels) in plain element order (default: each
 *                    lane starts at word (lane / 8) % 4 of its run, so a
 *                    warp's stores fall on distinct banks); bit 26 keeps
 *                    those plane runs where H*W mod 8 is 0 or 1 (every odd
 *                    square size) and each CTA streams at least five bands
 *                    (default there: each thread converts the 8 + (C-1) *
 *                    (H*W mod 8) consecutive pixels that hold one 16-byte
 *                    chunk of every plane's output tile, and writes each
 *                    chunk with one aligned store);
 *                    records made on the GPU in the same call
 *                    (tr_fused_norm_sampled_ex with TR_LAUNCH_OVERLAP_PREVIOUS):
 *                    bit 21 makes each CTA read its first bands' records from
 *                    the sampler's output once the sampler has completed
 *                    (default: the CTA makes them with the sampler's steps,
 *                    the same bits, so those bands convert while the kernel
 *                    before drains), bit 22 has the producer warp make them
 *                    one after another (default: one consumer warp each, in
 *                    parallel), bit 25 makes only the records of a CTA's
 *                    first S bands (default: its first 2S where it has 2S
 *                    consumer warps, so that once its wait for the sampler
 *                    returns, its next S bands need no read of the sampler's
 *                    output);
 *                    crop sources: bit 8 reads 16-byte chunks even where 32-byte
 *                    chunks fit, bit 9 asks TMA for 128-byte L2 promotion;
 *                    compact sources: erased source spans are left out of a
 *                    band's copies (one copy more per erased row) only when
 *                    they save at least 256 bytes a row and not in a CTA's
 *                    first S bands; bit 11 leaves them out of the first S
 *                    bands too, bits 12..15 = v != 0 set the threshold to
 *                    (v - 1) * 128 bytes; bit 16 keeps the band height of
 *                    about 32 KB of output where it leaves fewer than three
 *                    CTAs on an SM (default, with the exceptions given under
 *                    band_bytes: the largest lower height, down to half, at
 *                    which three fit), bit 18 keeps that height
 *                    even where a band's last stride of consumer threads is
 *                    mostly empty (default: the largest lower height, down to
 *                    half, at which a band's groups fill at least 84 % of the
 *                    consumer threads' strides), bit 19 plans the odd-row
 *                    form like the aligned one.
 * Results do not depend on the geometry.  Errors: TR_ERR_INVALID_ARGUMENT
 * for negative values or stages of 1 or above 8.                            */
int tr_tune_tiled(int band_bytes, int stages, int max_ctas_per_sm, int flags);

/* Number of kernels this library has launched in this process. */
uint64_t tr_launch_count(void);

/* Static text for a status code. */
const char* tr_status_string(int status);

/* Text of the last CUDA error seen by this thread in this library ("" if none). */
const char* tr_last_error_message(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int tr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TR_FUSED_NORM_H */

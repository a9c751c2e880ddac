// Fused normalisation kernels for sm_103a (GB300).
//
// The operation is the one described in the Tech-Renaissance article
// "(11) FusedNormalization: fuse the last step of data augmentation into one
// memory traversal" (tech-renaissance.cn/blog/?p=487): ToTensor (x/255) and
// Normalize ((x - mean)/std) in one pass (§五), read from the mirrored or the
// original position when flipping (§五, §七), erased output set to +0 (§十二),
// binary32 or binary16 output (§六), with the 4-channel padded layout (§八).
// The article's implementation is x86 SIMD on the CPU; nothing of it carries
// over.  This file is a GPU design:
//
//  * TILED: a persistent kernel.  The batch is cut into units of R rows of one
//    image ("row bands").  One thread per CTA streams the source bytes of the
//    next bands into a ring of shared-memory stages with TMA bulk copies
//    (cp.async.bulk + mbarrier transaction counts), leaving out the 16-byte
//    chunks that lie wholly inside a wide erased span.  The other warps
//    convert groups of 8 (C=3), 16 (C=1), 8 (C=2) or 4 (C=4) pixels: the
//    mirrored gather is done by choosing source byte lanes with PRMT, the
//    byte becomes 2^23 + x by the same PRMT, one exact FADD removes 2^23 and
//    the channel's integer shift, one FFMA applies scale and bias.  Results go to a double-buffered
//    shared-memory output tile that one TMA bulk store per band (per plane
//    for NCHW) writes to global memory.  With a crop source
//    (tr_fused_norm_crop) the bands come from windows of a strided source
//    through a TMA tensor copy (cp.async.bulk.tensor): the source is
//    described as {chunk, chunk index, row, image} with 16- or 32-byte
//    chunks, so a window may start at any byte; consumers realign the first
//    chunk's offset with funnel shifts.  Rows (or output rows, or an output
//    pointer) that are not 16-byte aligned take an odd-row form: bands staged
//    from the 16-byte boundary below them, groups realigned in registers,
//    output tiles that follow the band's global alignment.
//    Launches are chained with programmatic dependent launch: a CTA releases
//    the next grid once the previous one has completed; a launch its caller
//    declared independent of the previous one starts its copies before that
//    grid has completed (TR_LAUNCH_OVERLAP_PREVIOUS).
//  * GENERIC: one thread per output pixel, any shape, stride and alignment.
//
// Both kernels compute each value as fma(x - shift_c, scale_c, bias_c), the
// subtraction exact (shift_c is 255*mean_c rounded to an integer), with the
// same binary32 operands, so they agree bit for bit.
//
// Every wait in device code is bounded: a TMA stage that does not complete
// within about a second sets bit 0 of the device status word, the CTA drains
// what it has in flight (again bounded) and returns.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "aug_sampling.cuh"
#include "internal.h"

namespace trfn {

// bit 0: a pipeline wait timed out; bit 1 (checked build): a bounds or
// alignment check failed, and g_bounds_site holds the first failing check's
// site number (reported in bits 8..15 of tr_device_status)
__device__ unsigned int g_device_status;
__device__ unsigned int g_bounds_site;

namespace {

// The checked build (compiled with -DTRFN_BOUNDS=1, libtrfn_bounds.so) tests
// every shared-memory and global range the tiled kernel copies, loads or
// stores against the buffer it belongs to (and the 16-byte rules of bulk
// copies) before the access; a failed check sets bit 1 of the status word,
// records its site and skips the access.  A skipped copy leaves its stage
// incomplete, so the bounded waits then end the CTA.  In the default build
// TRFN_CHECK is the constant true and its condition is not compiled.
#ifndef TRFN_BOUNDS
#define TRFN_BOUNDS 0
#endif
#if TRFN_BOUNDS
__device__ __noinline__ void bounds_fail(int site) {
    atomicCAS(&g_bounds_site, 0u, (unsigned)(site & 255));
    atomicOr(&g_device_status, 2u);
}
#define TRFN_CHECK(cond, site) ((cond) ? true : (bounds_fail(site), false))
#else
#define TRFN_CHECK(cond, site) true
#endif

// Start of the dynamic shared memory (the same bytes as the kernels' smem).
extern __shared__ __align__(128) uint8_t trfn_dyn_smem[];

constexpr int kMaxStages = 8;
constexpr int kHeaderBytes = 384;          // mbarriers + per-stage unit records
constexpr int kEmptyOffset = 64;           // full[8] at 0, empty[8] at 64
constexpr int kRecOffset = 128;            // UnitRec[8] at 128
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s
constexpr uint32_t kStatusTimeout = 1u;

// ------------------------------------------------------------------ PTX ---

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named barrier 1 over `nthreads` threads; returns whether any of them passed
// a non-zero flag.
__device__ __forceinline__ bool named_barrier_or(uint32_t nthreads, bool flag) {
    uint32_t any;
    asm volatile(
        "{\n\t.reg .pred q, p;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(any)
        : "r"((uint32_t)flag), "r"(nthreads)
        : "memory");
    return any != 0;
}

// Programmatic dependent launch: wait for the preceding grid in the stream
// (complete, memory visible) / let the next grid start its prologue.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; false after ~1 s.
__device__ __noinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; it < (1u << 28); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

// TMA bulk copy global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst_smem),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Same, with an L2 eviction-priority policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst_smem, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst_smem),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// TMA tensor copy of one box of a 4-d tensor map into shared memory.
__device__ __forceinline__ void tensor_g2s_4d(uint32_t dst_smem, const void* tmap, int c0, int c1, int c2, int c3,
                                              uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst_smem),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
        : "memory");
}

// TMA bulk copy shared -> global in the current bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(src_smem), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_s2g_hint(void* dst, uint32_t src_smem, uint32_t bytes,
                                              uint64_t policy) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                 "r"(src_smem), "r"(bytes), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ arithmetic --

// Byte `sel` (0..3) of `word` minus the channel's integer shift, as a
// binary32 value: PRMT builds the pattern 0x4B0000xx = 2^23 + x and `base`
// is 2^23 + shift (an integer below 2^24), so the subtraction is exact.
__device__ __forceinline__ float byte_minus_shift(uint32_t word, uint32_t sel, float base) {
    const uint32_t bits = __byte_perm(word, 0x00004B00u, 0x5440u | sel);
    return __fsub_rn(__uint_as_float(bits), base);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);   // round to nearest even
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Pixels per group: the smallest pixel count whose bytes fill 16 (C=1,2,4)
// or 24 (C=3) bytes, so that a group's source is one or three aligned words.
template <int C>
struct Group {
    static constexpr int P = (C == 3) ? 8 : 16 / C;
    static constexpr int kBytes = P * C;   // 16 or 24
    static constexpr int kWords = kBytes / 4;
};

// Converts one group.  Output element k is pixel k/C, channel k%C; with FLIP
// its source is pixel P-1-k/C of the mirrored group (same channel).
template <int C, bool FLIP>
__device__ __forceinline__ void convert_group(const uint32_t (&w)[Group<C>::kWords], const float* base,
                                              const float* scale, const float* bias,
                                              float (&v)[Group<C>::kBytes]) {
    constexpr int P = Group<C>::P;
#pragma unroll
    for (int k = 0; k < P * C; ++k) {
        const int i = k / C;
        const int c = k % C;
        const int sb = FLIP ? ((P - 1 - i) * C + c) : k;
        v[k] = __fmaf_rn(byte_minus_shift(w[sb >> 2], sb & 3, base[c]), scale[c], bias[c]);
    }
}

// ---------------------------------------------------------------- tiled ---

struct TiledParams {
    CUtensorMap tmap;      // crop sources: {chunk, chunk index, row, image} of the source
    const int32_t* crop;   // crop sources: per-image window origin {top, left}, or null
    int src_H, src_W;      // crop sources: source image size
    uint32_t in_pitch;     // bytes per row of an input stage (W*C; chunks*chunk bytes for crop sources)
    int chunk_shift;       // crop sources: log2 of the tensor's innermost chunk (4 or 5: 16 or 32 bytes)
    const uint8_t* src;
    uint8_t* dst;
    const tr_aug_param* aug;
    int N, H, W;
    int R;                 // rows per band
    int bands;             // bands per image
    int num_units;         // N * bands
    int gpr;               // groups per row, W / P
    uint64_t gpr_inv;      // ceil(2^32 / gpr): g / gpr == (g * gpr_inv) >> 32 for g, gpr < 2^16
    uint64_t wc_inv;       // ceil(2^32 / (W*C)): e / (W*C) the same way, for e * W*C < 2^31
    uint64_t src_floor16;  // rows not a multiple of 16 bytes: the source's bytes rounded down to 16
    uint32_t in_stage;     // bytes per input stage (R*W*C, multiple of 16)
    uint32_t out_stage;    // bytes per output stage
    uint32_t plane_bytes;  // NCHW: bytes per plane of one band in the output stage (R*W*ob)
    int stages;
    unsigned int* ws;      // scheduling workspace (ticket counters, finished CTAs), or null
    int hints;             // tr_tune_tiled flags (include/tr_fused_norm.h): L2 policies
                           // (bits 0-2), late release of the next grid (3), exit after
                           // the last store's shared-memory reads (4), record before the
                           // first band (5), bounded-wait test hook (6), unrotated tile
                           // stores (7), erased-span rule (11, 12-15); set by the launch:
                           // overlap the previous grid (8), records written by it (9),
                           // odd-row element stores (10), plain order of 16-byte
                           // odd-row NCHW plane runs (20), odd-row NHWC groups aligned
                           // to the output tile (24), a sampled launch's first
                           // records made by the producer warp (22)
    float base[4];         // 2^23 + shift_c (see byte_minus_shift)
    float scale[4];
    float bias[4];
    // several batches in one launch (tr_fused_norm_batches): images per
    // batch, and each batch's source, output and records; image n of the
    // launch is image n % nb of batch n / nb.  0 = one batch (src, dst, aug).
    int nb;
    uint32_t smem_bytes;        // dynamic shared memory of a CTA (checked build)
    uint64_t src_batch_bytes;   // compact sources: bytes of one batch (checked build)
    uint64_t dst_batch_bytes;   // output bytes of one batch (checked build)
    // records made on the GPU (tr_fused_norm_sampled): the sampler's
    // settings, with which the kernel makes its CTAs' first records
    SampleSpec spec;
    const uint8_t* bsrc[TR_MAX_BATCHES];
    uint8_t* bdst[TR_MAX_BATCHES];
    const tr_aug_param* baug[TR_MAX_BATCHES];
};

// What a tiled launch covers, fixed at compile time so that each form
// carries only its own code: one batch whose records are read (or absent),
// several batches of one shape (tr_fused_norm_batches), or one batch whose
// records a sampler grid is writing while the launch starts, of which the
// kernel makes its CTAs' first ones itself (tr_fused_norm_sampled).
constexpr int kModeBatch = 0;
constexpr int kModeBatches = 1;
constexpr int kModeSampled = 2;

// Image n of the launch: its batch's source and output base pointers and
// its index in that batch.
struct ImageRef {
    const uint8_t* src;
    uint8_t* dst;
    int n;
};

template <int MODE>
__device__ __forceinline__ ImageRef image_ref(const TiledParams& p, int n) {
    if constexpr (MODE == kModeBatches) {
        const int k = n / p.nb;
        return ImageRef{p.bsrc[k], p.bdst[k], n - k * p.nb};
    } else {
        return ImageRef{p.src, p.dst, n};
    }
}

// Image n's record ({0} without records).
template <int MODE>
__device__ __forceinline__ tr_aug_param image_record(const TiledParams& p, int n) {
    tr_aug_param r = {0, 0, 0, 0, 0};
    if constexpr (MODE == kModeBatches) {
        const int k = n / p.nb;
        const tr_aug_param* a = p.baug[k];
        if (a != nullptr) r = a[n - k * p.nb];
    } else {
        if (p.aug != nullptr) r = p.aug[n];
    }
    return r;
}

// Per-stage record of the unit held in that stage.
struct UnitRec {
    int n, y_begin, rows;
    int flags;             // bit 0: flip; bits 8..12: byte offset of the window in its first chunk
    int erow_lo, erow_hi;  // erased output rows [lo, hi), clipped to the image
    int ecol_lo, ecol_hi;  // erased output columns [lo, hi), clipped
};
static_assert(sizeof(UnitRec) == 32, "UnitRec layout");
static_assert(kRecOffset + kMaxStages * sizeof(UnitRec) <= kHeaderBytes, "header holds barriers and records");

// Source bytes of unit u: rows [y_begin, y_begin + rows) of image n.
struct Band {
    int n, y_begin, rows;
};

__device__ __forceinline__ Band band_of(const TiledParams& p, int u) {
    Band b;
    b.n = u / p.bands;
    b.y_begin = (u - b.n * p.bands) * p.R;
    b.rows = min(p.R, p.H - b.y_begin);
    return b;
}

// Source bytes are read exactly once: by default they enter L2 with
// evict-first priority.
__device__ __forceinline__ void load_bytes(const TiledParams& p, uint32_t dst, const void* src, uint32_t bytes,
                                           uint32_t bar) {
    if (p.hints & 1) bulk_g2s(dst, src, bytes, bar);
    else bulk_g2s_hint(dst, src, bytes, bar, policy_evict_first());
}

// Fills stage s with unit u: records the unit for the consumers, arrives on
// full[s] with the byte count and issues the band's copies, leaving out (when
// allowed and worth a copy) the 16-byte chunks that lie wholly inside the
// erased source span of the erased
// rows.
template <int C, bool CROP, bool ODD, int MODE>
__device__ __forceinline__ void issue_unit(const TiledParams& p, int u, int s, uint8_t* smem,
                                           const tr_aug_param& a, bool allow_skip, int2 origin) {
    const Band b = band_of(p, u);
    const int y_begin = b.y_begin, rows = b.rows;
    int flip = 0, erow_lo = 0, erow_hi = 0, ecol_lo = 0, ecol_hi = 0;
    flip = (a.flip != 0);
    if (a.h > 0 && a.w > 0) {
        const long long y0 = a.y0, x0 = a.x0;
        const long long ylo = max(y0, 0ll), yhi = min(y0 + a.h, (long long)p.H);
        const long long xlo = max(x0, 0ll), xhi = min(x0 + a.w, (long long)p.W);
        if (ylo < yhi && xlo < xhi) {
            erow_lo = (int)ylo; erow_hi = (int)yhi;
            ecol_lo = (int)xlo; ecol_hi = (int)xhi;
        }
    }
    UnitRec* rec = reinterpret_cast<UnitRec*>(smem + kRecOffset) + s;
    rec->n = b.n; rec->y_begin = y_begin; rec->rows = rows; rec->flags = flip;
    rec->erow_lo = erow_lo; rec->erow_hi = erow_hi; rec->ecol_lo = ecol_lo; rec->ecol_hi = ecol_hi;

    if (CROP) {
        // The window's rows, from its 16-byte chunk on, as one box of R rows
        // (rows past the source image arrive as zeros and are not used).
        // the window origin (loaded by the caller with the record), clamped
        const int cy = min(max(origin.x, 0), p.src_H - p.H);
        const int cx = min(max(origin.y, 0), p.src_W - p.W);
        const int xb = cx * C;
        rec->flags = flip | ((xb & ((1 << p.chunk_shift) - 1)) << 8);
        const uint32_t bar = smem_u32(smem) + 8u * (uint32_t)s;
        const uint32_t box_dst = smem_u32(smem + kHeaderBytes) + (uint32_t)s * p.in_stage;
        mbar_arrive_expect_tx(bar, (uint32_t)p.R * p.in_pitch);
        if (TRFN_CHECK((uint64_t)p.R * p.in_pitch <= p.in_stage && (box_dst & 15u) == 0, 1))
            tensor_g2s_4d(box_dst, &p.tmap, 0, xb >> p.chunk_shift, cy + y_begin, b.n, bar,
                          (p.hints & 1) ? policy_evict_last() : policy_evict_first());
        return;
    }

    if (ODD) {
        // Rows that are not a multiple of 16 bytes: the band's bytes, from
        // the 16-byte boundary below them, by one bulk copy; the band then
        // starts `off` bytes into the stage (consumers realign), and any
        // bytes past the source's last whole 16 are copied by this thread.
        // (offsets from the image's batch, whose source starts 16-byte aligned)
        const ImageRef im = image_ref<MODE>(p, b.n);
        const uint64_t L = (uint64_t)p.W * C;
        const uint64_t base = ((uint64_t)im.n * p.H + y_begin) * L;
        const uint64_t end = base + (uint64_t)rows * L;
        const uint64_t a0 = base & ~15ull;
        uint64_t bulk_end = (end + 15) & ~15ull;
        if (bulk_end > p.src_floor16) bulk_end = p.src_floor16 > a0 ? p.src_floor16 : a0;
        rec->flags = flip | (int)((uint32_t)(base - a0) << 8);
        uint8_t* stage = smem + kHeaderBytes + (size_t)s * p.in_stage;
        for (uint64_t i = bulk_end; i < end; ++i)
            if (TRFN_CHECK(i - a0 < p.in_stage && i < p.src_batch_bytes, 2)) stage[i - a0] = im.src[i];
        const uint32_t bar = smem_u32(smem) + 8u * (uint32_t)s;   // full[s]
        const uint32_t bulk = (uint32_t)(bulk_end - a0);
        const uint32_t missing = ((p.hints & 64) && u == 0) ? 16u : 0u;   // bounded-wait test hook
        mbar_arrive_expect_tx(bar, bulk + missing);
        if (bulk > 0 && TRFN_CHECK(bulk <= p.in_stage && a0 + bulk <= p.src_batch_bytes && (bulk & 15u) == 0 &&
                                       ((uintptr_t)(im.src + a0) & 15u) == 0 && (smem_u32(stage) & 15u) == 0,
                                   3))
            load_bytes(p, smem_u32(stage), im.src + a0, bulk, bar);
        return;
    }

    const uint32_t L = (uint32_t)p.W * C;
    const ImageRef im = image_ref<MODE>(p, b.n);
    const uint8_t* g = im.src + ((size_t)im.n * p.H + y_begin) * L;
    const uint32_t sdst = smem_u32(smem + kHeaderBytes) + (uint32_t)s * p.in_stage;
    const uint32_t bar = smem_u32(smem) + 8u * (uint32_t)s;   // full[s]
    const uint32_t total = (uint32_t)rows * L;
    // Rows of this band inside the erase rectangle, and the 16-byte aligned
    // part of their erased source span (rows start 16-byte aligned).
    const int r_lo = max(erow_lo - y_begin, 0);
    const int r_hi = min(erow_hi - y_begin, rows);
    const int xs_lo = flip ? p.W - ecol_hi : ecol_lo;
    const int xs_hi = flip ? p.W - ecol_lo : ecol_hi;
    const uint32_t a_lo = ((uint32_t)xs_lo * C + 15u) & ~15u;
    const uint32_t a_hi = ((uint32_t)xs_hi * C) & ~15u;
    // test hook for the bounded waits: unit 0's stage then never completes
    const uint32_t missing = ((p.hints & 64) && u == 0) ? 16u : 0u;
    // An erased row's span is left out only when it saves at least
    // skip_min bytes: each one costs a copy more (tr_tune_tiled flags bits
    // 12..15 = v: 0 keeps 256 bytes, else (v - 1) * 128).
    const int v = (p.hints >> 12) & 15;
    const uint32_t skip_min = v == 0 ? 256u : (uint32_t)(v - 1) * 128u;
    // (checked build) a range [at, at + n) of the band: inside the stage and
    // the batch's source, 16-byte aligned at both ends
    auto band_range_ok = [&](uint32_t at, uint32_t n) {
        return (uint64_t)at + n <= total && total <= p.in_stage &&
               (uint64_t)(g - im.src) + at + n <= p.src_batch_bytes && ((uintptr_t)(g + at) & 15u) == 0 &&
               ((sdst + at) & 15u) == 0 && (n & 15u) == 0;
    };
    (void)band_range_ok;
    if (r_lo >= r_hi || a_hi <= a_lo || !allow_skip || a_hi - a_lo < skip_min) {
        mbar_arrive_expect_tx(bar, total + missing);
        if (TRFN_CHECK(band_range_ok(0, total), 4)) load_bytes(p, sdst, g, total, bar);
        return;
    }
    const uint32_t skipped = (uint32_t)(r_hi - r_lo) * (a_hi - a_lo);
    mbar_arrive_expect_tx(bar, total - skipped + missing);
    uint32_t pos = 0;
    for (int r = r_lo; r < r_hi; ++r) {
        const uint32_t seg_end = (uint32_t)r * L + a_lo;
        if (seg_end > pos && TRFN_CHECK(band_range_ok(pos, seg_end - pos), 5))
            load_bytes(p, sdst + pos, g + pos, seg_end - pos, bar);
        pos = (uint32_t)r * L + a_hi;
    }
    if (total > pos && TRFN_CHECK(band_range_ok(pos, total - pos), 5))
        load_bytes(p, sdst + pos, g + pos, total - pos, bar);
}

// Early form of issue_unit for a CTA's first unit (compact sources): the
// whole band is requested before the unit's record has arrived; only the
// expected byte count is posted, so the stage cannot complete before
// publish_unit has written the record and arrived.
template <int C, int MODE>
__device__ __forceinline__ void issue_unit_uncut(const TiledParams& p, int u, int s, uint8_t* smem) {
    const Band b = band_of(p, u);
    const uint32_t L = (uint32_t)p.W * C;
    const uint32_t total = (uint32_t)b.rows * L;
    const uint32_t bar = smem_u32(smem) + 8u * (uint32_t)s;
    const uint32_t missing = ((p.hints & 64) && u == 0) ? 16u : 0u;   // bounded-wait test hook
    mbar_expect_tx(bar, total + missing);
    const ImageRef im = image_ref<MODE>(p, b.n);
    const uint8_t* g = im.src + ((size_t)im.n * p.H + b.y_begin) * L;
    const uint32_t sdst = smem_u32(smem + kHeaderBytes) + (uint32_t)s * p.in_stage;
    if (TRFN_CHECK(total <= p.in_stage && (uint64_t)(g - im.src) + total <= p.src_batch_bytes &&
                       ((uintptr_t)g & 15u) == 0 && (sdst & 15u) == 0 && (total & 15u) == 0,
                   6))
        load_bytes(p, sdst, g, total, bar);
}

// Writes unit u's record (flip, clipped erase rectangle) for stage s and
// arrives on full[s] (release: consumers that see the phase see the record).
__device__ __forceinline__ void publish_unit(const TiledParams& p, int u, int s, uint8_t* smem,
                                             const tr_aug_param& a) {
    const Band b = band_of(p, u);
    int erow_lo = 0, erow_hi = 0, ecol_lo = 0, ecol_hi = 0;
    if (a.h > 0 && a.w > 0) {
        const long long y0 = a.y0, x0 = a.x0;
        const long long ylo = max(y0, 0ll), yhi = min(y0 + a.h, (long long)p.H);
        const long long xlo = max(x0, 0ll), xhi = min(x0 + a.w, (long long)p.W);
        if (ylo < yhi && xlo < xhi) {
            erow_lo = (int)ylo; erow_hi = (int)yhi;
            ecol_lo = (int)xlo; ecol_hi = (int)xhi;
        }
    }
    UnitRec* rec = reinterpret_cast<UnitRec*>(smem + kRecOffset) + s;
    rec->n = b.n; rec->y_begin = b.y_begin; rec->rows = b.rows; rec->flags = (a.flip != 0);
    rec->erow_lo = erow_lo; rec->erow_hi = erow_hi; rec->ecol_lo = ecol_lo; rec->ecol_hi = ecol_hi;
    mbar_arrive(smem_u32(smem) + 8u * (uint32_t)s);
}

// Writes a group's Q 16-byte output chunks to o.  Consecutive groups sit Q*16
// bytes apart, so when Q is a power of two the threads of a quarter-warp
// (eight 16-byte stores per shared-memory wavefront) would hit the same banks
// with chunk k: 8-way conflicts for Q >= 8, 4-way for Q = 4.  Each thread
// then stores its chunks rotated by a per-group amount (select stages on
// registers, no local memory), which puts the eight stores of a wavefront on
// eight different bank groups.  Measured at 256x224x224: binary32 NHWC4
// from 0.56 to 0.94 of the copy peak, Q = 4 layouts 1-6 % faster; for Q = 2
// (2-way conflicts) the selects cost more than they save, so it stays off.
template <int Q>
__device__ __forceinline__ void store_chunks(uint8_t* o, uint4 (&ch)[Q], int g, bool rotate) {
    constexpr bool kPow2 = Q >= 4 && (Q & (Q - 1)) == 0;
    if (kPow2 && rotate) {
        const int rot = (Q >= 8 ? g : ((g * Q) >> 3)) & (Q - 1);
#pragma unroll
        for (int b = 1; b < Q; b <<= 1) {
            const bool sw = (rot & b) != 0;
            uint4 t[Q];
#pragma unroll
            for (int i = 0; i < Q; ++i) t[i] = sw ? ch[(i + b) % Q] : ch[i];
#pragma unroll
            for (int i = 0; i < Q; ++i) ch[i] = t[i];
        }
        // ch[k] now holds chunk (k + rot) % Q
#pragma unroll
        for (int k = 0; k < Q; ++k) reinterpret_cast<uint4*>(o)[(k + rot) & (Q - 1)] = ch[k];
    } else {
#pragma unroll
        for (int k = 0; k < Q; ++k) reinterpret_cast<uint4*>(o)[k] = ch[k];
    }
}

template <int C, int OUT_F16, int LAYOUT>
__device__ __forceinline__ void store_group(const TiledParams& p, uint8_t* sout, int r, int gx,
                                            const float (&v)[Group<C>::kBytes]) {
    constexpr int P = Group<C>::P;
    constexpr int OB = OUT_F16 ? 2 : 4;
    const int g = r * p.gpr + gx;   // the group's index in the band: its output sits at g * Q * 16
    const bool rotate = !(p.hints & 128);
    // (checked build) the group's outputs lie in the output tile
    if (!TRFN_CHECK(LAYOUT == TR_LAYOUT_NCHW
                        ? (size_t)(C - 1) * p.plane_bytes + ((size_t)r * p.W + (size_t)(gx + 1) * P) * OB <=
                                  p.out_stage &&
                              ((size_t)r * p.W + (size_t)(gx + 1) * P) * OB <= p.plane_bytes
                        : ((size_t)r * p.W + (size_t)(gx + 1) * P) * (LAYOUT == TR_LAYOUT_NHWC4 ? 4 : C) * OB <=
                              p.out_stage,
                    9))
        return;
    if (LAYOUT == TR_LAYOUT_NHWC) {
        uint8_t* o = sout + ((size_t)r * p.W + (size_t)gx * P) * C * OB;
        if (OUT_F16) {
            constexpr int Q = P * C / 8;
            uint4 ch[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                ch[q].x = pack_half2(v[8 * q + 0], v[8 * q + 1]);
                ch[q].y = pack_half2(v[8 * q + 2], v[8 * q + 3]);
                ch[q].z = pack_half2(v[8 * q + 4], v[8 * q + 5]);
                ch[q].w = pack_half2(v[8 * q + 6], v[8 * q + 7]);
            }
            store_chunks<Q>(o, ch, g, rotate);
        } else {
            constexpr int Q = P * C / 4;
            uint4 ch[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q)
                ch[q] = make_uint4(__float_as_uint(v[4 * q + 0]), __float_as_uint(v[4 * q + 1]),
                                   __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
            store_chunks<Q>(o, ch, g, rotate);
        }
    } else if (LAYOUT == TR_LAYOUT_NHWC4) {
        // four channels per pixel, channels C..3 are +0
        uint8_t* o = sout + ((size_t)r * p.W + (size_t)gx * P) * 4 * OB;
        auto val = [&](int i, int c) { return c < C ? v[i * C + c] : 0.0f; };
        if (OUT_F16) {
            constexpr int Q = P / 2;
            uint4 ch[Q];
#pragma unroll
            for (int i = 0; i < P; i += 2) {
                ch[i / 2].x = pack_half2(val(i, 0), val(i, 1));
                ch[i / 2].y = pack_half2(val(i, 2), val(i, 3));
                ch[i / 2].z = pack_half2(val(i + 1, 0), val(i + 1, 1));
                ch[i / 2].w = pack_half2(val(i + 1, 2), val(i + 1, 3));
            }
            store_chunks<Q>(o, ch, g, rotate);
        } else {
            constexpr int Q = P;
            uint4 ch[Q];
#pragma unroll
            for (int i = 0; i < P; ++i)
                ch[i] = make_uint4(__float_as_uint(val(i, 0)), __float_as_uint(val(i, 1)),
                                   __float_as_uint(val(i, 2)), __float_as_uint(val(i, 3)));
            store_chunks<Q>(o, ch, g, rotate);
        }
    } else {  // NCHW: channel c of the group goes to plane c
#pragma unroll
        for (int c = 0; c < C; ++c) {
            uint8_t* o = sout + (size_t)c * p.plane_bytes + ((size_t)r * p.W + (size_t)gx * P) * OB;
            if (OUT_F16) {
                if (P % 8 == 0) {
#pragma unroll
                    for (int q = 0; q < P / 8; ++q) {
                        uint4 t;
                        t.x = pack_half2(v[(8 * q + 0) * C + c], v[(8 * q + 1) * C + c]);
                        t.y = pack_half2(v[(8 * q + 2) * C + c], v[(8 * q + 3) * C + c]);
                        t.z = pack_half2(v[(8 * q + 4) * C + c], v[(8 * q + 5) * C + c]);
                        t.w = pack_half2(v[(8 * q + 6) * C + c], v[(8 * q + 7) * C + c]);
                        reinterpret_cast<uint4*>(o)[q] = t;
                    }
                } else {  // P == 4
                    uint2 t;
                    t.x = pack_half2(v[0 * C + c], v[1 * C + c]);
                    t.y = pack_half2(v[2 * C + c], v[3 * C + c]);
                    *reinterpret_cast<uint2*>(o) = t;
                }
            } else {
#pragma unroll
                for (int q = 0; q < P / 4; ++q)
                    reinterpret_cast<float4*>(o)[q] =
                        make_float4(v[(4 * q + 0) * C + c], v[(4 * q + 1) * C + c],
                                    v[(4 * q + 2) * C + c], v[(4 * q + 3) * C + c]);
            }
        }
    }
}

// Rows that are not a multiple of 16 bytes: the output tile mirrors the
// band's global alignment (it starts at the band's global address mod 16,
// per plane for NCHW), so its bulk store can cover the 16-byte aligned
// middle; groups are written element by element, only their kv valid pixels.
template <int C, int OUT_F16, int LAYOUT, int MODE>
__device__ __forceinline__ uint32_t odd_shift(const TiledParams& p, const UnitRec& rec, int c) {
    constexpr int OC = (LAYOUT == TR_LAYOUT_NHWC4) ? 4 : C;
    constexpr int OB = OUT_F16 ? 2 : 4;
    const ImageRef im = image_ref<MODE>(p, rec.n);
    size_t e;   // the band's first output element in the plane or the batch
    if (LAYOUT == TR_LAYOUT_NCHW) e = (((size_t)im.n * C + c) * p.H + rec.y_begin) * p.W;
    else e = ((size_t)im.n * p.H + rec.y_begin) * p.W * OC;
    return (uint32_t)((uintptr_t)(im.dst + e * OB) & 15u);
}

// Writes len bytes (at least 16 - (s0 & 15), a multiple of EB) of the word
// stream w to tile + s0 (s0 a multiple of EB, tile 16-byte aligned), using
// only 16-byte stores for the chunks the range covers whole and at most three
// 2-, 4- or 8-byte stores at each end.  The stream is first moved to the
// tile's 16-byte frame: a funnel shift by s0 & 3 bytes, then a shift by
// (s0 >> 2) & 3 words in two select steps (registers only).  A chunk shared
// with a neighbouring group receives only this group's bytes, so threads
// writing neighbouring groups never touch the same bytes.
template <int NW, int EB>
__device__ __forceinline__ void put_stream(uint8_t* tile, uint32_t s0, uint32_t len, const uint32_t (&w)[NW]) {
    constexpr int NC = (4 * NW + 30) / 16;   // 16-byte chunks the range can touch
    constexpr int NO = 4 * NC;
    const uint32_t d = s0 & 15u, e = d + len;
    uint8_t* a = tile + (s0 - d);
    uint32_t sb[NW + 1];
    if (EB >= 4) {
#pragma unroll
        for (int i = 0; i < NW; ++i) sb[i] = w[i];
        sb[NW] = 0u;
    } else {
        const uint32_t db = (d & 3u) * 8u;
        sb[0] = __funnelshift_l(0u, w[0], db);
#pragma unroll
        for (int i = 1; i < NW; ++i) sb[i] = __funnelshift_l(w[i - 1], w[i], db);
        sb[NW] = __funnelshift_l(w[NW - 1], 0u, db);
    }
    const uint32_t dw = d >> 2;
    uint32_t t1[NO], o[NO];
#pragma unroll
    for (int j = 0; j < NO; ++j) {
        const uint32_t x0 = j <= NW ? sb[j] : 0u;
        const uint32_t x1 = (j >= 1 && j - 1 <= NW) ? sb[j - 1] : 0u;
        t1[j] = (dw & 1u) ? x1 : x0;
    }
#pragma unroll
    for (int j = 0; j < NO; ++j) o[j] = (dw & 2u) ? (j >= 2 ? t1[j - 2] : 0u) : t1[j];
    // the first chunk's part from byte d on
    if (d != 0) {
        const uint32_t s = 16u - d;
        if (s & 8u) *reinterpret_cast<uint2*>(a + 8) = make_uint2(o[2], o[3]);
        if (s & 4u) *reinterpret_cast<uint32_t*>(a + ((s & 8u) ? 4 : 12)) = (s & 8u) ? o[1] : o[3];
        if (EB < 4 && (s & 2u)) {
            const uint32_t lo = (d & 4u) ? o[1] : o[0], hi = (d & 4u) ? o[3] : o[2];
            *reinterpret_cast<uint16_t*>(a + d) = (uint16_t)(((d & 8u) ? hi : lo) >> 16);
        }
    }
    // whole chunks
    const uint32_t kt = e >> 4;
#pragma unroll
    for (int k = 0; k < NC; ++k)
        if ((k > 0 || d == 0) && (uint32_t)k < kt)
            *reinterpret_cast<uint4*>(a + 16 * k) = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
    // the last chunk's part below byte e & 15
    const uint32_t t = e & 15u;
    if (t != 0) {
        uint32_t c0 = o[4], c1 = o[5], c2 = o[6], c3 = o[7];
#pragma unroll
        for (int k = 2; k < NC; ++k)
            if (kt == (uint32_t)k) { c0 = o[4 * k]; c1 = o[4 * k + 1]; c2 = o[4 * k + 2]; c3 = o[4 * k + 3]; }
        uint8_t* q = a + 16u * kt;
        if (t & 8u) *reinterpret_cast<uint2*>(q) = make_uint2(c0, c1);
        if (t & 4u) *reinterpret_cast<uint32_t*>(q + (t & 8u)) = (t & 8u) ? c2 : c0;
        if (EB < 4 && (t & 2u)) {
            const uint32_t lo = (t & 4u) ? c1 : c0, hi = (t & 4u) ? c3 : c2;
            *reinterpret_cast<uint16_t*>(q + (t & 12u)) = (uint16_t)((t & 8u) ? hi : lo);
        }
    }
}

template <int C, int OUT_F16, int LAYOUT, int MODE>
__device__ __forceinline__ void store_group_odd(const TiledParams& p, uint8_t* sout, const UnitRec& rec, int r,
                                                int gx, int kv, const float (&v)[Group<C>::kBytes]) {
    constexpr int P = Group<C>::P;
    constexpr int OC = (LAYOUT == TR_LAYOUT_NHWC4) ? 4 : C;
    constexpr int OB = OUT_F16 ? 2 : 4;
    auto put = [&](uint8_t* q, float x) {
        if (OUT_F16) *reinterpret_cast<__half*>(q) = __float2half_rn(x);
        else *reinterpret_cast<float*>(q) = x;
    };
    // Register realignment pays where the element path stores 2-, 4- or
    // 12-byte pixels or short planes element by element: NHWC pixels of 2, 4,
    // 6 or 12 bytes, NCHW plane runs of 32 bytes or more.  Pixels of 8 or 16
    // bytes keep one aligned store each, and 16-byte plane runs would spend
    // more on the shifts than they save (measured at 256x299x299).
    constexpr bool kStreamNHWC = LAYOUT == TR_LAYOUT_NHWC && (C * OB) % 8 != 0;
    constexpr bool kStreamNCHW = LAYOUT == TR_LAYOUT_NCHW && P * OB >= 32;
    const bool streams = !(p.hints & 1024);
    // (checked build) the group's outputs, after the tile's alignment shift
    // (below 16 bytes), lie in the output tile (per plane for NCHW)
    if (!TRFN_CHECK(LAYOUT == TR_LAYOUT_NCHW
                        ? (size_t)(C - 1) * p.plane_bytes + p.plane_bytes <= p.out_stage &&
                              15 + ((size_t)r * p.W + (size_t)gx * P + kv) * OB <= p.plane_bytes
                        : 15 + ((size_t)r * p.W + (size_t)gx * P + kv) * OC * OB <= p.out_stage,
                    10))
        return;
    if (kStreamNHWC && streams) {
        // the group's kv pixels are one run of output bytes
        constexpr int NW = P * C * OB / 4;
        const uint32_t s0 = odd_shift<C, OUT_F16, LAYOUT, MODE>(p, rec, 0) + ((uint32_t)r * p.W + (uint32_t)gx * P) * (C * OB);
        const uint32_t len = (uint32_t)kv * (C * OB);
        if ((s0 & 15u) + len >= 16u) {
            uint32_t w[NW];
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                if constexpr (OUT_F16 != 0) w[i] = pack_half2(v[2 * i], v[2 * i + 1]);
                else w[i] = __float_as_uint(v[i]);
            }
            put_stream<NW, OB>(sout, s0, len, w);
            return;
        }
    }
    if (kStreamNCHW && streams) {
        // per plane, the group's kv pixels are one run of output bytes
        constexpr int NW = P * OB / 4;
        const uint32_t at = ((uint32_t)r * p.W + (uint32_t)gx * P) * OB;
        const uint32_t len = (uint32_t)kv * OB;
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const uint32_t s0 = odd_shift<C, OUT_F16, LAYOUT, MODE>(p, rec, c) + at;
            uint8_t* plane = sout + (size_t)c * p.plane_bytes;
            if ((s0 & 15u) + len >= 16u) {
                uint32_t w[NW];
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    if constexpr (OUT_F16 != 0) w[i] = pack_half2(v[(2 * i) * C + c], v[(2 * i + 1) * C + c]);
                    else w[i] = __float_as_uint(v[i * C + c]);
                }
                put_stream<NW, OB>(plane, s0, len, w);
            } else {
#pragma unroll
                for (int i = 0; i < P; ++i)
                    if (i < kv) put(plane + s0 + (size_t)i * OB, v[i * C + c]);
            }
        }
        return;
    }
    if (LAYOUT == TR_LAYOUT_NCHW) {
        // 16-byte binary16 plane runs (2 or 3 channels): the 32 lanes of a
        // warp hold consecutive groups, 16 bytes apart, so storing element i
        // of every lane's run at once hits each bank four times.  Each lane
        // instead walks its run's four words starting at word (lane / 8) % 4:
        // then every store instruction of the warp falls on 32 different
        // banks (lanes 8 apart take different words, lanes closer than 8 lie
        // in different 16-byte chunks).  Measured at 256x299x299, waiting
        // launches: two channels 38.9 -> 37.2 us, three channels 55.2 ->
        // 55.5 us (no gain); four-channel binary32 runs lost 3 % and keep
        // the plain order.  tr_tune_tiled flags bit 20 keeps the plain order.
        constexpr bool kRotate16 = (P * OB == 16) && OUT_F16;
        if (kRotate16 && !(p.hints & 1048576)) {
            const uint32_t q = (threadIdx.x >> 3) & 3u;
#pragma unroll
            for (int c = 0; c < C; ++c) {
                uint8_t* o = sout + (size_t)c * p.plane_bytes + odd_shift<C, OUT_F16, LAYOUT, MODE>(p, rec, c) +
                             ((size_t)r * p.W + (size_t)gx * P) * OB;
                uint32_t w[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    if constexpr (OUT_F16 != 0) w[m] = pack_half2(v[(2 * m) * C + c], v[(2 * m + 1) * C + c]);
                    else w[m] = __float_as_uint(v[m * C + c]);
                }
                // rotate: w[m] <- word (m + q) % 4 (two select stages, registers only)
                uint32_t t[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) t[m] = (q & 1u) ? w[(m + 1) & 3] : w[m];
#pragma unroll
                for (int m = 0; m < 4; ++m) w[m] = (q & 2u) ? t[(m + 2) & 3] : t[m];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t wi = (m + q) & 3u;   // the word of the run w[m] holds
                    uint8_t* at = o + 4u * wi;
                    if constexpr (OUT_F16 != 0) {
                        if ((int)(2 * wi) < kv) *reinterpret_cast<uint16_t*>(at) = (uint16_t)(w[m] & 0xFFFFu);
                        if ((int)(2 * wi + 1) < kv) *reinterpret_cast<uint16_t*>(at + 2) = (uint16_t)(w[m] >> 16);
                    } else {
                        if ((int)wi < kv) *reinterpret_cast<uint32_t*>(at) = w[m];
                    }
                }
            }
            return;
        }
#pragma unroll
        for (int c = 0; c < C; ++c) {
            uint8_t* o = sout + (size_t)c * p.plane_bytes + odd_shift<C, OUT_F16, LAYOUT, MODE>(p, rec, c) +
                         ((size_t)r * p.W + (size_t)gx * P) * OB;
#pragma unroll
            for (int i = 0; i < P; ++i)
                if (i < kv) put(o + (size_t)i * OB, v[i * C + c]);
        }
    } else {
        // a pixel's outputs as one 4-, 8- or 16-byte store where they are
        // that long and aligned, else element by element (runs of 4-byte
        // stores for 6-byte binary16 pixels measured slower)
        constexpr int PB = OC * OB;
        uint8_t* o = sout + odd_shift<C, OUT_F16, LAYOUT, MODE>(p, rec, 0) + ((size_t)r * p.W + (size_t)gx * P) * PB;
#pragma unroll
        for (int i = 0; i < P; ++i) {
            if (i < kv) {
                uint8_t* q = o + (size_t)i * PB;
                uint32_t w[(PB + 3) / 4];
                if (OUT_F16) {
#pragma unroll
                    for (int c = 0; c < OC; c += 2)
                        w[c / 2] = pack_half2(c < C ? v[i * C + c] : 0.0f, c + 1 < C ? v[i * C + c + 1] : 0.0f);
                } else {
#pragma unroll
                    for (int c = 0; c < OC; ++c) w[c] = __float_as_uint(c < C ? v[i * C + c] : 0.0f);
                }
                constexpr int NW = (PB + 3) / 4;
                if (PB == 16 && ((uintptr_t)q & 15u) == 0) {
                    *reinterpret_cast<uint4*>(q) = make_uint4(w[0], w[1 % NW], w[2 % NW], w[3 % NW]);
                } else if (PB == 8 && ((uintptr_t)q & 7u) == 0) {
                    *reinterpret_cast<uint2*>(q) = make_uint2(w[0], w[1 % NW]);
                } else if (PB == 4 && ((uintptr_t)q & 3u) == 0) {
                    *reinterpret_cast<uint32_t*>(q) = w[0];
                } else {
#pragma unroll
                    for (int c = 0; c < OC; ++c) put(q + (size_t)c * OB, c < C ? v[i * C + c] : 0.0f);
                }
            }
        }
    }
}

// The odd-row form's NHWC output with 1 or 3 channels (hints bit 24).  A
// band's output is one run of rows*W*C elements, element e at tile offset
// sh + e*OB, where sh (below 16) follows the band's global alignment, and the
// unflipped source byte of element e is the band's byte e.  Pixel-aligned
// groups (8 pixels, 24 elements, or 16 grayscale pixels) therefore start at
// arbitrary bytes of the tile, and their outputs had to be moved into its
// 16-byte frame in registers (19 % of the kernel's time at 256x299x299x3 ->
// f16).  Here group g takes the elements [g*GE - psi, g*GE - psi + GE), psi
// in [0, GE) chosen per band so that every group starts both on a pixel
// (psi = 0 mod C) and on a 16-byte boundary of the tile (psi = (sh/OB) mod
// (16/OB)); GE is a multiple of both.  A group's outputs leave as aligned
// 16-byte stores, its conversion is the pixel groups' own (convert_group),
// and only the source side changes: unflipped, the group's GE source bytes
// are contiguous even across rows; flipped within one row, they are the
// mirrored run of its P pixels; flipped across two rows, the two rows'
// mirrored runs, the first row's pixels in the run's upper bytes.  Elements
// before the band start fall before sh and elements past its end into the
// tile's slack: neither is stored to global memory.

// NWD words of the bytes starting at q (any alignment): aligned 4-byte loads
// and funnel shifts.
template <int NWD>
__device__ __forceinline__ void load_bytes_at(const uint8_t* q, uint32_t (&w)[NWD]) {
    const uint32_t* wp = reinterpret_cast<const uint32_t*>((uintptr_t)q & ~(uintptr_t)3);
    const uint32_t sh = (uint32_t)((uintptr_t)q & 3u) * 8u;
    uint32_t raw[NWD + 1];
#pragma unroll
    for (int i = 0; i <= NWD; ++i) raw[i] = wp[i];
#pragma unroll
    for (int i = 0; i < NWD; ++i) w[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

// Checked-build guard of a shared-memory read of `bytes` at q.
__device__ __forceinline__ bool smem_read_ok(const TiledParams& p, const uint8_t* q, int bytes, int site) {
    (void)p; (void)q; (void)bytes; (void)site;
    return TRFN_CHECK(q >= trfn_dyn_smem && q + bytes <= trfn_dyn_smem + p.smem_bytes, site);
}

template <int C, int OUT_F16>
__device__ __forceinline__ void odd_nhwc_group(const TiledParams& p, const uint8_t* sin, uint8_t* tile0,
                                               const uint8_t* tile_end, const UnitRec& rec, int g, int psi,
                                               int E, int off_in, bool band_erased) {
    constexpr int OB = OUT_F16 ? 2 : 4;
    constexpr int P = Group<C>::P;
    constexpr int GE = P * C;                    // elements (source bytes) of a group
    constexpr int NW = GE / 4;
    constexpr int NCH = GE * OB / 16;            // 16-byte output chunks
    constexpr int EPC = 16 / OB;                 // elements per chunk
    const int WC = p.W * C;
    const int e0 = g * GE - psi;
    const bool flip = (rec.flags & 1) != 0;
    // the row of the group's last element (or the band's last row when the
    // group runs past the band: those elements are not stored) and the
    // group's pixels in the row before it; needed only where the band is
    // flipped or meets the erased rows (both uniform over the band)
    int r1 = 0, split_px = 0;
    if (flip || band_erased) {
        r1 = min((int)(((uint64_t)(uint32_t)(e0 + GE - 1) * p.wc_inv) >> 32), rec.rows - 1);
        const int split = r1 * WC - e0;          // elements k < split lie in row r1 - 1
        split_px = split > 0 ? split / C : 0;
    }
    uint32_t w[NW];
    if (!flip) {
        const uint8_t* q = sin + off_in + e0;
        if (smem_read_ok(p, q, 4 * (NW + 1), 15)) load_bytes_at<NW>(q, w);
        else for (int i = 0; i < NW; ++i) w[i] = 0u;
    } else {
        // row r1's mirrored run: the group's pixels x = e/C - r1*W (the first
        // ones negative when the group starts in row r1 - 1) take the row's
        // pixels W-1-x, i.e. the P pixels from W - x0 - P on, reversed
        const int x0b = (e0 - r1 * WC) / C;   // exact: e0 - r1*WC is a multiple of C
        const uint8_t* qb = sin + off_in + r1 * WC + C * (p.W - x0b - P);
        if (smem_read_ok(p, qb, 4 * (NW + 1), 16)) load_bytes_at<NW>(qb, w);
        else for (int i = 0; i < NW; ++i) w[i] = 0u;
        if (split_px > 0 && r1 > 0) {
            // the pixels k < split_px lie in row r1 - 1 (x = x0b + W + k):
            // its mirrored run fills the run's bytes from C*(P - split_px) on
            uint32_t wa[NW];
            const uint8_t* qa = qb - WC - C * p.W;   // row r1 - 1, first pixel x0b + W
            if (smem_read_ok(p, qa, 4 * (NW + 1), 17)) load_bytes_at<NW>(qa, wa);
            else for (int i = 0; i < NW; ++i) wa[i] = 0u;
            const int thr = C * (P - split_px);   // bytes [thr, GE) from row r1 - 1
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                const int m = thr - 4 * i;      // bytes of word i from row r1
                if (m <= 0) w[i] = wa[i];
                else if (m < 4) w[i] = __byte_perm(w[i], wa[i], m == 1 ? 0x7650u : m == 2 ? 0x7610u : 0x7210u);
            }
        }
    }
    float v[GE];
    if (flip) convert_group<C, true>(w, p.base, p.scale, p.bias, v);
    else convert_group<C, false>(w, p.base, p.scale, p.bias, v);
    // erased pixels: those of row r1 - 1 ([0, split_px)) and of row r1
    if (band_erased) {
        const int ya = rec.y_begin + r1 - 1, yb = ya + 1;
        const int xa = (e0 - (r1 - 1) * WC) / C;   // pixel x of group pixel 0 in row r1 - 1 (if any)
        const int xb = (e0 - r1 * WC) / C;         // ... in row r1 (negative when it starts before)
        int lo_a = 0, hi_a = 0, lo_b = 0, hi_b = 0;
        if (split_px > 0 && ya >= rec.erow_lo && ya < rec.erow_hi) {
            lo_a = max(rec.ecol_lo - xa, 0);
            hi_a = min(rec.ecol_hi - xa, split_px);
        }
        if (yb >= rec.erow_lo && yb < rec.erow_hi) {
            lo_b = max(rec.ecol_lo - xb, split_px);
            hi_b = min(rec.ecol_hi - xb, P);
        }
        if (lo_a < hi_a || lo_b < hi_b) {
#pragma unroll
            for (int k = 0; k < GE; ++k) {
                const int i = k / C;
                if ((i >= lo_a && i < hi_a) || (i >= lo_b && i < hi_b)) v[k] = 0.0f;
            }
        }
    }
    uint8_t* o = tile0 + (size_t)g * GE * OB;
#pragma unroll
    for (int qc = 0; qc < NCH; ++qc) {
        if (e0 + qc * EPC >= E) break;   // past the band (the tile's slack holds a chunk's overhang)
        if (e0 + (qc + 1) * EPC <= 0) continue;   // wholly before the band (outside the tile)
        uint4 ch;
        if (OUT_F16) {
            ch.x = pack_half2(v[8 * qc + 0], v[8 * qc + 1]);
            ch.y = pack_half2(v[8 * qc + 2], v[8 * qc + 3]);
            ch.z = pack_half2(v[8 * qc + 4], v[8 * qc + 5]);
            ch.w = pack_half2(v[8 * qc + 6], v[8 * qc + 7]);
        } else {
            ch = make_uint4(__float_as_uint(v[4 * qc + 0]), __float_as_uint(v[4 * qc + 1]),
                            __float_as_uint(v[4 * qc + 2]), __float_as_uint(v[4 * qc + 3]));
        }
        if (TRFN_CHECK(o + 16 * (qc + 1) <= tile_end && ((uintptr_t)(o + 16 * qc) & 15u) == 0, 18))
            reinterpret_cast<uint4*>(o)[qc] = ch;
    }
}

template <int C, int OUT_F16>
__device__ __forceinline__ void odd_nhwc_band(const TiledParams& p, const uint8_t* sin, uint8_t* sout,
                                              const UnitRec& rec, int tid, int nthr, uint32_t sh) {
    constexpr int OB = OUT_F16 ? 2 : 4;
    constexpr int GE = Group<C>::P * C;
    constexpr int EPC = 16 / OB;
    const int phi = (int)((sh / OB) % EPC);
    int psi = phi;   // psi = phi mod EPC and psi = 0 mod C, in [0, GE)
    while (psi % C != 0) psi += EPC;
    const int E = rec.rows * p.W * C;
    const int off_in = rec.flags >> 8;
    uint8_t* tile0 = sout + (sh - (uint32_t)phi * OB) - (psi - phi) * OB;
    const uint8_t* tile_end = sout + p.out_stage;
    const int ng = (E + psi + GE - 1) / GE;
    // whether any of the band's rows is erased (then per group below)
    const bool band_erased = rec.erow_lo < rec.erow_hi && rec.erow_lo < rec.y_begin + rec.rows &&
                             rec.erow_hi > rec.y_begin;
    for (int g = tid; g < ng; g += nthr)
        odd_nhwc_group<C, OUT_F16>(p, sin, tile0, tile_end, rec, g, psi, E, off_in, band_erased);
}

// NCHW output of the odd-row form (2 or 3 channels), windows laid on the
// plane tiles' 16-byte frames.  A 16-byte chunk holds EPC = 16 / OB
// elements (8 binary16, 4 binary32).  Plane c's tile holds the band's
// rows*W elements from byte sh_c on, so its chunks start at the band's
// pixels EPC*k - phi_c (phi_c = sh_c / OB).  An image's planes lie H*W
// elements apart: phi_c = phi_0 + c*D (mod EPC) with D = (H*W) mod EPC.
// For D = 0 or 1 (every odd square size: 227, 299, ...) the
// WP = EPC + (C-1)*D consecutive pixels from EPC*g - phi_0 - (C-1)*D on
// hold, for every plane c, the plane's chunk that starts at window pixel
// (C-1-c)*D (the band's pixel EPC*g - phi_0 - c*D).  Lane g converts each
// channel of its window once (the window's source bytes are contiguous like
// a tile-aligned NHWC group's, with the same flip and erase handling) and
// writes C aligned 16-byte chunks: no element stores and no realignment of
// the output.
template <int C, int OUT_F16, int D>
struct NchwWindow {
    static constexpr int EPC = OUT_F16 ? 8 : 4;      // elements per 16-byte chunk
    static constexpr int WP = EPC + (C - 1) * D;    // window pixels
    static constexpr int GEW = WP * C;              // its source bytes
    static constexpr int NWW = (GEW + 3) / 4;       // its words
};

// Plane c's chunk of window g: its EPC pixels are window pixels (C-1-c)*D
// on (FLIP: their bytes in the mirrored run), erased ones written as +0.
template <int C, int OUT_F16, int D, bool FLIP>
__device__ __forceinline__ void odd_nchw_chunks(const TiledParams& p, const uint32_t (&w)[NchwWindow<C, OUT_F16, D>::NWW],
                                                const uint8_t* sout, uint8_t* const (&tile)[C], int g, int pw,
                                                int E, int lo_a, int hi_a, int lo_b, int hi_b) {
    constexpr int EPC = NchwWindow<C, OUT_F16, D>::EPC;
    constexpr int WP = NchwWindow<C, OUT_F16, D>::WP;
    // every plane's chunk lies in the band unless the window meets an end
    const bool inner = pw >= 0 && pw + WP <= E;
#pragma unroll
    for (int c = 0; c < C; ++c) {
        const int sc = pw + (C - 1 - c) * D;     // the first pixel of plane c's chunk
        if (!inner && (sc + EPC <= 0 || sc >= E)) continue;   // wholly outside the band
        float v[EPC];
#pragma unroll
        for (int i = 0; i < EPC; ++i) {
            const int j = (C - 1 - c) * D + i;   // window pixel
            const int sb = FLIP ? C * (WP - 1 - j) + c : C * j + c;
            v[i] = __fmaf_rn(byte_minus_shift(w[sb >> 2], sb & 3, p.base[c]), p.scale[c], p.bias[c]);
        }
        if (lo_a < hi_a || lo_b < hi_b) {
#pragma unroll
            for (int i = 0; i < EPC; ++i) {
                const int j = (C - 1 - c) * D + i;
                if ((j >= lo_a && j < hi_a) || (j >= lo_b && j < hi_b)) v[i] = 0.0f;
            }
        }
        uint4 ch;
        if constexpr (OUT_F16 != 0) {
            ch = make_uint4(pack_half2(v[0], v[1]), pack_half2(v[2], v[3]), pack_half2(v[4 % EPC], v[5 % EPC]),
                            pack_half2(v[6 % EPC], v[7 % EPC]));
        } else {
            ch = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                            __float_as_uint(v[3]));
        }
        uint8_t* const q = tile[c] + 16 * g;
        (void)sout;
        // (checked build) inside plane c's tile, on its 16-byte frame
        if (TRFN_CHECK(q >= sout + (size_t)c * p.plane_bytes && q + 16 <= sout + (size_t)(c + 1) * p.plane_bytes &&
                           ((uintptr_t)q & 15u) == 0,
                       22))
            *reinterpret_cast<uint4*>(q) = ch;
    }
}

template <int C, int OUT_F16, int D>
__device__ __forceinline__ void odd_nchw_window(const TiledParams& p, const uint8_t* sin, const uint8_t* sout,
                                                uint8_t* const (&tile)[C], const UnitRec& rec, int g, int phi0,
                                                int E, int off_in, bool band_erased) {
    constexpr int EPC = NchwWindow<C, OUT_F16, D>::EPC;
    constexpr int WP = NchwWindow<C, OUT_F16, D>::WP;
    constexpr int GEW = NchwWindow<C, OUT_F16, D>::GEW;
    constexpr int NWW = NchwWindow<C, OUT_F16, D>::NWW;
    const int WC = p.W * C;
    const int pw = EPC * g - phi0 - (C - 1) * D;   // the window's first pixel (band-relative)
    const int e0 = pw * C;                         // its first source element
    const bool flip = (rec.flags & 1) != 0;
    // the row of the window's last element (clamped to the band's last row:
    // pixels past the band are not stored) and its pixels in the row before
    // (the last element's index e0 + GEW - 1 = C * (EPC*g - phi0 + EPC) - 1 > 0)
    int r1 = 0, split_px = 0;
    if (flip || band_erased) {
        r1 = min((int)(((uint64_t)(uint32_t)(e0 + GEW - 1) * p.wc_inv) >> 32), rec.rows - 1);
        const int split = r1 * WC - e0;
        split_px = split > 0 ? split / C : 0;
    }
    uint32_t w[NWW];
    if (!flip) {
        const uint8_t* q = sin + off_in + e0;
        if (smem_read_ok(p, q, 4 * (NWW + 1), 19)) load_bytes_at<NWW>(q, w);
        else for (int i = 0; i < NWW; ++i) w[i] = 0u;
    } else {
        // window pixel j (x = x0b + j in row r1) takes the row's pixel
        // W-1-x: the WP pixels from W - x0b - WP on, reversed, so that
        // pixel j's bytes sit at C*(WP-1-j)
        const int x0b = (e0 - r1 * WC) / C;
        const uint8_t* qb = sin + off_in + r1 * WC + C * (p.W - x0b - WP);
        if (smem_read_ok(p, qb, 4 * (NWW + 1), 20)) load_bytes_at<NWW>(qb, w);
        else for (int i = 0; i < NWW; ++i) w[i] = 0u;
        if (split_px > 0 && r1 > 0) {
            // pixels j < split_px lie in row r1 - 1: its mirrored run (same
            // byte positions) fills the bytes from C*(WP - split_px) on
            uint32_t wa[NWW];
            const uint8_t* qa = qb - WC - C * p.W;
            if (smem_read_ok(p, qa, 4 * (NWW + 1), 21)) load_bytes_at<NWW>(qa, wa);
            else for (int i = 0; i < NWW; ++i) wa[i] = 0u;
            const int thr = C * (WP - split_px);
#pragma unroll
            for (int i = 0; i < NWW; ++i) {
                const int m = thr - 4 * i;
                if (m <= 0) w[i] = wa[i];
                else if (m < 4) w[i] = __byte_perm(w[i], wa[i], m == 1 ? 0x7650u : m == 2 ? 0x7610u : 0x7210u);
            }
        }
    }
    // erased window pixels: [lo_a, hi_a) in row r1 - 1, [lo_b, hi_b) in row r1
    int lo_a = 0, hi_a = 0, lo_b = 0, hi_b = 0;
    if (band_erased) {
        const int ya = rec.y_begin + r1 - 1, yb = ya + 1;
        const int xa = (e0 - (r1 - 1) * WC) / C;
        const int xb = (e0 - r1 * WC) / C;
        if (split_px > 0 && ya >= rec.erow_lo && ya < rec.erow_hi) {
            lo_a = max(rec.ecol_lo - xa, 0);
            hi_a = min(rec.ecol_hi - xa, split_px);
        }
        if (yb >= rec.erow_lo && yb < rec.erow_hi) {
            lo_b = max(rec.ecol_lo - xb, split_px);
            hi_b = min(rec.ecol_hi - xb, WP);
        }
    }
    if (flip) odd_nchw_chunks<C, OUT_F16, D, true>(p, w, sout, tile, g, pw, E, lo_a, hi_a, lo_b, hi_b);
    else odd_nchw_chunks<C, OUT_F16, D, false>(p, w, sout, tile, g, pw, E, lo_a, hi_a, lo_b, hi_b);
}

template <int C, int OUT_F16, int D, int MODE>
__device__ __forceinline__ void odd_nchw_band(const TiledParams& p, const uint8_t* sin, uint8_t* sout,
                                              const UnitRec& rec, int tid, int nthr) {
    constexpr int OB = OUT_F16 ? 2 : 4;
    constexpr int EPC = NchwWindow<C, OUT_F16, D>::EPC;
    const int phi0 = (int)((odd_shift<C, OUT_F16, TR_LAYOUT_NCHW, MODE>(p, rec, 0) / OB) % EPC);
    // plane c's chunk of window g is its tile's chunk g - (phi0 + c*D) / EPC,
    // at tile[c] + 16 g
    uint8_t* tile[C];
#pragma unroll
    for (int c = 0; c < C; ++c) tile[c] = sout + (size_t)c * p.plane_bytes - 16 * ((phi0 + c * D) / EPC);
    const int E = rec.rows * p.W;
    const int off_in = rec.flags >> 8;
    const int ng = (E - 1 + phi0 + (C - 1) * D) / EPC + 1;
    const bool band_erased = rec.erow_lo < rec.erow_hi && rec.erow_lo < rec.y_begin + rec.rows &&
                             rec.erow_hi > rec.y_begin;
    for (int g = tid; g < ng; g += nthr)
        odd_nchw_window<C, OUT_F16, D>(p, sin, sout, tile, rec, g, phi0, E, off_in, band_erased);
}

template <int C, int OUT_F16, int LAYOUT, bool CROP, bool ODD, int MODE>
__device__ __forceinline__ void compute_unit(const TiledParams& p, const uint8_t* sin,
                                             uint8_t* sout, const UnitRec& rec, int tid, int nthr) {
    constexpr int P = Group<C>::P;
    constexpr int GB = Group<C>::kBytes;
    if constexpr (ODD && LAYOUT == TR_LAYOUT_NHWC && (C == 1 || C == 3)) {
        if (p.hints & 16777216) {
            // (the producer's end mark, rows = 0, carries no other valid
            // field: nothing of it is read)
            if (rec.rows > 0)
                odd_nhwc_band<C, OUT_F16>(p, sin, sout, rec, tid, nthr, odd_shift<C, OUT_F16, LAYOUT, MODE>(p, rec, 0));
            return;
        }
    }
    if constexpr (ODD && LAYOUT == TR_LAYOUT_NCHW && (C == 2 || C == 3)) {
        if (p.hints & 134217728) {
            if (rec.rows > 0) {
                if (p.hints & 268435456) odd_nchw_band<C, OUT_F16, 1, MODE>(p, sin, sout, rec, tid, nthr);
                else odd_nchw_band<C, OUT_F16, 0, MODE>(p, sin, sout, rec, tid, nthr);
            }
            return;
        }
    }
    const int L = p.W * C;
    const int groups = rec.rows * p.gpr;
    for (int g = tid; g < groups; g += nthr) {
        const int r = (int)(((uint64_t)(uint32_t)g * p.gpr_inv) >> 32);
        const int gx = g - r * p.gpr;
        const int y = rec.y_begin + r;
        const int kv = ODD ? min(P, p.W - gx * P) : P;   // valid pixels (the last group of an odd row is short)
        int lo = 0, hi = 0;  // erased pixels [lo, hi) of this group
        if (y >= rec.erow_lo && y < rec.erow_hi) {
            lo = min(max(rec.ecol_lo - gx * P, 0), P);
            hi = min(max(rec.ecol_hi - gx * P, 0), P);
        }
        float v[GB];
        if (lo == 0 && hi == P) {
#pragma unroll
            for (int k = 0; k < GB; ++k) v[k] = 0.0f;
        } else {
            const int sgx = (rec.flags & 1) ? (p.gpr - 1 - gx) : gx;
            const uint8_t* s = sin + (size_t)r * L + (size_t)sgx * GB;
            uint32_t w[Group<C>::kWords];
            if (CROP || ODD) {
                // the group starts at any byte: aligned words, then funnel
                // shifts.  For a short mirrored group of an odd row the
                // window starts before the row (those pixels are dropped).
                const uint32_t* wp;
                uint32_t sh;
                if (ODD) {
                    const int src_px = (rec.flags & 1) ? (p.W - gx * P - P) : gx * P;
                    const uint8_t* q = sin + ((int)(rec.flags >> 8) + r * L + src_px * C);
                    wp = reinterpret_cast<const uint32_t*>((uintptr_t)q & ~(uintptr_t)3);
                    sh = (uint32_t)((uintptr_t)q & 3u) * 8u;
                } else {
                    const uint32_t at = (uint32_t)r * p.in_pitch + (uint32_t)(rec.flags >> 8) + (uint32_t)sgx * GB;
                    wp = reinterpret_cast<const uint32_t*>(sin + (at & ~3u));
                    sh = (at & 3u) * 8u;
                }
                uint32_t raw[Group<C>::kWords + 1];
                // (checked build) the words read lie in the dynamic shared
                // memory (a short mirrored group may start before its stage)
                const bool rd_ok = TRFN_CHECK(reinterpret_cast<const uint8_t*>(wp) >= trfn_dyn_smem &&
                                                  reinterpret_cast<const uint8_t*>(wp + Group<C>::kWords + 1) <=
                                                      trfn_dyn_smem + p.smem_bytes,
                                              8);
#pragma unroll
                for (int q = 0; q <= Group<C>::kWords; ++q) raw[q] = rd_ok ? wp[q] : 0u;
#pragma unroll
                for (int q = 0; q < Group<C>::kWords; ++q) w[q] = __funnelshift_r(raw[q], raw[q + 1], sh);
            } else if (!TRFN_CHECK(s >= sin && (size_t)(s - sin) + GB <= p.in_stage &&
                                       ((uintptr_t)s & (GB == 16 ? 15u : 7u)) == 0,
                                   7)) {
#pragma unroll
                for (int q = 0; q < Group<C>::kWords; ++q) w[q] = 0u;
            } else if (GB == 16) {
                const uint4 t = *reinterpret_cast<const uint4*>(s);
                w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
            } else {
#pragma unroll
                for (int q = 0; q < GB / 8; ++q) {
                    const uint2 t = reinterpret_cast<const uint2*>(s)[q];
                    w[2 * q] = t.x;
                    w[2 * q + 1] = t.y;
                }
            }
            if (rec.flags & 1) convert_group<C, true>(w, p.base, p.scale, p.bias, v);
            else convert_group<C, false>(w, p.base, p.scale, p.bias, v);
            if (lo < hi) {
#pragma unroll
                for (int k = 0; k < GB; ++k) {
                    const int i = k / C;
                    if (i >= lo && i < hi) v[k] = 0.0f;
                }
            }
        }
        if (ODD) store_group_odd<C, OUT_F16, LAYOUT, MODE>(p, sout, rec, r, gx, kv, v);
        else store_group<C, OUT_F16, LAYOUT>(p, sout, r, gx, v);
    }
}

template <int C, int OUT_F16, int LAYOUT, bool ODD, int MODE>
__device__ __forceinline__ void store_unit(const TiledParams& p, const uint8_t* sout,
                                           const UnitRec& rec, int lane) {
    constexpr int OB = OUT_F16 ? 2 : 4;
    const uint32_t src = smem_u32(sout);
    // Output lines go to L2 evict-first by default (a streamed result); a
    // caller whose next kernel reads the output from L2 can ask for normal
    // or evict-last priority.
    const bool plain = (p.hints & 6) == 2;
    const uint64_t pol = (p.hints & 4) ? policy_evict_last() : policy_evict_first();
    auto put = [&](void* g, uint32_t from, uint32_t bytes) {
        if (plain) bulk_s2g(g, from, bytes);
        else bulk_s2g_hint(g, from, bytes, pol);
    };
    if (ODD) {
        // per plane (NCHW) or for the band: the 16-byte aligned middle by a
        // bulk store (lane 0), the unaligned first and last bytes element by
        // element, spread over the storer's warp (up to 14 elements a plane:
        // one thread storing them all kept the other consumers waiting at
        // the next band's barrier)
        constexpr int OC = (LAYOUT == TR_LAYOUT_NHWC4) ? 4 : C;
        constexpr int NP = (LAYOUT == TR_LAYOUT_NCHW) ? C : 1;
        const ImageRef im = image_ref<MODE>(p, rec.n);
#pragma unroll
        for (int c = 0; c < NP; ++c) {
            size_t e;
            uint32_t bytes;
            if (LAYOUT == TR_LAYOUT_NCHW) {
                e = (((size_t)im.n * C + c) * p.H + rec.y_begin) * p.W;
                bytes = (uint32_t)rec.rows * p.W * OB;
            } else {
                e = ((size_t)im.n * p.H + rec.y_begin) * p.W * OC;
                bytes = (uint32_t)rec.rows * p.W * OC * OB;
            }
            uint8_t* g = im.dst + e * OB;
            const uint32_t sh = (uint32_t)((uintptr_t)g & 15u);
            const uint8_t* t = sout + (size_t)c * p.plane_bytes + sh;
            const uint32_t head = min(bytes, (16u - sh) & 15u);
            const uint32_t mid = (bytes - head) & ~15u;
            // (checked build) the band's bytes lie in the batch's output and
            // in the tile (its plane for NCHW)
            if (!TRFN_CHECK((uint64_t)(g - im.dst) + bytes <= p.dst_batch_bytes &&
                                (size_t)c * p.plane_bytes + sh + bytes <=
                                    (LAYOUT == TR_LAYOUT_NCHW ? (size_t)(c + 1) * p.plane_bytes : p.out_stage),
                            13))
                continue;
            const uint32_t nh = head / OB, ne = nh + (bytes - head - mid) / OB;
            for (uint32_t k = (uint32_t)lane; k < ne; k += 32u) {
                const uint32_t i = k < nh ? k * OB : head + mid + (k - nh) * OB;
                if (OUT_F16) *reinterpret_cast<uint16_t*>(g + i) = *reinterpret_cast<const uint16_t*>(t + i);
                else *reinterpret_cast<uint32_t*>(g + i) = *reinterpret_cast<const uint32_t*>(t + i);
            }
            if (lane == 0 && mid > 0 &&
                TRFN_CHECK(((uintptr_t)(g + head) & 15u) == 0 &&
                               ((src + (uint32_t)(c * p.plane_bytes + sh + head)) & 15u) == 0,
                           14))
                put(g + head, src + (uint32_t)(c * p.plane_bytes + sh + head), mid);
        }
        if (lane == 0) bulk_commit();
        return;
    }
    const ImageRef im = image_ref<MODE>(p, rec.n);
    if (LAYOUT == TR_LAYOUT_NCHW) {
        const uint32_t bytes = (uint32_t)rec.rows * p.W * OB;
#pragma unroll
        for (int c = 0; c < C; ++c) {
            uint8_t* g = im.dst + ((((size_t)im.n * C + c) * p.H + rec.y_begin) * p.W) * OB;
            // (checked build) inside the batch's output and the tile's plane,
            // 16-byte aligned at both ends
            if (TRFN_CHECK((uint64_t)(g - im.dst) + bytes <= p.dst_batch_bytes && bytes <= p.plane_bytes &&
                               ((uintptr_t)g & 15u) == 0 && ((src + (uint32_t)c * p.plane_bytes) & 15u) == 0 &&
                               (bytes & 15u) == 0,
                           12))
                put(g, src + (uint32_t)c * p.plane_bytes, bytes);
        }
    } else {
        const int ch = (LAYOUT == TR_LAYOUT_NHWC4) ? 4 : C;
        const size_t row_bytes = (size_t)p.W * ch * OB;
        uint8_t* g = im.dst + ((size_t)im.n * p.H + rec.y_begin) * row_bytes;
        const uint32_t bytes = (uint32_t)(rec.rows * row_bytes);
        if (TRFN_CHECK((uint64_t)(g - im.dst) + bytes <= p.dst_batch_bytes && bytes <= p.out_stage &&
                           ((uintptr_t)g & 15u) == 0 && (src & 15u) == 0 && (bytes & 15u) == 0,
                       11))
            put(g, src, bytes);
    }
    bulk_commit();
}

// Scheduling workspace: kTicketGroups ticket counters, each on its own
// 128-byte line, then the count of finished CTAs.  With g = min(kTicketGroups,
// gridDim.x) groups, CTA b draws from counter b % g, which hands out the
// dynamic units whose index is congruent to b modulo g.
constexpr int kTicketGroups = 8;
constexpr int kTicketStride = 32;   // uint32 words between counters (128 bytes)
constexpr int kDoneWord = kTicketGroups * kTicketStride;

// The producer's last steps (lane 0), after it has issued `j` fills: the
// wait for the previous grid if it has not been taken, the release of the
// next one, the status or the workspace reset by the last CTA to finish, and
// the wait for the bands in flight (bounded).  Fill k's phase is the latest
// of its stage only if no later fill used the stage: after a normal end the
// end mark took stage j % S, so fill j - S is done and superseded.
__device__ __forceinline__ void producer_finish(const TiledParams& p, uint32_t full0, int j, int S, bool ok,
                                                bool waited) {
    if (!waited) grid_dependency_wait();
    grid_launch_dependents();
    if (!ok) {
        atomicOr(&g_device_status, kStatusTimeout);
    } else if (p.ws != nullptr) {
        __threadfence();
        if (atomicAdd(p.ws + kDoneWord, 1u) == gridDim.x - 1) {
            for (int g = 0; g < kTicketGroups; ++g) p.ws[g * kTicketStride] = 0;
            p.ws[kDoneWord] = 0;
            __threadfence();
        }
    }
    for (int k = max(0, ok ? j - S + 1 : j - S); k < j; ++k) {
        if (!mbar_wait_bounded(full0 + 8u * (k % S), (uint32_t)(k / S) & 1u)) {
            atomicOr(&g_device_status, kStatusTimeout);
            break;
        }
    }
}

// Records made on the GPU in the same call (tr_fused_norm_sampled with
// TR_LAUNCH_OVERLAP_PREVIOUS, compact source with 16-byte aligned rows): the
// sampler grid launched just before writes them all, but they are readable
// only once it has completed, which is after the kernel before it in the
// stream.  So a CTA's first S records are made in the kernel, with the
// sampler's steps (a lane per Philox draw, the decisions on every lane with
// the draws shuffled in: the same bits), and those bands convert while the
// kernel before drains; later units' records are read from the sampler's
// output after the wait.  Consumer warps 1..S make the first S records in
// parallel while the first copies are in flight (they have nothing to
// convert yet); named barrier 2 orders each publication after the producer
// has posted the stage's byte count.  Where a CTA has fewer consumer warps
// than stages, or tr_tune_tiled flags bit 22 asks for it, the producer warp
// makes them one after another instead.
__device__ __forceinline__ bool first_records_by_consumers(const TiledParams& p) {
    return p.stages <= (int)(blockDim.x >> 5) - 1 && !(p.hints & 4194304);
}

// Where the consumer warps number at least 2S, warps S+1..2S make the records
// of the CTA's units S..2S-1 at the same time, into the unit-record slots
// S..2S-1 that the stage ring leaves free, and arrive on the barrier slot of
// stage S (also outside the ring).  The CTA's first 2S units are then static,
// and once the producer's wait for the sampler (hence for the kernel before
// it) returns, its next S bands are requested without a read of the
// sampler's output on the way (tr_tune_tiled flags bit 25 keeps S).  The
// wait itself stays after the first S bands: taken later, it also releases
// the next kernel in the stream later, which measured slower.
// Returns the count of units whose records the kernel makes.
__device__ __forceinline__ int sampled_prefix(const TiledParams& p) {
    const int S = p.stages;
    const bool twice = first_records_by_consumers(p) && 2 * S <= (int)(blockDim.x >> 5) - 1 &&
                       2 * S <= kMaxStages && !(p.hints & 33554432);
    return twice ? 2 * S : S;
}

__device__ __forceinline__ tr_aug_param* later_record_slot(uint8_t* smem, int j) {
    return reinterpret_cast<tr_aug_param*>(smem + kRecOffset + (size_t)j * sizeof(UnitRec));
}

__device__ __forceinline__ void named_barrier_arrive(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Consumer warp w (0-based): the record of the CTA's w-th unit, published on
// stage w once the producer has posted the band's bytes.
__device__ __forceinline__ void consumer_first_record(const TiledParams& p, uint8_t* smem, int w) {
    const int lane = (int)(threadIdx.x & 31u);
    const int uu = (int)blockIdx.x + w * (int)gridDim.x;
    tr_aug_param r = {0, 0, 0, 0, 0};
    if (uu < p.num_units) r = sample_record_warp(p.spec, uu / p.bands, lane);
    named_barrier_sync(2, (uint32_t)(p.stages + 1) * 32u);
    if (uu < p.num_units && lane == 0) publish_unit(p, uu, w, smem, r);
}

// Consumer warp w, S <= w < 2S: the record of the CTA's w-th unit, left in
// slot w for the producer.
__device__ __forceinline__ void consumer_later_record(const TiledParams& p, uint8_t* smem, int w) {
    const int lane = (int)(threadIdx.x & 31u);
    const int uu = (int)blockIdx.x + w * (int)gridDim.x;
    tr_aug_param r = {0, 0, 0, 0, 0};
    if (uu < p.num_units) r = sample_record_warp(p.spec, uu / p.bands, lane);
    if (lane == 0) {
        *later_record_slot(smem, w) = r;
        mbar_arrive(smem_u32(smem) + 8u * (uint32_t)p.stages);
    }
}

// The producer warp's start in such a launch (all 32 lanes): lane 0
// requests the first S bands whole, then the records are made (by the
// consumers, or here).  Returns the number of bands requested.
template <int C>
__device__ __forceinline__ int first_bands_sampled(const TiledParams& p, uint8_t* smem) {
    const int lane = (int)threadIdx.x;
    const int S = p.stages;
    const int G = (int)gridDim.x;
    int j = 0;
    if (lane == 0) {
        for (; j < S; ++j) {
            const int uu = (int)blockIdx.x + j * G;
            if (uu >= p.num_units) break;
            issue_unit_uncut<C, kModeSampled>(p, uu, j, smem);
        }
    }
    j = __shfl_sync(0xffffffffu, j, 0);
    if (first_records_by_consumers(p)) {
        named_barrier_arrive(2, (uint32_t)(S + 1) * 32u);
    } else {
        for (int t = 0; t < j; ++t) {
            const int uu = (int)blockIdx.x + t * G;
            const tr_aug_param r = sample_record_warp(p.spec, uu / p.bands, lane);
            if (lane == 0) publish_unit(p, uu, t, smem, r);
        }
    }
    return j;
}

// Warp 0 is the producer: its lane 0 fills stage s = j % S with the CTA's
// j-th unit once the consumers have released the stage (empty[s]), counting
// the bytes on full[s], and ends with an empty fill (rows = 0).  Without a
// workspace the CTA's units are blockIdx.x + j*gridDim.x; with one, the first
// S are those and the rest come from ticket counters, so CTAs that run faster
// take more bands and all finish together.  The last CTA to finish returns
// the counters to zero.
// Warps 1.. are consumers: they wait for full[s], convert the band into the
// output tile i % 2, meet on named barrier 1, and one of them releases the
// stage and issues the TMA store of the tile.
// (An explicit minimum of one CTA per SM lets ptxas use up to 63 registers
// here, against 61 without it, and measured 0.9 % faster at 256x224x224x3.)
// The odd-row forms bound by their conversion are compiled for four CTAs per
// SM (64 registers, no spills): 16-byte NCHW plane runs, NCHW with 2 or 3
// channels (the plane-aligned windows; binary32 RGB 256x299x299 79.7 ->
// 65.9 us, 256x227x227 40.5 -> 35.8 us, at three CTAs with 80 registers
// before) and NHWC with 1 or 3 channels.
template <int C, int OUT_F16, int LAYOUT, bool CROP, bool ODD>
constexpr int tiled_min_blocks() {
    return ((ODD && LAYOUT == TR_LAYOUT_NCHW && (Group<C>::P * (OUT_F16 ? 2 : 4) == 16 || C == 2 || C == 3)) ||
            (ODD && LAYOUT == TR_LAYOUT_NHWC && (C == 1 || C == 3)))
               ? 4
               : 1;
}

template <int C, int OUT_F16, int LAYOUT, bool CROP, bool ODD, int MODE>
__global__ void __launch_bounds__(256, (tiled_min_blocks<C, OUT_F16, LAYOUT, CROP, ODD>()))
    tiled_kernel(const __grid_constant__ TiledParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = p.stages;
    const uint32_t full0 = smem_u32(smem);
    const uint32_t empty0 = full0 + kEmptyOffset;
    const UnitRec* recs = reinterpret_cast<const UnitRec*>(smem + kRecOffset);
    const uint8_t* sin = smem + kHeaderBytes;
    uint8_t* sout = smem + kHeaderBytes + (size_t)S * p.in_stage;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        if constexpr (MODE == kModeSampled) {
            if (sampled_prefix(p) > S) mbar_init(full0 + 8u * S, (uint32_t)(sampled_prefix(p) - S));
        }
        fence_mbar_init();
    }
    __syncthreads();
    // everything above overlaps the previous grid in the stream; global
    // memory is touched only below, after that grid has completed, unless
    // the caller has promised that this launch shares no buffer with it
    // (hints bit 8): then the copies start at once, the producer waits for
    // the previous grid once it has issued its first S bands, and each
    // CTA's storer waits for it again before it exits, so this grid still
    // completes after it and later work in the stream sees both.
    // A CTA releases the next grid in the stream only after the previous one
    // has completed, so that no more than two grids of the stream (this one
    // and the next, which its caller declared independent of this one) are
    // ever in flight: here when this launch waited above, else after the
    // producer's wait.  (hints bit 3 delays the release until the CTA's
    // copies are all issued.)
    const bool overlapped = (p.hints & 256) != 0;
    if (!overlapped) grid_dependency_wait();
    if (!overlapped && !(p.hints & 8) && threadIdx.x == 0) grid_launch_dependents();

    if (threadIdx.x < 32) {
        // The producer: lane 0 waits on barriers, issues copies, takes
        // tickets and loads the records; the other lanes leave (after the
        // first records of a sampled launch).
        int j = 0;
        if constexpr (MODE == kModeSampled) j = first_bands_sampled<C>(p, smem);
        if (threadIdx.x != 0) return;
        const int G = gridDim.x;
        const int ngroups = min(kTicketGroups, G);   // every group must have a CTA
        const int group = (int)blockIdx.x % ngroups;
        // the CTA's first SP units are static: S, or 2S in a sampled launch
        // whose consumers make that many records
        const int SP = (MODE == kModeSampled) ? sampled_prefix(p) : S;
        const int n_dyn = max(0, p.num_units - SP * G);   // units handed out by tickets
        // unit u's record and, for crop sources, its image's window origin:
        // requested together, ahead of the wait for the stage they go to
        int2 org = make_int2(0, 0);
        auto unit_record = [&](int u) {
            const tr_aug_param r = image_record<MODE>(p, u / p.bands);
            if (CROP && p.crop != nullptr) {
                org.x = p.crop[2 * (size_t)(u / p.bands)];
                org.y = p.crop[2 * (size_t)(u / p.bands) + 1];
            }
            return r;
        };
        // the CTA's jn-th unit: static for the first SP (or without a
        // workspace), else from this CTA's ticket counter
        auto next_unit = [&](int jn) {
            if (p.ws == nullptr || jn < SP) return (int)blockIdx.x + jn * G;
            const int k = group + (int)atomicAdd(p.ws + group * kTicketStride, 1u) * ngroups;
            return k < n_dyn ? SP * G + k : p.num_units;
        };
        int u = blockIdx.x;
        tr_aug_param a = {0, 0, 0, 0, 0};
        // records written by the previous grid (the device sampler) while
        // this launch overlaps it (hints bit 9, compact aligned sources): the
        // first S bands are requested whole before that grid has completed,
        // and their records are read and published after the wait
        const bool recdep = !CROP && !ODD && overlapped && (p.hints & 512);
        // the first unit's band is requested before its record has arrived
        // (its erased span is then read too); measured 0.9 % faster at
        // 256x224x224x3 than waiting for the record
        const bool early0 = !CROP && !ODD && !recdep && !(p.hints & 32) && u < p.num_units;
        if (!early0 && !recdep && u < p.num_units) a = unit_record(u);
        bool ok = true;
        bool waited = !overlapped;   // the previous grid has completed
        if (MODE == kModeSampled) {
            // the first S bands and their records are under way; units S..SP-1
            // take the records the consumers make, the rest the sampler's,
            // readable after the wait
            u = next_unit(j);
            const bool made = j < SP && u < p.num_units;
            if (made) {
                if (mbar_wait_bounded(full0 + 8u * S, 0u)) {
                    a = *later_record_slot(smem, j);
                } else {
                    atomicOr(&g_device_status, kStatusTimeout);
                    u = p.num_units;
                }
            }
            grid_dependency_wait();
            waited = true;
            if (!(p.hints & 8)) grid_launch_dependents();
            if (!made && u < p.num_units) a = unit_record(u);
        } else if (recdep) {
            // the first S units are blockIdx.x + t * G (no array: it would
            // live in local memory)
            for (; j < S; ++j) {
                const int uu = (int)blockIdx.x + j * G;
                if (uu >= p.num_units) break;
                issue_unit_uncut<C, MODE>(p, uu, j, smem);
            }
            grid_dependency_wait();
            waited = true;
            if (!(p.hints & 8)) grid_launch_dependents();
            for (int t = 0; t < j; ++t) {
                const int uu = (int)blockIdx.x + t * G;
                publish_unit(p, uu, t, smem, unit_record(uu));
            }
            u = next_unit(j);
            if (u < p.num_units) a = unit_record(u);
        }
        for (;; ++j) {
            const int s = j % S;
            if (j >= S && !mbar_wait_bounded(empty0 + 8u * s, (uint32_t)(j / S - 1) & 1u)) {
                ok = false;
                break;
            }
            if (u >= p.num_units) {
                UnitRec* rec = reinterpret_cast<UnitRec*>(smem + kRecOffset) + s;
                rec->rows = 0;
                mbar_arrive(full0 + 8u * s);
                break;
            }
            if (j == 0 && early0) {
                issue_unit_uncut<C, MODE>(p, u, s, smem);
                a = unit_record(u);
                publish_unit(p, u, s, smem, a);
            } else {
                // a CTA's first S bands are copied whole (measured faster:
                // they are the ramp every launch starts with)
                issue_unit<C, CROP, ODD, MODE>(p, u, s, smem, a, (p.hints & 2048) || j >= S, org);
            }
            // the next unit and its record: requested now, used after the
            // next empty wait
            u = next_unit(j + 1);
            if constexpr (MODE == kModeSampled) {
                // a record the consumers made (their barrier was passed
                // above), else the sampler's (the wait was taken above)
                if (j + 1 < SP) a = *later_record_slot(smem, j + 1);
                else if (u < p.num_units) a = unit_record(u);
            } else {
                if (u < p.num_units) a = unit_record(u);
                if (!waited && j + 1 >= S) {
                    // overlapped launch: its first S bands are in flight
                    grid_dependency_wait();
                    waited = true;
                    if (!(p.hints & 8)) grid_launch_dependents();
                }
            }
        }
        producer_finish(p, full0, j, S, ok, waited);
        return;
    }

    if constexpr (MODE == kModeSampled) {
        const int w = (int)(threadIdx.x >> 5) - 1;
        if (first_records_by_consumers(p)) {
            if (w < S) consumer_first_record(p, smem, w);
            else if (w < sampled_prefix(p)) consumer_later_record(p, smem, w);
        }
    }
    const int tid = threadIdx.x - 32;
    const int nthr = blockDim.x - 32;
    // The storer is the first thread of the last consumer warp: where a
    // band's groups leave the consumers' last stride partly empty, the
    // empty slots fall on the last warps (groups go to consumer threads in
    // order), so the store work goes to a warp with less conversion work.
    const int store_base = nthr - 32;
    const bool storer = (tid == store_base);
    // the odd-row form's stores take the storer's whole warp (element stores
    // at the bands' unaligned edges); its first lane issues the bulk stores
    const bool store_warp = ODD ? (tid >= store_base) : storer;
    bool aborted = false;
    for (int i = 0;; ++i) {
        const int s = i % S;
        const bool ok = mbar_wait_bounded(full0 + 8u * s, (uint32_t)(i / S) & 1u);
        const UnitRec rec = recs[s];
        uint8_t* ob = sout + (size_t)(i & 1) * p.out_stage;
        if (ok) compute_unit<C, OUT_F16, LAYOUT, CROP, ODD, MODE>(p, sin + (size_t)s * p.in_stage, ob, rec, tid, nthr);
        fence_proxy_async_smem();
        // The store issued last iteration reads the other output tile, which
        // the next iteration overwrites: it must be done reading first.
        if (storer) bulk_wait_read<0>();
        if (named_barrier_or((uint32_t)nthr, !ok)) { aborted = true; break; }
        if (rec.rows == 0) break;   // the producer's end mark
        if (store_warp) {
            if (storer) mbar_arrive(empty0 + 8u * s);
            store_unit<C, OUT_F16, LAYOUT, ODD, MODE>(p, ob, rec, tid - store_base);
        }
    }
    if (storer) {
        if (aborted) atomicOr(&g_device_status, kStatusTimeout);
        if (p.hints & 16) bulk_wait_read<0>();
        else bulk_wait_all<0>();
        if (p.hints & 256) grid_dependency_wait();
    }
}

// -------------------------------------------------------------- generic ---

// Unsigned division by a divisor fixed for the launch, by one high multiply
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994, Figure 4.1): for d >= 1 and l = ceil(log2 d),
// m = floor(2^32 (2^l - d) / d) + 1; then for any 32-bit x,
// t = mulhi(m, x) and x / d = (t + ((x - t) >> 1)) >> (l - 1) (x / 1 = x).
struct DivU32 {
    uint32_t d = 1, m = 0;
    int l = 0;
};

inline DivU32 make_div(uint32_t d) {
    DivU32 v;
    v.d = d;
    int l = 0;
    while (l < 32 && (1ull << l) < d) ++l;
    v.l = l;
    v.m = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
    return v;
}

__device__ __forceinline__ uint32_t div_u32(uint32_t x, const DivU32& v) {
    if (v.l == 0) return x;   // d == 1
    const uint32_t t = __umulhi(v.m, x);
    return (t + ((x - t) >> 1)) >> (v.l - 1);
}

struct GenericParams {
    const uint8_t* src;
    uint8_t* dst;
    const tr_aug_param* aug;
    const int32_t* crop;   // per-image window origin {top, left}, or null
    long long image_stride, row_stride;   // source strides in bytes
    int N, H, W;
    int src_H, src_W;      // source image size (H, W for compact sources)
    DivU32 div_w, div_h;   // x / W and x / H for 32-bit pixel indices
    float shift[4];        // integer-valued: x - shift_c is exact
    float scale[4];
    float bias[4];
    int overlap;           // the launch shares no buffer with the previous grid in the stream
};

// One thread per output pixel, consecutive threads on consecutive pixels of
// a row, so each channel's loads and stores cover contiguous spans; a
// pixel's outputs go out as one 4-, 8- or 16-byte store where they are that
// long and aligned.  Pixel indices below 2^31 use 32-bit arithmetic with the
// invariant-divisor division above.
template <int C, int OUT_F16, int LAYOUT>
__global__ void __launch_bounds__(256) generic_kernel(const __grid_constant__ GenericParams p) {
    constexpr int OC = (LAYOUT == TR_LAYOUT_NHWC4) ? 4 : C;
    constexpr int OB = OUT_F16 ? 2 : 4;
    // Global memory only after the previous grid in the stream has completed,
    // unless the caller declared this launch independent of it: then thread
    // 0 of each block waits for it while the others start, so the grid still
    // completes after it.  Either way a block releases the next grid only
    // once the previous one has completed (as the tiled kernel does).
    if (!p.overlap || threadIdx.x == 0) {
        grid_dependency_wait();
        if (threadIdx.x == 0) grid_launch_dependents();
    }
    const long long pixels = (long long)p.N * p.H * p.W;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < pixels; t += stride) {
        int n, y, x;
        if (pixels <= 0x7FFFFFFFll) {
            const uint32_t ti = (uint32_t)t;
            const uint32_t row = div_u32(ti, p.div_w);
            x = (int)(ti - row * (uint32_t)p.W);
            n = (int)div_u32(row, p.div_h);
            y = (int)(row - (uint32_t)n * (uint32_t)p.H);
        } else {
            const long long row = t / p.W;
            x = (int)(t - row * p.W);
            n = (int)(row / p.H);
            y = (int)(row - (long long)n * p.H);
        }
        int cy = 0, cx = 0;
        if (p.crop != nullptr) {
            cy = min(max(p.crop[2 * (size_t)n], 0), p.src_H - p.H);
            cx = min(max(p.crop[2 * (size_t)n + 1], 0), p.src_W - p.W);
        }
        const uint8_t* row = p.src + (size_t)n * p.image_stride + (size_t)(cy + y) * p.row_stride + (size_t)cx * C;
        // the pixel and its mirror in the same row are requested with the
        // record, so the record's latency does not come before the pixel's
        uint8_t here[C], mirror[C];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            here[c] = __ldg(row + (size_t)x * C + c);
            mirror[c] = p.aug != nullptr ? __ldg(row + (size_t)(p.W - 1 - x) * C + c) : here[c];
        }
        bool flip = false, erased = false;
        if (p.aug != nullptr) {
            const tr_aug_param a = p.aug[n];
            flip = (a.flip != 0);
            erased = a.h > 0 && a.w > 0 && y >= a.y0 && (long long)y < (long long)a.y0 + a.h && x >= a.x0 &&
                     (long long)x < (long long)a.x0 + a.w;
        }
        float v[OC];
#pragma unroll
        for (int c = 0; c < OC; ++c) v[c] = 0.0f;
        if (!erased) {
#pragma unroll
            for (int c = 0; c < C; ++c)
                v[c] = __fmaf_rn(__fsub_rn((float)(flip ? mirror[c] : here[c]), p.shift[c]), p.scale[c], p.bias[c]);
        }
        const size_t pix = ((size_t)n * p.H + y) * p.W + x;
        if (LAYOUT == TR_LAYOUT_NCHW) {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const size_t o = ((size_t)n * C + c) * p.H * p.W + (size_t)y * p.W + x;
                if (OUT_F16) reinterpret_cast<__half*>(p.dst)[o] = __float2half_rn(v[c]);
                else reinterpret_cast<float*>(p.dst)[o] = v[c];
            }
        } else {
            uint8_t* o = p.dst + pix * OC * OB;
            constexpr int PB = OC * OB;   // bytes of one pixel's outputs
            uint32_t w[(PB + 3) / 4];
            if (OUT_F16) {
#pragma unroll
                for (int c = 0; c < OC; c += 2) w[c / 2] = pack_half2(v[c], c + 1 < OC ? v[c + 1] : 0.0f);
            } else {
#pragma unroll
                for (int c = 0; c < OC; ++c) w[c] = __float_as_uint(v[c]);
            }
            if (PB == 16 && ((uintptr_t)o & 15u) == 0) {
                *reinterpret_cast<uint4*>(o) = make_uint4(w[0], w[1], w[2 % ((PB + 3) / 4)], w[3 % ((PB + 3) / 4)]);
            } else if (PB == 8 && ((uintptr_t)o & 7u) == 0) {
                *reinterpret_cast<uint2*>(o) = make_uint2(w[0], w[1 % ((PB + 3) / 4)]);
            } else if (PB == 4 && ((uintptr_t)o & 3u) == 0) {
                *reinterpret_cast<uint32_t*>(o) = w[0];
            } else {
#pragma unroll
                for (int c = 0; c < OC; ++c) {
                    if (OUT_F16) reinterpret_cast<__half*>(o)[c] = __float2half_rn(v[c]);
                    else reinterpret_cast<float*>(o)[c] = v[c];
                }
            }
        }
    }
}

// ------------------------------------------------------------ host side ---

struct DeviceInfo {
    int sm_count = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;      // shared memory of one SM
    int smem_reserved = 0;    // shared memory the system reserves per resident CTA
};

DeviceInfo device_info(int dev) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return DeviceInfo{};
    if (cache[dev].sm_count == 0) {
        cudaDeviceGetAttribute(&cache[dev].sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&cache[dev].smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&cache[dev].smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&cache[dev].smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    }
    return cache[dev];
}

using TiledFn = void (*)(TiledParams);
using GenericFn = void (*)(GenericParams);

template <int C, int F16, bool CROP, bool ODD, int MODE>
TiledFn pick_tiled_layout(int layout) {
    switch (layout) {
    case TR_LAYOUT_NHWC: return tiled_kernel<C, F16, TR_LAYOUT_NHWC, CROP, ODD, MODE>;
    case TR_LAYOUT_NCHW: return tiled_kernel<C, F16, TR_LAYOUT_NCHW, CROP, ODD, MODE>;
    default: return tiled_kernel<C, F16, TR_LAYOUT_NHWC4, CROP, ODD, MODE>;
    }
}

template <int C, bool CROP, bool ODD, int MODE>
TiledFn pick_tiled_dtype(int f16, int layout) {
    return f16 ? pick_tiled_layout<C, 1, CROP, ODD, MODE>(layout) : pick_tiled_layout<C, 0, CROP, ODD, MODE>(layout);
}

template <bool CROP, bool ODD, int MODE>
TiledFn pick_tiled_c(int C, int f16, int layout) {
    switch (C) {
    case 1: return pick_tiled_dtype<1, CROP, ODD, MODE>(f16, layout);
    case 2: return pick_tiled_dtype<2, CROP, ODD, MODE>(f16, layout);
    case 3: return pick_tiled_dtype<3, CROP, ODD, MODE>(f16, layout);
    default: return pick_tiled_dtype<4, CROP, ODD, MODE>(f16, layout);
    }
}

// odd: compact sources whose rows (or NCHW output rows, or the output
// pointer) are not 16-byte aligned.  Several batches: compact sources only;
// records made in the kernel: compact sources with aligned rows only.
TiledFn pick_tiled(int C, int f16, int layout, bool crop, bool odd, int mode) {
    if (crop) return pick_tiled_c<true, false, kModeBatch>(C, f16, layout);
    if (mode == kModeSampled) return pick_tiled_c<false, false, kModeSampled>(C, f16, layout);
    if (mode == kModeBatches)
        return odd ? pick_tiled_c<false, true, kModeBatches>(C, f16, layout)
                   : pick_tiled_c<false, false, kModeBatches>(C, f16, layout);
    return odd ? pick_tiled_c<false, true, kModeBatch>(C, f16, layout)
               : pick_tiled_c<false, false, kModeBatch>(C, f16, layout);
}

template <int C, int F16>
GenericFn pick_generic_layout(int layout) {
    switch (layout) {
    case TR_LAYOUT_NHWC: return generic_kernel<C, F16, TR_LAYOUT_NHWC>;
    case TR_LAYOUT_NCHW: return generic_kernel<C, F16, TR_LAYOUT_NCHW>;
    default: return generic_kernel<C, F16, TR_LAYOUT_NHWC4>;
    }
}

template <int C>
GenericFn pick_generic_dtype(int f16, int layout) {
    return f16 ? pick_generic_layout<C, 1>(layout) : pick_generic_layout<C, 0>(layout);
}

GenericFn pick_generic(int C, int f16, int layout) {
    switch (C) {
    case 1: return pick_generic_dtype<1>(f16, layout);
    case 2: return pick_generic_dtype<2>(f16, layout);
    case 3: return pick_generic_dtype<3>(f16, layout);
    default: return pick_generic_dtype<4>(f16, layout);
    }
}


int group_pixels(int C) { return C == 3 ? 8 : 16 / C; }

// Tiled launch geometry for one problem.
struct TiledPlan {
    bool ok = false;
    int R = 0, bands = 0, stages = 0, threads = 0;
    uint32_t in_stage = 0, out_stage = 0, plane_bytes = 0;
    size_t smem = 0;
};

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Geometry knobs (tr_tune_tiled); 0 keeps the default.
std::atomic<int> g_band_bytes{0}, g_stages{0}, g_ctas_per_sm{0}, g_flags{0};

// pitch: bytes of one staged source row (W*C, or the crop box's chunks*chunk);
// slack: extra bytes after a stage's rows (crop consumers read one word past).
TiledPlan plan_tiled_r(int H, int W, int C, int f16, int layout, int smem_limit, size_t pitch, size_t slack,
                       int R_force, bool odd = false, int S_force = 0);

TiledPlan plan_tiled(int H, int W, int C, int f16, int layout, int smem_limit, size_t pitch = 0,
                     size_t slack = 0) {
    return plan_tiled_r(H, W, C, f16, layout, smem_limit, pitch, slack, 0);
}

// CTAs of a plan that fit one SM's shared memory.
int smem_residency(const TiledPlan& pl, int smem_per_sm, int reserved) {
    return pl.ok ? (int)((size_t)smem_per_sm / (pl.smem + (size_t)reserved)) : 0;
}

// The largest lower band height (down to half, divisors of H first, same
// stage count) at which `want` CTAs fit an SM's shared memory; pl itself if
// it already fits them, or if no such height exists or the band height is set
// by tr_tune_tiled.
TiledPlan lower_to_residency(const TiledPlan& pl, int want, int H, int W, int C, int f16, int layout,
                             int smem_limit, int smem_per_sm, int reserved, size_t pitch, size_t slack, bool odd) {
    if (!pl.ok || smem_per_sm <= 0 || g_band_bytes.load(std::memory_order_relaxed) > 0) return pl;
    if (smem_residency(pl, smem_per_sm, reserved) >= want) return pl;
    for (int pass = 0; pass < 2; ++pass) {
        for (int r = pl.R - 1; r >= (pl.R + 1) / 2 && r >= 1; --r) {
            if (pass == 0 && H % r != 0) continue;
            const TiledPlan q = plan_tiled_r(H, W, C, f16, layout, smem_limit, pitch, slack, r, odd);
            if (q.ok && q.stages == pl.stages && smem_residency(q, smem_per_sm, reserved) >= want) return q;
        }
    }
    return pl;
}

// Compact sources: the band height of about 32 KB of output per band, lowered
// where that leaves fewer than three CTAs on an SM (wide rows: at 256x299x299
// binary16 13-row bands fit two).  Three resident CTAs keep three times
// `stages` bands in flight per SM and 21 converting warps.  Only for plans of
// at most three stages (bands above 8 KB of source): at 256x224x224 it takes
// 3-stage binary16 plans from 0.53 to 0.59 of the copy peak (grayscale), 0.84
// to 0.88 (four channels), 256x256x3 from 0.84 to 0.88, while the 4-stage
// binary32 plans it would touch ran 1-3 % slower with three CTAs of smaller
// bands than with two.  tr_tune_tiled flags bit 16 keeps the 32 KB height.
constexpr int kWantResidency = 3;
constexpr long long kStreamMinBandsPerCta = 5;

// Share of the consumer threads' group slots that hold a group: consumers
// walk a band's groups in strides of their thread count and all meet at the
// end of the band, so a last stride that is mostly empty idles most of them.
double stride_fill(const TiledPlan& pl, int gpr) {
    const long long groups = (long long)pl.R * gpr;
    const long long nc = pl.threads - 32;
    const long long strides = (groups + nc - 1) / nc;
    return strides > 0 ? (double)groups / (double)(strides * nc) : 0.0;
}

// The largest height from pl.R down to half (same stage count, at least
// `want` CTAs per SM) whose strides are at least 84 % full; pl if none is.
// Measured at 256x299x299 (38 groups a row for RGB, 19 for grayscale):
// binary16 RGB 12 rows (456 groups: 68 % full) 0.58 of the copy peak, 11 rows
// (93 %) 0.60; binary32 RGB 7 rows (59 %) 0.83, 5 rows (99 %) 0.93; grayscale
// 36 rows (76 %) 0.37, 23 rows (98 %) 0.43.  tr_tune_tiled flags bit 18
// keeps the height as it was.
constexpr double kMinStrideFill = 0.84;

TiledPlan balance_strides(const TiledPlan& pl, int want, int H, int W, int C, int f16, int layout, int smem_limit,
                          int smem_per_sm, int reserved, size_t pitch, size_t slack, bool odd) {
    if (!pl.ok || g_band_bytes.load(std::memory_order_relaxed) > 0) return pl;
    if (g_flags.load(std::memory_order_relaxed) & 262144) return pl;
    const int P = group_pixels(C);
    const int gpr = odd ? (W + P - 1) / P : W / P;
    if (stride_fill(pl, gpr) >= kMinStrideFill) return pl;
    for (int r = pl.R - 1; r >= (pl.R + 1) / 2 && r >= 1; --r) {
        const TiledPlan q = plan_tiled_r(H, W, C, f16, layout, smem_limit, pitch, slack, r, odd);
        if (q.ok && q.stages == pl.stages && smem_residency(q, smem_per_sm, reserved) >= want &&
            stride_fill(q, gpr) >= kMinStrideFill)
            return q;
    }
    return pl;
}

TiledPlan plan_tiled_compact(int H, int W, int C, int f16, int layout, int smem_limit, int smem_per_sm,
                             int reserved, bool odd, long long N, int sm_count, bool overlapped) {
    const size_t slack = odd ? 64 : 0;
    const TiledPlan pl = plan_tiled_r(H, W, C, f16, layout, smem_limit, 0, slack, 0, odd);
    if (g_flags.load(std::memory_order_relaxed) & 65536) return pl;
    // 4-stage plans (small bands) are lowered only where each CTA gets few
    // bands, so that latency, not bandwidth, bounds the launch (1024x50x50x3
    // to binary32: 0.48 -> 0.55 of the copy peak with the lower height), or
    // where the launch overlaps the previous one, whose drain then hides the
    // extra bands' cost (256x224x224 binary32, overlapping: grayscale 0.938 ->
    // 0.965, four channels 0.998 -> 1.003, RGB NHWC4 0.995 -> 0.997)
    const long long slots = (long long)std::max(1, smem_residency(pl, smem_per_sm, reserved)) * std::max(1, sm_count);
    const bool few_bands = pl.ok && N * pl.bands < kStreamMinBandsPerCta * slots;
    const TiledPlan fit = (pl.stages > 3 && !few_bands && !overlapped)
                              ? pl
                              : lower_to_residency(pl, kWantResidency, H, W, C, f16, layout, smem_limit, smem_per_sm,
                                                   reserved, 0, slack, odd);
    const int want = std::min(kWantResidency, smem_residency(fit, smem_per_sm, reserved));
    return balance_strides(fit, want, H, W, C, f16, layout, smem_limit, smem_per_sm, reserved, 0, slack, odd);
}

// The odd-row form is bound by its conversion (realigning loads, element or
// realigned stores), not by copies in flight: two stages, and the largest
// height from the 32 KB one down to half at which the most CTAs per SM (up to
// four, as the kernel's registers allow: reg_res) fit with strides at least
// 84 % full.  The launch takes this plan only where each CTA streams at least
// five bands and it raises the CTAs per SM.  Measured at 256x299x299 against
// the aligned form's planning (three stages, three CTAs): binary16 RGB NHWC
// 0.60 -> 0.67 of the copy peak (10-row bands, four CTAs), 256x227x227 0.56 ->
// 0.59, grayscale 0.39 -> 0.43, two channels 0.49 -> 0.53.  tr_tune_tiled
// flags bit 19 plans the odd-row form like the aligned one.
TiledPlan plan_tiled_odd(int H, int W, int C, int f16, int layout, int smem_limit, int smem_per_sm, int reserved,
                         int reg_res) {
    const int sknob = g_stages.load(std::memory_order_relaxed);
    const int S = sknob >= 2 ? sknob : 2;
    const TiledPlan base = plan_tiled_r(H, W, C, f16, layout, smem_limit, 0, 64, 0, true, S);
    if (!base.ok || smem_per_sm <= 0 || g_band_bytes.load(std::memory_order_relaxed) > 0) return base;
    const int gpr = (W + group_pixels(C) - 1) / group_pixels(C);
    for (int want = std::max(1, std::min(4, reg_res)); want >= 1; --want) {
        for (int r = base.R; r >= (base.R + 1) / 2 && r >= 1; --r) {
            const TiledPlan q = plan_tiled_r(H, W, C, f16, layout, smem_limit, 0, 64, r, true, S);
            if (q.ok && q.stages == base.stages && smem_residency(q, smem_per_sm, reserved) >= want &&
                stride_fill(q, gpr) >= kMinStrideFill)
                return q;
        }
    }
    return base;
}

// A crop box stages wider rows than the window (whole chunks), which can cost
// one resident CTA per SM against the compact geometry; then take the largest
// lower band height that restores it.
TiledPlan plan_tiled_crop(int H, int W, int C, int f16, int layout, int smem_limit, int smem_per_sm,
                          int reserved, size_t pitch, size_t slack, long long N, int sm_count, bool overlapped) {
    const TiledPlan pl = plan_tiled(H, W, C, f16, layout, smem_limit, pitch, slack);
    const int want = smem_residency(plan_tiled_compact(H, W, C, f16, layout, smem_limit, smem_per_sm, reserved, false,
                                                       N, sm_count, overlapped),
                                    smem_per_sm, reserved);
    return lower_to_residency(pl, want, H, W, C, f16, layout, smem_limit, smem_per_sm, reserved, pitch, slack, false);
}

// odd: rows that are not a multiple of 16 bytes (the last group of a row is
// short, and each output tile region gets 16 bytes to follow its band's
// global alignment).
TiledPlan plan_tiled_r(int H, int W, int C, int f16, int layout, int smem_limit, size_t pitch, size_t slack,
                       int R_force, bool odd, int S_force) {
    TiledPlan pl;
    const int ob = f16 ? 2 : 4;
    const int P = group_pixels(C);
    const size_t L = (size_t)W * C;
    const int gpr = odd ? (W + P - 1) / P : W / P;
    const int out_ch = (layout == TR_LAYOUT_NHWC4) ? 4 : C;
    const size_t out_row = (size_t)W * out_ch * ob;
    // About 32 KB of output per band (band_bytes overrides with source bytes);
    // prefer a band height that divides H.  Measured at 224x224x3: 16 rows for
    // binary16 NHWC and NHWC4 and 8 for binary32 beat the other heights tried
    // (7 to 16 rows).
    const int knob = g_band_bytes.load(std::memory_order_relaxed);
    int R = (int)std::max<size_t>(1, std::min<size_t>((size_t)H, knob > 0 ? (size_t)knob / L
                                                                          : 32768 / out_row));
    bool divides = false;
    for (int r = R; r >= (R + 1) / 2; --r) {
        if (H % r == 0) { R = r; divides = true; break; }
    }
    // otherwise the same number of bands with heights as even as a fixed
    // height allows (75 rows at a 72-row target: 38 + 37, not 72 + 3)
    if (!divides) R = (H + (H + R - 1) / R - 1) / ((H + R - 1) / R);
    if (R_force > 0) R = std::min(R_force, H);
    while (R > 1 && (size_t)R * gpr >= 65536) --R;
    if ((size_t)R * gpr >= 65536) return pl;
    const int sknob = g_stages.load(std::memory_order_relaxed);
    const int stages0 = std::min(S_force >= 2 ? S_force : sknob >= 2 ? sknob : ((size_t)R * L > 8192 ? 3 : 4),
                                 kMaxStages);
    int stages = stages0;
    if (pitch == 0) pitch = L;
    for (;;) {
        const size_t in_stage = round_up((size_t)R * pitch + slack, 128);
        const size_t plane = odd ? round_up((size_t)R * W * ob + 16, 16) : (size_t)R * W * ob;
        // odd rows: 16 bytes for the tile to follow the band's alignment,
        // and 16 more for the overhang of the last 16-byte chunk of the
        // aligned-output groups
        const size_t out_stage = !odd ? round_up((size_t)R * out_row, 128)
                                 : layout == TR_LAYOUT_NCHW ? round_up((size_t)C * plane, 128)
                                                            : round_up((size_t)R * out_row + 32, 128);
        const size_t smem = kHeaderBytes + stages * in_stage + 2 * out_stage;
        if (in_stage < (1u << 20) && smem <= (size_t)smem_limit && R <= 256) {
            pl.ok = true;
            pl.R = R;
            pl.bands = (H + R - 1) / R;
            pl.stages = stages;
            pl.in_stage = (uint32_t)in_stage;
            pl.out_stage = (uint32_t)out_stage;
            pl.plane_bytes = (uint32_t)plane;
            pl.smem = smem;
            const int groups = R * gpr;
            pl.threads = 32 + (int)std::min<size_t>(224, std::max<size_t>(64, round_up(groups, 32)));
            return pl;
        }
        if (stages > 2) { --stages; continue; }
        if (R > 1) { R = std::max(1, R / 2); stages = stages0; continue; }
        return pl;
    }
}

// Launch with programmatic stream serialization: the grid may be scheduled
// while the preceding kernel in the stream drains; the kernels call
// griddepcontrol.wait before their first global memory access, so stream
// order is kept.
cudaError_t launch_pdl(const void* fn, unsigned grid, int threads, size_t smem, void* stream,
                       void* params) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[1] = {params};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

bool check_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return true;
    set_last_error(what, (int)e);
    return false;
}

// The source of a crop launch as a 4-d tensor {chunk, chunk index, row,
// image} for TMA tensor copies; the box is {chunk, nch, R, 1}.  Reads outside
// the tensor (rows past an image, chunks past a row) arrive as zeros.  With
// 32-byte chunks every request covers whole L2 sectors; without L2 promotion
// DRAM is read in sectors, so a window row costs at most one partial sector
// at each end.
int encode_crop_map(CUtensorMap* map, const LaunchArgs& a, uint32_t chunk, uint32_t nch, uint32_t R,
                    bool promote) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (encode == nullptr) {
        set_last_error("cuTensorMapEncodeTiled unavailable", (int)cudaErrorNotSupported);
        return TR_ERR_CUDA;
    }
    const cuuint64_t dims[4] = {chunk, (cuuint64_t)a.src_W * a.C / chunk, (cuuint64_t)a.src_H, (cuuint64_t)a.N};
    const cuuint64_t strides[3] = {chunk, (cuuint64_t)a.src_row_stride, (cuuint64_t)a.src_image_stride};
    const cuuint32_t box[4] = {chunk, nch, R, 1};
    const cuuint32_t elem[4] = {1, 1, 1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(a.src), dims, strides,
                              box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              promote ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_NONE,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_last_error("cuTensorMapEncodeTiled", (int)cudaErrorInvalidValue);
        return TR_ERR_CUDA;
    }
    return TR_OK;
}

// CTAs of fn with this many threads and bytes of dynamic shared memory that
// fit one SM (cached per kernel, device and geometry), after the kernel's
// one-time opt-in to the device's largest dynamic shared memory.
int tiled_occupancy(TiledFn fn, int dev, int smem_optin, int threads, size_t smem, int* blocks) {
    struct Cached { const void* fn; int dev; size_t smem; int threads; int blocks; };
    static std::mutex mu;
    static Cached cache[256];
    static int ncache = 0;
    static const void* opted[64][64];
    static int nopted[64];
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return TR_ERR_CUDA;
    bool done = false;
    for (int k = 0; k < nopted[dev]; ++k) done = done || opted[dev][k] == (const void*)fn;
    if (!done) {
        if (!check_cuda(cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin),
                        "cudaFuncSetAttribute"))
            return TR_ERR_CUDA;
        if (nopted[dev] < 64) opted[dev][nopted[dev]++] = (const void*)fn;
    }
    for (int k = 0; k < ncache; ++k) {
        if (cache[k].fn == (const void*)fn && cache[k].dev == dev && cache[k].smem == smem &&
            cache[k].threads == threads) {
            *blocks = cache[k].blocks;
            return TR_OK;
        }
    }
    int b = 0;
    if (!check_cuda(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, (const void*)fn, threads, smem),
                    "cudaOccupancyMaxActiveBlocksPerMultiprocessor"))
        return TR_ERR_CUDA;
    if (ncache < 256 && b > 0) cache[ncache++] = Cached{(const void*)fn, dev, smem, threads, b};
    *blocks = b;
    return TR_OK;
}

// Everything a tiled launch decides before its parameters: the kernel form,
// the band plan, CTAs per SM and the grid (shared by the launch and by
// tr_fused_norm_geometry).
struct TiledSetup {
    TiledPlan pl;
    TiledFn fn = nullptr;
    bool crop = false, odd = false;
    int chunk_shift = 4;
    size_t chunk = 16, nch = 0;
    int blocks_per_sm = 0;
    long long grid = 0, waves = 0;
    int tflags = 0;
};

int setup_tiled(const LaunchArgs& a, TiledSetup* t) {
    int dev = 0;
    if (!check_cuda(cudaGetDevice(&dev), "cudaGetDevice")) return TR_ERR_CUDA;
    const DeviceInfo di = device_info(dev);
    if (di.sm_count <= 0) {
        set_last_error("cudaDeviceGetAttribute", (int)cudaGetLastError());
        return TR_ERR_CUDA;
    }
    const int f16 = (a.out_dtype == TR_OUT_F16);
    const bool crop = a.crop_src;
    const size_t L = (size_t)a.W * a.C;
    // crop sources: a box of R rows of `nch` chunks covers a window that
    // starts anywhere in its first chunk; 32-byte chunks when the source rows
    // allow (tr_tune_tiled flags bit 8 forces 16, bit 9 asks for L2 promotion)
    const int tflags = g_flags.load(std::memory_order_relaxed);
    const int chunk_shift = (crop && ((size_t)a.src_W * a.C) % 32 == 0 && !(tflags & 256)) ? 5 : 4;
    const size_t chunk = (size_t)1 << chunk_shift;
    const size_t nch = crop ? (L + 2 * (chunk - 1)) / chunk : 0;
    if (crop && nch > 256) return TR_ERR_NOT_SUPPORTED;
    // compact sources whose rows, NCHW output rows or output pointer are
    // not 16-byte aligned take the odd-row form of the kernel
    const bool odd = !crop && !tiled_aligned(a.src, a.dst, a.W, a.C, f16, a.out_layout);
    const int mode = a.sample_in_kernel ? kModeSampled : a.batch_images > 0 ? kModeBatches : kModeBatch;
    if (mode == kModeSampled && (crop || odd || !a.overlap_prev || !a.records_from_prev))
        return TR_ERR_NOT_SUPPORTED;
    const TiledFn fn = pick_tiled(a.C, f16, a.out_layout, crop, odd, mode);
    TiledPlan pl;
    if (crop) {
        pl = plan_tiled_crop(a.H, a.W, a.C, f16, a.out_layout, di.smem_optin, di.smem_per_sm, di.smem_reserved,
                             nch * chunk, 16, a.N, di.sm_count, a.overlap_prev);
    } else if (odd && !(tflags & 524288)) {
        // Launches in which each CTA streams many bands are bound by the
        // conversion: there the odd-row planning (two stages, more CTAs per
        // SM) is taken when it does raise the CTAs per SM.  With few bands a
        // CTA the copies' latency dominates and the aligned form's planning
        // does better (100x100 and 50x50 images), as it does where the odd-row
        // planning cannot add a CTA (binary32 RGB, 4-channel outputs).
        pl = plan_tiled_compact(a.H, a.W, a.C, f16, a.out_layout, di.smem_optin, di.smem_per_sm, di.smem_reserved,
                                true, a.N, di.sm_count, a.overlap_prev);
        int res = 0, reg_res = 0;
        int rc = pl.ok ? tiled_occupancy(fn, dev, di.smem_optin, pl.threads, pl.smem, &res) : TR_OK;
        if (rc == TR_OK) rc = tiled_occupancy(fn, dev, di.smem_optin, 256, 0, &reg_res);
        if (rc != TR_OK) return rc;
        const long long units = (long long)a.N * pl.bands;
        const long long slots = (long long)std::max(1, res) * di.sm_count;
        if (pl.ok && (units + slots - 1) / slots >= kStreamMinBandsPerCta) {
            const TiledPlan q = plan_tiled_odd(a.H, a.W, a.C, f16, a.out_layout, di.smem_optin, di.smem_per_sm,
                                               di.smem_reserved, reg_res);
            int qres = 0;
            if (q.ok) {
                rc = tiled_occupancy(fn, dev, di.smem_optin, q.threads, q.smem, &qres);
                if (rc != TR_OK) return rc;
            }
            if (qres > res) pl = q;
        }
    } else {
        pl = plan_tiled_compact(a.H, a.W, a.C, f16, a.out_layout, di.smem_optin, di.smem_per_sm, di.smem_reserved,
                                odd, a.N, di.sm_count, a.overlap_prev);
    }
    if (!pl.ok) return TR_ERR_NOT_SUPPORTED;

    int blocks_per_sm = 0;
    {
        const int rc = tiled_occupancy(fn, dev, di.smem_optin, pl.threads, pl.smem, &blocks_per_sm);
        if (rc != TR_OK) return rc;
        if (blocks_per_sm <= 0) return TR_ERR_NOT_SUPPORTED;
    }
    const int cap = g_ctas_per_sm.load(std::memory_order_relaxed);
    if (cap > 0) blocks_per_sm = std::min(blocks_per_sm, cap);
    const long long num_units = (long long)a.N * pl.bands;
    const long long max_ctas = (long long)blocks_per_sm * di.sm_count;
    long long grid = std::min<long long>(num_units, max_ctas);
    // equalise the number of units per CTA (the static schedule); the
    // dynamic one balances by itself and takes every slot (GB300,
    // overlapping launches: 256x299x299x3 -> f16 33.69 -> 33.35 us, NHWC4
    // 21.29 -> 21.04, 256x224x224 grayscale 6.99 -> 6.84, the headline and
    // binary32 unchanged)
    const long long waves = (num_units + grid - 1) / grid;
    if (a.workspace == nullptr) grid = (num_units + waves - 1) / waves;

    t->pl = pl;
    t->fn = fn;
    t->crop = crop;
    t->odd = odd;
    t->chunk_shift = chunk_shift;
    t->chunk = chunk;
    t->nch = nch;
    t->blocks_per_sm = blocks_per_sm;
    t->grid = grid;
    t->waves = waves;
    t->tflags = tflags;
    return TR_OK;
}

int launch_tiled(const LaunchArgs& a) {
    TiledSetup t;
    {
        const int rc = setup_tiled(a, &t);
        if (rc != TR_OK) return rc;
    }
    const TiledPlan& pl = t.pl;
    const bool crop = t.crop, odd = t.odd;
    const size_t chunk = t.chunk, nch = t.nch;
    const int tflags = t.tflags;
    const size_t L = (size_t)a.W * a.C;

    TiledParams p;
    p.crop = a.crop;
    p.src_H = crop ? a.src_H : a.H;
    p.src_W = crop ? a.src_W : a.W;
    p.in_pitch = (uint32_t)(crop ? nch * chunk : L);
    p.chunk_shift = t.chunk_shift;
    if (crop) {
        const int rc = encode_crop_map(&p.tmap, a, (uint32_t)chunk, (uint32_t)nch, (uint32_t)pl.R,
                                       (tflags & 512) != 0);
        if (rc != TR_OK) return rc;
    }
    p.src = a.src;
    p.dst = static_cast<uint8_t*>(a.dst);
    p.aug = a.aug;
    p.N = a.N; p.H = a.H; p.W = a.W;
    p.R = pl.R;
    p.bands = pl.bands;
    p.num_units = a.N * pl.bands;
    p.gpr = odd ? (a.W + group_pixels(a.C) - 1) / group_pixels(a.C) : a.W / group_pixels(a.C);
    // the source bytes of one batch rounded down to 16 (odd-row form)
    p.src_floor16 = ((uint64_t)(a.batch_images > 0 ? a.batch_images : a.N) * a.H * a.W * a.C) & ~15ull;
    p.nb = a.batch_images;
    {
        const uint64_t n1 = (uint64_t)(a.batch_images > 0 ? a.batch_images : a.N);
        const uint64_t oc = (a.out_layout == TR_LAYOUT_NHWC4) ? 4 : (uint64_t)a.C;
        p.smem_bytes = (uint32_t)pl.smem;
        p.src_batch_bytes = crop ? 0 : n1 * a.H * a.W * a.C;
        p.dst_batch_bytes = n1 * a.H * a.W * oc * (a.out_dtype == TR_OUT_F16 ? 2 : 4);
    }
    for (int k = 0; k < TR_MAX_BATCHES; ++k) {
        p.bsrc[k] = a.bsrc[k];
        p.bdst[k] = static_cast<uint8_t*>(a.bdst[k]);
        p.baug[k] = a.baug[k];
    }
    p.gpr_inv = ((1ull << 32) + (uint64_t)p.gpr - 1) / (uint64_t)p.gpr;
    p.wc_inv = ((1ull << 32) + (uint64_t)a.W * a.C - 1) / ((uint64_t)a.W * a.C);
    p.in_stage = pl.in_stage;
    p.out_stage = pl.out_stage;
    p.plane_bytes = pl.plane_bytes;
    p.stages = pl.stages;
    p.hints = g_flags.load(std::memory_order_relaxed) &
              (255 | 1024 | 2048 | 0xF000 | 1048576 | 4194304 | 33554432);
    // copies may start before the previous grid completes; records that grid
    // wrote are read after it (compact aligned sources; the crop and
    // odd-row forms then wait for it before they touch memory)
    if (a.overlap_prev && !(a.records_from_prev && (crop || odd))) p.hints |= 256;
    if (a.overlap_prev && a.records_from_prev && !crop && !odd) p.hints |= 512;
    // first records made in the kernel: the sampler's settings
    p.spec = a.sample_in_kernel ? *a.spec : SampleSpec();
    p.ws = static_cast<unsigned int*>(a.workspace);
    for (int c = 0; c < 4; ++c) {
        p.base[c] = 8388608.0f + a.shift[c];   // exact: |shift| <= 2^20
        p.scale[c] = a.scale[c];
        p.bias[c] = a.bias[c];
    }

    // The odd-row form's register realignment of group outputs lengthens a
    // band's conversion: it pays when a CTA streams many bands (6 to 13 for
    // 227- and 299-pixel rows: 0.51 to 0.56 and 0.53 to 0.58 of the copy peak
    // for binary16 RGB NHWC, 0.64 to 0.83 for binary32, 0.36 to 0.37 for
    // binary16 grayscale), not when each CTA converts one to four bands and
    // the conversion is on the critical path (28x28 to 100x100 images: 2-12 %
    // slower).  Those launches keep the element stores (tr_tune_tiled flags
    // bit 17 asks for the realignment regardless).
    if (odd && t.waves < kStreamMinBandsPerCta && !(tflags & 131072)) p.hints |= 1024;
    // odd-row NHWC output with 1 or 3 channels, where each CTA streams
    // enough bands for the register realignment above: groups aligned to the
    // output tile instead (each row at least one group long; element indices
    // small enough for the one-multiply row division).  GB300, waiting /
    // overlapping launches: 256x299x299x3 -> f16 43.5 / 39.8 -> 37.3 / 34.5
    // us, 256x227x227x3 28.5 / 24.6 -> 25.3 / 22.1, 256x299x299 grayscale
    // 22.9 / 17.8 -> 20.3 / 15.9, binary32 the same; batches of 28x28
    // images (element stores) were 6-8 % slower with it.  tr_tune_tiled
    // flags bit 23 keeps the pixel-aligned groups.
    {
        const uint64_t wc = (uint64_t)a.W * a.C;
        const uint64_t ge = (uint64_t)group_pixels(a.C) * a.C;
        if (odd && a.out_layout == TR_LAYOUT_NHWC && (a.C == 1 || a.C == 3) && !(p.hints & 1024) && wc >= ge &&
            ((uint64_t)pl.R * wc + ge) * wc < (1ull << 31) && !(tflags & 8388608))
            p.hints |= 16777216;
    }
    // odd-row NCHW output with 2 or 3 channels, where each CTA streams enough
    // bands: windows laid on the plane tiles' 16-byte frames (planes H*W
    // elements apart must keep their frames 0 or 1 element apart, which
    // every odd square size does; each row at least one window long;
    // element indices small enough for the one-multiply row division).
    // tr_tune_tiled flags bit 26 keeps the per-group plane runs.
    {
        const uint64_t wc = (uint64_t)a.W * a.C;
        const int epc = a.out_dtype == TR_OUT_F16 ? 8 : 4;
        const int d = (int)(((uint64_t)a.H * a.W) % (uint64_t)epc);
        const int wp = epc + (a.C - 1) * d;
        if (odd && a.out_layout == TR_LAYOUT_NCHW && (a.C == 2 || a.C == 3) && d <= 1 && !(p.hints & 1024) &&
            a.W >= wp && ((uint64_t)pl.R * wc + 64) * wc < (1ull << 31) && !(tflags & 67108864)) {
            p.hints |= 134217728;
            if (d == 1) p.hints |= 268435456;
        }
    }

    if (!check_cuda(launch_pdl((const void*)t.fn, (unsigned)t.grid, pl.threads, pl.smem, a.stream, &p),
                    "tiled kernel launch"))
        return TR_ERR_CUDA;
    count_launch();
    return TR_OK;
}

int launch_generic(const LaunchArgs& a) {
    int dev = 0;
    if (!check_cuda(cudaGetDevice(&dev), "cudaGetDevice")) return TR_ERR_CUDA;
    const DeviceInfo di = device_info(dev);
    if (di.sm_count <= 0) {
        set_last_error("cudaDeviceGetAttribute", (int)cudaGetLastError());
        return TR_ERR_CUDA;
    }
    const int f16 = (a.out_dtype == TR_OUT_F16);
    GenericParams p;
    p.src = a.src;
    p.dst = static_cast<uint8_t*>(a.dst);
    p.aug = a.aug;
    p.N = a.N; p.H = a.H; p.W = a.W;
    p.crop = a.crop_src ? a.crop : nullptr;
    p.src_H = a.crop_src ? a.src_H : a.H;
    p.src_W = a.crop_src ? a.src_W : a.W;
    p.row_stride = a.crop_src ? (long long)a.src_row_stride : (long long)a.W * a.C;
    p.image_stride = a.crop_src ? (long long)a.src_image_stride : (long long)a.H * a.W * a.C;
    for (int c = 0; c < 4; ++c) { p.shift[c] = a.shift[c]; p.scale[c] = a.scale[c]; p.bias[c] = a.bias[c]; }
    const int threads = 256;
    p.div_w = make_div((uint32_t)a.W);
    p.div_h = make_div((uint32_t)a.H);
    // records written by the previous grid (the device sampler) are read only
    // after it has completed
    p.overlap = (a.overlap_prev && !a.records_from_prev) ? 1 : 0;
    const long long pixels = (long long)a.N * a.H * a.W;
    // about 8 pixels per thread, between 8 and 32 blocks per SM (measured:
    // 32 blocks per SM 11 % faster for 256 x 227x227x3, 8 better for 1024
    // x 28x28x1)
    long long grid = pixels / ((long long)threads * 8);
    grid = std::max<long long>(grid, (long long)di.sm_count * 8);
    grid = std::min<long long>(grid, (long long)di.sm_count * 32);
    grid = std::min<long long>(grid, (pixels + threads - 1) / threads);
    if (grid < 1) grid = 1;
    if (!check_cuda(launch_pdl((const void*)pick_generic(a.C, f16, a.out_layout), (unsigned)grid, threads, 0,
                               a.stream, &p),
                    "generic kernel launch"))
        return TR_ERR_CUDA;
    count_launch();
    return TR_OK;
}

std::atomic<uint64_t> g_launches{0};

}  // namespace

// The aligned form's conditions: 16-byte aligned pointers, source rows (and
// NCHW output rows) a multiple of 16 bytes.
bool tiled_aligned(const uint8_t* src, const void* dst, int W, int C, int f16, int out_layout) {
    const int ob = f16 ? 2 : 4;
    if (((uintptr_t)src & 15u) != 0 || ((uintptr_t)dst & 15u) != 0) return false;
    if (((long long)W * C) % 16 != 0) return false;
    if (out_layout == TR_LAYOUT_NCHW && ((long long)W * ob) % 16 != 0) return false;
    return true;
}

// The tiled kernel takes compact sources with a 16-byte aligned base; rows
// of any length (the odd-row form realigns them).
bool tiled_supported(const uint8_t* src, const void* dst, int N, int H, int W, int C, int out_dtype,
                     int out_layout) {
    (void)dst;
    (void)out_dtype;
    (void)out_layout;
    if (C < 1 || C > 4) return false;
    if (((uintptr_t)src & 15u) != 0) return false;
    if ((long long)N * H > (1LL << 31) - 1) return false;   // unit indices are int
    if ((long long)W * C > (1 << 24)) return false;         // int byte offsets within a band
    return true;
}

bool tiled_crop_supported(const uint8_t* src, const void* dst, int N, int H, int W, int C, int out_dtype,
                          int out_layout, int src_H, int src_W, size_t row_stride, size_t image_stride) {
    if (!tiled_supported(src, dst, N, H, W, C, out_dtype, out_layout)) return false;
    if (!tiled_aligned(src, dst, W, C, out_dtype == TR_OUT_F16, out_layout)) return false;
    if (((size_t)src_W * C) % 16 != 0 || row_stride % 16 != 0 || image_stride % 16 != 0) return false;
    if (image_stride < (size_t)src_H * row_stride) return false;
    if (((size_t)W * C + 30) / 16 > 256) return false;
    if ((size_t)src_W * C / 16 > 0xFFFFFFFFull) return false;   // chunk count of a source row (uint32)
    return true;
}

int tiled_geometry(const LaunchArgs& a, TiledGeometry* g) {
    TiledSetup t;
    const int rc = setup_tiled(a, &t);
    if (rc != TR_OK) return rc;
    g->rows = t.pl.R;
    g->stages = t.pl.stages;
    g->threads = t.pl.threads;
    g->ctas_per_sm = t.blocks_per_sm;
    g->grid = (int)t.grid;
    g->odd_form = t.odd ? 1 : 0;
    return TR_OK;
}

int launch(const LaunchArgs& a, int variant) {
    if (a.spec != nullptr && !a.records_from_prev) {
        // Records made on the GPU: the sampler writes them first, and the
        // kernel reads them in stream order.  A tiled launch in its aligned
        // compact form that overlaps the kernel before it also makes its
        // CTAs' first records itself (the same bits), so that it need not
        // wait for the sampler, hence for that kernel, before converting
        // (tr_tune_tiled flags bit 21 turns this off).
        int rc = launch_sampler(*a.spec, a.N, a.records_out, a.stream, a.overlap_prev);
        if (rc != TR_OK) return rc;
        LaunchArgs b = a;
        b.aug = a.records_out;
        b.records_from_prev = true;
        const int f16 = (a.out_dtype == TR_OUT_F16);
        b.sample_in_kernel = variant == TR_VARIANT_TILED && a.overlap_prev && !a.crop_src && a.batch_images == 0 &&
                             tiled_aligned(a.src, a.dst, a.W, a.C, f16, a.out_layout) &&
                             !(g_flags.load(std::memory_order_relaxed) & 2097152);
        if (!b.sample_in_kernel) b.spec = nullptr;
        return launch(b, variant);
    }
    if (variant == TR_VARIANT_TILED) return launch_tiled(a);
    return launch_generic(a);
}

int read_device_status(int* flags, bool clear) {
    unsigned int v = 0, site = 0;
    if (!check_cuda(cudaMemcpyFromSymbol(&v, g_device_status, sizeof v), "cudaMemcpyFromSymbol") ||
        !check_cuda(cudaMemcpyFromSymbol(&site, g_bounds_site, sizeof site), "cudaMemcpyFromSymbol"))
        return TR_ERR_CUDA;
    if (clear) {
        const unsigned int zero = 0;
        if (!check_cuda(cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero), "cudaMemcpyToSymbol") ||
            !check_cuda(cudaMemcpyToSymbol(g_bounds_site, &zero, sizeof zero), "cudaMemcpyToSymbol"))
            return TR_ERR_CUDA;
    }
    if (flags) *flags = (int)(v | ((site & 255u) << 8));
    return TR_OK;
}

void tune_tiled(int band_bytes, int stages, int ctas_per_sm, int flags) {
    g_flags.store(flags);
    g_band_bytes.store(band_bytes > 0 ? band_bytes : 0);
    g_stages.store(stages > 0 ? stages : 0);
    g_ctas_per_sm.store(ctas_per_sm > 0 ? ctas_per_sm : 0);
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
uint64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

}  // namespace trfn

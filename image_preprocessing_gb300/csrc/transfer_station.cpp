// Double-buffered feeding of the fused kernel from pinned host memory.
//
// The TransferStation of the Tech-Renaissance article "(10) Multi-threaded
// preprocessing, NUMA awareness, asynchronous double buffering"
// (tech-renaissance.cn/blog/?p=481, §四) alternates two pinned buffers A/B with
// four atomic readable/writeable flags and a condition variable, so that the
// CPU fills one buffer while the GPU consumes the other.  On GB300 the
// preprocessing itself runs on the GPU, so the buffers that alternate are two
// device input slots, and the hand-over is expressed with CUDA events between
// a copy stream and a compute stream instead of host flags:
//
//   batch k, slot s = k % 2
//   copy stream:    wait done[s]   (the kernel that last read slot s)
//                   H2D images (and records) -> slot s;   record copied[s]
//   compute stream: wait copied[s]; [wait d2h[s]]  (result copy of batch k-2)
//                   fused kernel slot s -> d_dst;         record done[s]
//   d2h stream:     wait done[s];  D2H d_dst -> h_dst;    record d2h[s]
//
// so the copy of batch k+1 overlaps the kernel of batch k.  The host never
// blocks except in tr_ts_sync(), which polls the events against a deadline.
// Slot layout: [images][records][filler image][filler record], each zone on a
// 256-byte boundary, after the article's [labels][padding][image] zones (§四).
// A short batch is padded to full size with the filler, the first image of the
// first batch (the article's incomplete-batch filling, §四.1).

#include <cuda_runtime.h>

#include <chrono>
#include <mutex>
#include <new>
#include <thread>

#include "internal.h"

struct tr_transfer_station {
    int device = 0;
    uint8_t* slot[2] = {nullptr, nullptr};
    size_t slot_bytes = 0;
    cudaStream_t copy = nullptr, compute = nullptr, d2h = nullptr;
    cudaEvent_t copied[2] = {nullptr, nullptr};
    cudaEvent_t done[2] = {nullptr, nullptr};
    cudaEvent_t d2h_done[2] = {nullptr, nullptr};
    bool done_used[2] = {false, false};
    bool d2h_used[2] = {false, false};
    bool filler_saved = false;   // the first batch's first image and record are in both slots
    long long next_batch = 0;
    std::mutex mu;
};

namespace {

// A staged zone to give back once its upload has finished.  Each submit
// queues its own (a host function of an earlier batch may not have run yet
// when the next batch on the same slot is queued).
struct StagedRelease {
    tr_staging* st = nullptr;
    long long batch = 0;
};
void CUDART_CB release_staged(void* arg) {
    StagedRelease* r = static_cast<StagedRelease*>(arg);
    trfn::stage_release_from_stream(r->st, r->batch);
    delete r;
}

}  // namespace

namespace {

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

// Slot layout: [N images][pad][N records][pad][filler image][pad][filler
// record][pad][scheduling workspace].  The filler is the first image (and
// record) of the first batch, kept for padding short batches (the article's
// incomplete-batch filling, §四.1).  The workspace (tr_workspace_bytes) lets
// the station's kernels hand out bands dynamically; the kernels run one after
// another on the compute stream, so slot A's workspace serves them all.
struct SlotLayout {
    size_t img, images, records, filler, filler_rec, ws, total;
};

SlotLayout slot_layout(int N, int H, int W, int C) {
    SlotLayout l;
    l.img = (size_t)H * W * C;
    l.images = 0;
    l.records = align256((size_t)N * l.img);
    l.filler = l.records + align256((size_t)N * sizeof(tr_aug_param));
    l.filler_rec = l.filler + align256(l.img);
    l.ws = l.filler_rec + align256(sizeof(tr_aug_param));
    l.total = l.ws + align256(tr_workspace_bytes());
    return l;
}

bool ok(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return true;
    trfn::set_last_error(what, (int)e);
    return false;
}

// Makes `device` current for the lifetime of the guard.
class DeviceGuard {
 public:
    explicit DeviceGuard(int device) {
        if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
        if (prev_ != device) cudaSetDevice(device);
    }
    ~DeviceGuard() {
        if (prev_ >= 0) cudaSetDevice(prev_);
    }

 private:
    int prev_ = -1;
};

void destroy_events(tr_transfer_station* ts) {
    for (int s = 0; s < 2; ++s) {
        if (ts->copied[s]) cudaEventDestroy(ts->copied[s]);
        if (ts->done[s]) cudaEventDestroy(ts->done[s]);
        if (ts->d2h_done[s]) cudaEventDestroy(ts->d2h_done[s]);
        ts->copied[s] = ts->done[s] = ts->d2h_done[s] = nullptr;
    }
}

// TR_OK when every used event has completed, TR_ERR_TIMEOUT at the deadline.
int wait_events(tr_transfer_station* ts, int timeout_ms) {
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        bool all = true;
        for (int s = 0; s < 2; ++s) {
            cudaEvent_t evs[2] = {ts->done_used[s] ? ts->done[s] : nullptr,
                                  ts->d2h_used[s] ? ts->d2h_done[s] : nullptr};
            for (cudaEvent_t ev : evs) {
                if (!ev) continue;
                const cudaError_t e = cudaEventQuery(ev);
                if (e == cudaErrorNotReady) {
                    all = false;
                } else if (e != cudaSuccess) {
                    trfn::set_last_error("cudaEventQuery", (int)e);
                    return TR_ERR_CUDA;
                }
            }
        }
        if (all) return TR_OK;
        if (timeout_ms >= 0) {
            const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                                std::chrono::steady_clock::now() - t0)
                                .count();
            if (ms >= timeout_ms) return TR_ERR_TIMEOUT;
        }
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

}  // namespace

extern "C" {

size_t tr_ts_slot_bytes(int N, int H, int W, int C) {
    if (N < 0 || H < 1 || W < 1 || C < 1) return 0;
    return slot_layout(N, H, W, C).total;
}

int tr_ts_create(int device, void* const d_slot[2], size_t slot_bytes, void* copy_stream,
                 void* compute_stream, void* d2h_stream, tr_transfer_station** out) {
    if (out == nullptr || d_slot == nullptr || d_slot[0] == nullptr || d_slot[1] == nullptr ||
        slot_bytes == 0 || copy_stream == nullptr || compute_stream == nullptr || device < 0)
        return TR_ERR_INVALID_ARGUMENT;
    *out = nullptr;
    tr_transfer_station* ts = new (std::nothrow) tr_transfer_station();
    if (ts == nullptr) return TR_ERR_INVALID_ARGUMENT;
    ts->device = device;
    ts->slot[0] = static_cast<uint8_t*>(d_slot[0]);
    ts->slot[1] = static_cast<uint8_t*>(d_slot[1]);
    ts->slot_bytes = slot_bytes;
    ts->copy = static_cast<cudaStream_t>(copy_stream);
    ts->compute = static_cast<cudaStream_t>(compute_stream);
    ts->d2h = static_cast<cudaStream_t>(d2h_stream);
    DeviceGuard guard(device);
    for (int s = 0; s < 2; ++s) {
        if (!ok(cudaEventCreateWithFlags(&ts->copied[s], cudaEventDisableTiming), "cudaEventCreate") ||
            !ok(cudaEventCreateWithFlags(&ts->done[s], cudaEventDisableTiming), "cudaEventCreate") ||
            !ok(cudaEventCreateWithFlags(&ts->d2h_done[s], cudaEventDisableTiming), "cudaEventCreate")) {
            destroy_events(ts);
            delete ts;
            return TR_ERR_CUDA;
        }
    }
    *out = ts;
    return TR_OK;
}

}  // extern "C"

namespace {

// Batch k of N images, of which the first n_valid come from the host and the
// rest repeat the filler; see tr_ts_submit and tr_ts_submit_partial.
int submit_impl(tr_transfer_station* ts, const uint8_t* h_src, const tr_aug_param* h_params, int n_valid,
                void* d_dst, void* h_dst, int N, int H, int W, int C, const float* mean, const float* std,
                int out_dtype, int out_layout, long long* batch_index, tr_staging* stage = nullptr,
                long long stage_batch = 0) {
    if (ts == nullptr || h_src == nullptr || d_dst == nullptr || N < 1 || n_valid < 1 || n_valid > N)
        return TR_ERR_INVALID_ARGUMENT;
    if (h_dst != nullptr && ts->d2h == nullptr) return TR_ERR_INVALID_ARGUMENT;
    // the kernel's own argument checks (shape, type, layout, mean/std), with
    // nothing launched, before any copy is queued
    int rc = tr_fused_norm(nullptr, nullptr, 0, H, W, C, mean, std, nullptr, out_dtype, out_layout, nullptr);
    if (rc != TR_OK) return rc;
    const SlotLayout l = slot_layout(N, H, W, C);
    const bool room_for_filler = l.ws <= ts->slot_bytes;
    const bool room_for_ws = l.total <= ts->slot_bytes;
    if (l.filler > ts->slot_bytes && (h_params != nullptr || n_valid < N)) return TR_ERR_INVALID_ARGUMENT;
    if (l.records > ts->slot_bytes) return TR_ERR_INVALID_ARGUMENT;
    if (n_valid < N && !room_for_filler) return TR_ERR_INVALID_ARGUMENT;
    const size_t out_bytes = (size_t)N * H * W * (out_layout == TR_LAYOUT_NHWC4 ? 4 : C) *
                             (out_dtype == TR_OUT_F16 ? 2 : 4);

    std::lock_guard<std::mutex> lock(ts->mu);
    DeviceGuard guard(ts->device);
    const long long k = ts->next_batch;
    const int s = (int)(k & 1);
    uint8_t* slot = ts->slot[s];
    const tr_aug_param* d_params =
        h_params ? reinterpret_cast<const tr_aug_param*>(slot + l.records) : nullptr;
    const size_t rec = sizeof(tr_aug_param);

    if (ts->done_used[s] && !ok(cudaStreamWaitEvent(ts->copy, ts->done[s], 0), "cudaStreamWaitEvent"))
        return TR_ERR_CUDA;
    if (!ok(cudaMemcpyAsync(slot, h_src, (size_t)n_valid * l.img, cudaMemcpyHostToDevice, ts->copy),
            "cudaMemcpyAsync"))
        return TR_ERR_CUDA;
    if (h_params && !ok(cudaMemcpyAsync(slot + l.records, h_params, (size_t)n_valid * rec,
                                        cudaMemcpyHostToDevice, ts->copy),
                        "cudaMemcpyAsync"))
        return TR_ERR_CUDA;
    if (stage != nullptr) {
        // the host zone is free again once the copies above have finished
        StagedRelease* r = new (std::nothrow) StagedRelease{stage, stage_batch};
        if (r == nullptr) return TR_ERR_INVALID_ARGUMENT;
        trfn::stage_release_queued(stage);
        const cudaError_t e = cudaLaunchHostFunc(ts->copy, release_staged, r);
        if (e != cudaSuccess) {
            // not queued: release now (the copies may still be reading the
            // zone, so wait for them first)
            cudaStreamSynchronize(ts->copy);
            release_staged(r);
            trfn::set_last_error("cudaLaunchHostFunc", (int)e);
            return TR_ERR_CUDA;
        }
    }
    if (!ts->filler_saved && room_for_filler) {
        // the first batch's first image and record become the filler, in
        // both slots (the other slot is not in use before batch 1)
        for (int t = 0; t < 2; ++t) {
            if (!ok(cudaMemcpyAsync(ts->slot[t] + l.filler, slot, l.img, cudaMemcpyDeviceToDevice, ts->copy),
                    "cudaMemcpyAsync"))
                return TR_ERR_CUDA;
            const cudaError_t e =
                h_params ? cudaMemcpyAsync(ts->slot[t] + l.filler_rec, slot + l.records, rec,
                                           cudaMemcpyDeviceToDevice, ts->copy)
                         : cudaMemsetAsync(ts->slot[t] + l.filler_rec, 0, rec, ts->copy);
            if (!ok(e, "filler record")) return TR_ERR_CUDA;
        }
        ts->filler_saved = true;
    }
    for (int i = n_valid; i < N; ++i) {
        if (!ok(cudaMemcpyAsync(slot + (size_t)i * l.img, slot + l.filler, l.img, cudaMemcpyDeviceToDevice,
                                ts->copy),
                "cudaMemcpyAsync"))
            return TR_ERR_CUDA;
        if (h_params && !ok(cudaMemcpyAsync(slot + l.records + (size_t)i * rec, slot + l.filler_rec, rec,
                                            cudaMemcpyDeviceToDevice, ts->copy),
                            "cudaMemcpyAsync"))
            return TR_ERR_CUDA;
    }
    if (!ok(cudaEventRecord(ts->copied[s], ts->copy), "cudaEventRecord")) return TR_ERR_CUDA;

    if (!ok(cudaStreamWaitEvent(ts->compute, ts->copied[s], 0), "cudaStreamWaitEvent")) return TR_ERR_CUDA;
    if (ts->d2h_used[s] &&
        !ok(cudaStreamWaitEvent(ts->compute, ts->d2h_done[s], 0), "cudaStreamWaitEvent"))
        return TR_ERR_CUDA;
    void* ws = nullptr;
    if (room_for_ws) {
        // cleared before every kernel: a kernel leaves it zero, except one
        // whose bounded waits ran out, and a batch costs far more than 2 KB
        ws = ts->slot[0] + l.ws;
        if (!ok(cudaMemsetAsync(ws, 0, tr_workspace_bytes(), ts->compute), "cudaMemsetAsync")) return TR_ERR_CUDA;
    }
    rc = tr_fused_norm_ws(slot, d_dst, N, H, W, C, mean, std, d_params, out_dtype, out_layout, ts->compute,
                          TR_VARIANT_AUTO, ws);
    if (rc != TR_OK) return rc;
    if (!ok(cudaEventRecord(ts->done[s], ts->compute), "cudaEventRecord")) return TR_ERR_CUDA;
    ts->done_used[s] = true;

    if (h_dst != nullptr) {
        if (!ok(cudaStreamWaitEvent(ts->d2h, ts->done[s], 0), "cudaStreamWaitEvent")) return TR_ERR_CUDA;
        if (!ok(cudaMemcpyAsync(h_dst, d_dst, out_bytes, cudaMemcpyDeviceToHost, ts->d2h),
                "cudaMemcpyAsync"))
            return TR_ERR_CUDA;
        if (!ok(cudaEventRecord(ts->d2h_done[s], ts->d2h), "cudaEventRecord")) return TR_ERR_CUDA;
        ts->d2h_used[s] = true;
    }
    ts->next_batch = k + 1;
    if (batch_index) *batch_index = k;
    return TR_OK;
}

}  // namespace

extern "C" {

int tr_ts_submit(tr_transfer_station* ts, const uint8_t* h_src, const tr_aug_param* h_params,
                 void* d_dst, void* h_dst, int N, int H, int W, int C, const float* mean,
                 const float* std, int out_dtype, int out_layout, long long* batch_index) {
    return submit_impl(ts, h_src, h_params, N, d_dst, h_dst, N, H, W, C, mean, std, out_dtype, out_layout,
                       batch_index);
}

int tr_ts_submit_partial(tr_transfer_station* ts, const uint8_t* h_src, const tr_aug_param* h_params,
                         int n_valid, void* d_dst, void* h_dst, int N, int H, int W, int C,
                         const float* mean, const float* std, int out_dtype, int out_layout,
                         long long* batch_index) {
    return submit_impl(ts, h_src, h_params, n_valid, d_dst, h_dst, N, H, W, C, mean, std, out_dtype,
                       out_layout, batch_index);
}

int tr_ts_submit_staged(tr_transfer_station* ts, tr_staging* st, const tr_stage_batch* b, int with_records,
                        void* d_dst, void* h_dst, int N, int H, int W, int C, const float* mean,
                        const float* std, int out_dtype, int out_layout, long long* batch_index) {
    if (ts == nullptr) return TR_ERR_INVALID_ARGUMENT;
    const int rc = trfn::stage_batch_ok(st, b, N, H, W, C);
    if (rc != TR_OK) return rc;
    return submit_impl(ts, b->images, with_records ? b->records : nullptr, b->count, d_dst, h_dst, N, H, W, C,
                       mean, std, out_dtype, out_layout, batch_index, st, b->batch);
}

int tr_ts_sync(tr_transfer_station* ts, int timeout_ms) {
    if (ts == nullptr) return TR_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(ts->mu);
    DeviceGuard guard(ts->device);
    return wait_events(ts, timeout_ms);
}

int tr_ts_destroy(tr_transfer_station* ts) {
    if (ts == nullptr) return TR_ERR_INVALID_ARGUMENT;
    int rc;
    {
        std::lock_guard<std::mutex> lock(ts->mu);
        DeviceGuard guard(ts->device);
        rc = wait_events(ts, -1);
        destroy_events(ts);
    }
    delete ts;
    return rc;
}

}  // extern "C"

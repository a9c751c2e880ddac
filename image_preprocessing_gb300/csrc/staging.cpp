// Host staging zones for the TransferStation: preprocessing workers (host
// threads) write samples into one of two caller-owned host zones while the
// station uploads the other.
//
// The Tech-Renaissance article "(10) Multi-threaded preprocessing, NUMA
// awareness, asynchronous double buffering" (tech-renaissance.cn/blog/?p=481)
// describes this hand-over in §四: workers fill the current pinned buffer; a
// buffer that holds a whole batch, or the last samples once every worker has
// run out, becomes readable for the GPU side, and the workers move on to the
// other buffer, waiting for it to be given back if the GPU has not finished
// with it.  §四.2 gives two ways of placing a sample: a shared request
// counter that hands out the next free place (fast), or a place computed from
// the sample's own number, so that every run lays batches out identically
// (reproducible).
//
// Here batch b always lives in zone b % 2 and a zone is writeable for exactly
// one batch at a time (zone_batch).  A producer claims a place with
// tr_stage_acquire (waiting, with a deadline, until the zone holds its
// batch), writes the image and record there and calls tr_stage_commit.  When
// a batch's last place is committed the zone turns readable; the consumer
// takes batches in order with tr_stage_wait_readable and gives each zone back
// with tr_stage_release, which assigns it batch b + 2 and wakes the producers
// waiting for it.  tr_stage_close marks the end of the data: the last batch
// is then readable with fewer than N samples (the station pads it, §四.1).
//
// Fast mode claims with one compare-and-swap on the request counter while the
// target zone is writeable; only waits take the mutex.  Commits are a per-place
// state change and a counter increment; the mutex is taken when a batch may
// have completed.

#include <atomic>
#include <chrono>
#include <condition_variable>
#include <memory>
#include <mutex>
#include <new>

#include "internal.h"

namespace {

constexpr long long kSealed = 1LL << 62;   // request counter sealed by tr_stage_close (fast mode)

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

enum PlaceState : unsigned char { kFree = 0, kClaimed = 1, kCommitted = 2 };

}  // namespace

struct tr_staging {
    uint8_t* zone[2] = {nullptr, nullptr};
    int N = 0;
    size_t img = 0;          // bytes of one image
    size_t records = 0;      // byte offset of the record array in a zone
    int mode = TR_STAGE_FAST;

    std::atomic<long long> zone_batch[2];   // the batch each zone is writeable for
    std::atomic<int> committed[2];          // places of that batch committed so far
    std::unique_ptr<std::atomic<unsigned char>[]> place[2];   // PlaceState per place
    bool readable[2] = {false, false};      // under mu
    bool handed_out[2] = {false, false};    // given to the consumer, not yet released (under mu)

    std::atomic<long long> request{0};      // fast mode: next sample number
    long long max_claimed = -1;             // reproducible mode: highest sample claimed (under mu)
    std::atomic<bool> closed{false};
    long long total = 0;                    // samples in the data set, once closed
    long long next_consume = 0;             // next batch for the consumer (under mu)

    std::atomic<int> pending_releases{0};   // releases queued on a CUDA stream
    std::mutex mu;
    std::condition_variable cv_writeable;   // a zone was given back, or the data was closed
    std::condition_variable cv_readable;    // a batch completed, or the data was closed
    std::condition_variable cv_pending;     // a queued release ran
};

namespace {

// Number of samples batch b holds once complete: N, or the remainder for the
// last batch of closed data.  Caller holds mu, or `closed` was read true.
int batch_target(const tr_staging* st, long long b) {
    if (!st->closed.load()) return st->N;
    const long long last = st->total > 0 ? (st->total - 1) / st->N : -1;
    if (b < last) return st->N;
    if (b == last) return (int)(st->total - last * st->N);
    return 0;
}

// Marks zone z readable when its batch is complete.  Caller holds mu.
void check_complete(tr_staging* st, int z) {
    if (st->readable[z] || st->handed_out[z]) return;
    const long long b = st->zone_batch[z].load();
    const int target = batch_target(st, b);
    if (target > 0 && st->committed[z].load() == target) {
        st->readable[z] = true;
        st->cv_readable.notify_all();
    }
}

template <class Pred>
bool wait_until(std::condition_variable& cv, std::unique_lock<std::mutex>& lock, int timeout_ms, Pred pred) {
    if (timeout_ms < 0) {
        cv.wait(lock, pred);
        return true;
    }
    return cv.wait_for(lock, std::chrono::milliseconds(timeout_ms), pred);
}

void fill_slot(const tr_staging* st, long long sample, tr_stage_slot* slot) {
    const long long b = sample / st->N;
    const int i = (int)(sample - b * st->N);
    const int z = (int)(b & 1);
    slot->image = st->zone[z] + (size_t)i * st->img;
    slot->record = reinterpret_cast<tr_aug_param*>(st->zone[z] + st->records) + i;
    slot->sample = sample;
    slot->batch = b;
    slot->index = i;
    slot->zone = z;
}

int acquire_fast(tr_staging* st, int timeout_ms, tr_stage_slot* slot) {
    for (;;) {
        long long r = st->request.load();
        if (r & kSealed) return TR_END_OF_DATA;
        const long long b = r / st->N;
        const int z = (int)(b & 1);
        if (st->zone_batch[z].load() == b) {
            // the zone holds this batch and cannot be given back before this
            // place is committed, so winning the counter claims the place
            if (st->request.compare_exchange_weak(r, r + 1)) {
                st->place[z][r - b * st->N].store(kClaimed);
                fill_slot(st, r, slot);
                return TR_OK;
            }
            continue;
        }
        std::unique_lock<std::mutex> lock(st->mu);
        const bool ok = wait_until(st->cv_writeable, lock, timeout_ms, [&] {
            const long long r2 = st->request.load();
            return (r2 & kSealed) || r2 != r || st->zone_batch[z].load() == b;
        });
        if (!ok) return TR_ERR_TIMEOUT;
    }
}

int acquire_reproducible(tr_staging* st, long long sample, int timeout_ms, tr_stage_slot* slot) {
    const long long b = sample / st->N;
    const int i = (int)(sample - b * st->N);
    const int z = (int)(b & 1);
    std::unique_lock<std::mutex> lock(st->mu);
    if (st->closed.load() && sample >= st->total) return TR_END_OF_DATA;
    if (st->zone_batch[z].load() > b) return TR_ERR_INVALID_ARGUMENT;   // batch already consumed
    const bool ok = wait_until(st->cv_writeable, lock, timeout_ms, [&] {
        return st->zone_batch[z].load() >= b || (st->closed.load() && sample >= st->total);
    });
    if (!ok) return TR_ERR_TIMEOUT;
    if (st->closed.load() && sample >= st->total) return TR_END_OF_DATA;
    if (st->zone_batch[z].load() != b) return TR_ERR_INVALID_ARGUMENT;
    unsigned char expect = kFree;
    if (!st->place[z][i].compare_exchange_strong(expect, kClaimed)) return TR_ERR_INVALID_ARGUMENT;
    if (sample > st->max_claimed) st->max_claimed = sample;
    fill_slot(st, sample, slot);
    return TR_OK;
}

// Gives zone z (holding batch b) back to the producers for batch b + 2.
void release_zone(tr_staging* st, int z, long long b) {
    std::lock_guard<std::mutex> lock(st->mu);
    for (int i = 0; i < st->N; ++i) st->place[z][i].store(kFree);
    st->committed[z].store(0);
    st->readable[z] = false;
    st->handed_out[z] = false;
    st->zone_batch[z].store(b + 2);
    st->cv_writeable.notify_all();
}

}  // namespace

extern "C" {

size_t tr_stage_zone_bytes(int N, int H, int W, int C) {
    if (N < 1 || H < 1 || W < 1 || C < 1) return 0;
    return align256((size_t)N * H * W * C) + align256((size_t)N * sizeof(tr_aug_param));
}

int tr_stage_create(void* const zone[2], size_t zone_bytes, int N, int H, int W, int C, int mode,
                    tr_staging** out) {
    if (out == nullptr) return TR_ERR_INVALID_ARGUMENT;
    *out = nullptr;
    if (zone == nullptr || zone[0] == nullptr || zone[1] == nullptr || zone[0] == zone[1])
        return TR_ERR_INVALID_ARGUMENT;
    if (mode != TR_STAGE_FAST && mode != TR_STAGE_REPRODUCIBLE) return TR_ERR_INVALID_ARGUMENT;
    const size_t need = tr_stage_zone_bytes(N, H, W, C);
    if (need == 0 || zone_bytes < need) return TR_ERR_INVALID_ARGUMENT;
    const uintptr_t a = (uintptr_t)zone[0], b = (uintptr_t)zone[1];
    if (a < b + zone_bytes && b < a + zone_bytes) return TR_ERR_INVALID_ARGUMENT;   // zones overlap
    if (a % alignof(tr_aug_param) || b % alignof(tr_aug_param)) return TR_ERR_INVALID_ARGUMENT;
    tr_staging* st = new (std::nothrow) tr_staging();
    if (st == nullptr) return TR_ERR_INVALID_ARGUMENT;
    st->zone[0] = static_cast<uint8_t*>(zone[0]);
    st->zone[1] = static_cast<uint8_t*>(zone[1]);
    st->N = N;
    st->img = (size_t)H * W * C;
    st->records = align256((size_t)N * st->img);
    st->mode = mode;
    for (int z = 0; z < 2; ++z) {
        st->zone_batch[z].store(z);
        st->committed[z].store(0);
        st->place[z].reset(new (std::nothrow) std::atomic<unsigned char>[N]);
        if (!st->place[z]) {
            delete st;
            return TR_ERR_INVALID_ARGUMENT;
        }
        for (int i = 0; i < N; ++i) st->place[z][i].store(kFree);
    }
    *out = st;
    return TR_OK;
}

int tr_stage_acquire(tr_staging* st, long long sample, int timeout_ms, tr_stage_slot* slot) {
    if (st == nullptr || slot == nullptr) return TR_ERR_INVALID_ARGUMENT;
    if (st->mode == TR_STAGE_FAST) return acquire_fast(st, timeout_ms, slot);
    if (sample < 0) return TR_ERR_INVALID_ARGUMENT;
    return acquire_reproducible(st, sample, timeout_ms, slot);
}

int tr_stage_commit(tr_staging* st, const tr_stage_slot* slot) {
    if (st == nullptr || slot == nullptr || slot->zone < 0 || slot->zone > 1 || slot->index < 0 ||
        slot->index >= st->N || slot->batch < 0)
        return TR_ERR_INVALID_ARGUMENT;
    const int z = slot->zone;
    if ((slot->batch & 1) != z || st->zone_batch[z].load() != slot->batch) return TR_ERR_INVALID_ARGUMENT;
    unsigned char expect = kClaimed;
    if (!st->place[z][slot->index].compare_exchange_strong(expect, kCommitted)) return TR_ERR_INVALID_ARGUMENT;
    const int c = st->committed[z].fetch_add(1) + 1;
    if (c == st->N || st->closed.load()) {
        std::lock_guard<std::mutex> lock(st->mu);
        check_complete(st, z);
    }
    return TR_OK;
}

int tr_stage_close(tr_staging* st, long long total_samples) {
    if (st == nullptr || total_samples < -1) return TR_ERR_INVALID_ARGUMENT;
    std::lock_guard<std::mutex> lock(st->mu);
    if (st->closed.load()) return TR_ERR_INVALID_ARGUMENT;
    long long total;
    if (st->mode == TR_STAGE_FAST) {
        // seal the counter: no place is handed out after this point
        long long r = st->request.load();
        for (;;) {
            if (total_samples >= 0 && total_samples != r) return TR_ERR_INVALID_ARGUMENT;
            if (st->request.compare_exchange_weak(r, r | kSealed)) break;
        }
        total = r;
    } else {
        total = total_samples >= 0 ? total_samples : st->max_claimed + 1;
        if (total <= st->max_claimed) return TR_ERR_INVALID_ARGUMENT;
    }
    if (total < st->next_consume * (long long)st->N) return TR_ERR_INVALID_ARGUMENT;
    st->total = total;
    st->closed.store(true);
    check_complete(st, 0);
    check_complete(st, 1);
    st->cv_writeable.notify_all();
    st->cv_readable.notify_all();
    return TR_OK;
}

int tr_stage_wait_readable(tr_staging* st, int timeout_ms, tr_stage_batch* batch) {
    if (st == nullptr || batch == nullptr) return TR_ERR_INVALID_ARGUMENT;
    std::unique_lock<std::mutex> lock(st->mu);
    const long long b = st->next_consume;
    const int z = (int)(b & 1);
    bool end = false;
    const bool ok = wait_until(st->cv_readable, lock, timeout_ms, [&] {
        if (st->readable[z] && !st->handed_out[z] && st->zone_batch[z].load() == b) return true;
        if (st->closed.load() && batch_target(st, b) == 0) {
            end = true;
            return true;
        }
        return false;
    });
    if (!ok) return TR_ERR_TIMEOUT;
    if (end) return TR_END_OF_DATA;
    st->handed_out[z] = true;
    st->next_consume = b + 1;
    batch->images = st->zone[z];
    batch->records = reinterpret_cast<tr_aug_param*>(st->zone[z] + st->records);
    batch->batch = b;
    batch->count = st->committed[z].load();
    batch->zone = z;
    return TR_OK;
}

int tr_stage_release(tr_staging* st, long long batch) {
    if (st == nullptr || batch < 0) return TR_ERR_INVALID_ARGUMENT;
    const int z = (int)(batch & 1);
    {
        std::lock_guard<std::mutex> lock(st->mu);
        if (!st->handed_out[z] || st->zone_batch[z].load() != batch) return TR_ERR_INVALID_ARGUMENT;
    }
    release_zone(st, z, batch);
    return TR_OK;
}

int tr_stage_destroy(tr_staging* st) {
    if (st == nullptr) return TR_ERR_INVALID_ARGUMENT;
    {
        // releases queued on a stream (tr_ts_submit_staged) still refer to st
        std::unique_lock<std::mutex> lock(st->mu);
        st->cv_pending.wait(lock, [&] { return st->pending_releases.load() == 0; });
    }
    delete st;
    return TR_OK;
}

}  // extern "C"

namespace trfn {

// Parts of a staged batch that the station needs (see transfer_station.cpp).
int stage_batch_ok(const tr_staging* st, const tr_stage_batch* b, int N, int H, int W, int C) {
    if (st == nullptr || b == nullptr || b->zone < 0 || b->zone > 1) return TR_ERR_INVALID_ARGUMENT;
    if (st->N != N || st->img != (size_t)H * W * C) return TR_ERR_INVALID_ARGUMENT;
    if (b->count < 1 || b->count > N || b->images != st->zone[b->zone]) return TR_ERR_INVALID_ARGUMENT;
    if (st->zone_batch[b->zone].load() != b->batch) return TR_ERR_INVALID_ARGUMENT;
    return TR_OK;
}

void stage_release_queued(tr_staging* st) { st->pending_releases.fetch_add(1); }

// Runs on a CUDA stream (cudaLaunchHostFunc) once the zone's upload has
// finished: gives the zone back.  Makes no CUDA call.
void stage_release_from_stream(tr_staging* st, long long batch) {
    const int z = (int)(batch & 1);
    bool still_out;
    {
        std::lock_guard<std::mutex> lock(st->mu);
        still_out = st->handed_out[z] && st->zone_batch[z].load() == batch;
    }
    if (still_out) release_zone(st, z, batch);   // else the consumer released it already
    std::lock_guard<std::mutex> lock(st->mu);
    st->pending_releases.fetch_sub(1);
    st->cv_pending.notify_all();
}

}  // namespace trfn

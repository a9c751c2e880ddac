// Host-only record of the workspace that this library's last launch on each
// stream used.  A launch that asks to overlap the kernel before it in its
// stream (TR_LAUNCH_OVERLAP_PREVIOUS) must not share that kernel's workspace:
// its ticket counters are still in use and are zeroed by that kernel's last
// CTA.  No CUDA header is needed, so the logic is testable on any host.
#pragma once

#include <mutex>

namespace trfn {

template <int kEntries>
class StreamWorkspaceGuard {
 public:
    // Records `workspace` as the last one used on `stream` and returns true
    // when the launch must not overlap on that account: its workspace is the
    // one the previous launch on the stream used, or the stream is missing
    // from the table after an entry has been replaced (its entry may have
    // been the one dropped).  A null workspace is never shared.  A fixed
    // table (oldest entry replaced): nothing is allocated.
    bool note(void* stream, void* workspace) {
        std::lock_guard<std::mutex> lock(mu_);
        if (table_[last_].used && table_[last_].stream == stream) return hit(last_, workspace);
        for (int i = 0; i < kEntries; ++i)
            if (table_[i].used && table_[i].stream == stream) return hit(i, workspace);
        if (table_[next_].used) replaced_ = true;
        table_[next_] = Entry{stream, workspace, true};
        last_ = next_;
        next_ = (next_ + 1) % kEntries;
        return replaced_ && workspace != nullptr;
    }

 private:
    struct Entry {
        void* stream = nullptr;
        void* ws = nullptr;
        bool used = false;
    };

    bool hit(int i, void* workspace) {
        Entry& e = table_[i];
        const bool same = (workspace != nullptr && e.ws == workspace);
        e.ws = workspace;
        last_ = i;   // one comparison on the next call from a single stream
        return same;
    }

    std::mutex mu_;
    Entry table_[kEntries];
    int next_ = 0;
    int last_ = 0;
    bool replaced_ = false;
};

}  // namespace trfn

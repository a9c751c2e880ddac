// Host test of the stream/workspace guard that decides whether a launch may
// overlap the kernel before it (image_preprocessing_gb300/csrc/stream_guard.h).
// Exit status 0 when every check holds; each failure is printed.

#include <cstdint>
#include <cstdio>
#include <thread>
#include <vector>

#include "stream_guard.h"

static int g_failures = 0;

#define CHECK(cond)                                                          \
    do {                                                                     \
        if (!(cond)) {                                                       \
            std::printf("FAILED line %d: %s\n", __LINE__, #cond);            \
            ++g_failures;                                                    \
        }                                                                    \
    } while (0)

static void* P(uintptr_t v) { return reinterpret_cast<void*>(v); }

int main() {
    {
        trfn::StreamWorkspaceGuard<4> g;
        void *s1 = P(0x1000), *s2 = P(0x2000), *A = P(0xA000), *B = P(0xB000);
        CHECK(!g.note(s1, A));        // first launch on a stream
        CHECK(g.note(s1, A));         // the same workspace as the launch before it
        CHECK(!g.note(s1, B));        // another workspace
        CHECK(g.note(s1, B));
        CHECK(!g.note(s1, nullptr));  // no workspace: nothing shared
        CHECK(!g.note(s1, nullptr));
        CHECK(!g.note(s1, A));
        CHECK(!g.note(s2, A));        // another stream: its own previous kernel
        CHECK(g.note(s2, A));
        CHECK(g.note(s1, A));         // s1's last launch (before s2's) used A
    }
    {
        // alternating streams keep their own records (the last-entry shortcut
        // must not mix them up)
        trfn::StreamWorkspaceGuard<4> g;
        void *s1 = P(0x10), *s2 = P(0x20), *s3 = P(0x30), *A = P(0xA0), *B = P(0xB0);
        CHECK(!g.note(s1, A));
        CHECK(!g.note(s2, B));
        CHECK(!g.note(s3, A));
        CHECK(g.note(s1, A));
        CHECK(g.note(s2, B));
        CHECK(!g.note(s3, B));
        CHECK(!g.note(s1, B));
        CHECK(!g.note(s2, A));
        CHECK(g.note(s3, B));
    }
    {
        // more streams than entries: once an entry has been replaced, a stream
        // missing from the table may be one whose entry was dropped, so its
        // launch with a workspace is treated as sharing; without a workspace
        // it is not
        trfn::StreamWorkspaceGuard<4> g;
        void* A = P(0xA00);
        void* B = P(0xB00);
        for (uintptr_t k = 1; k <= 4; ++k) CHECK(!g.note(P(k * 0x100), A));   // entries 0..3
        CHECK(g.note(P(0x100), A));          // still present: the same workspace
        CHECK(g.note(P(0x500), B));          // replaces entry 0 (0x100): a new stream, conservative
        CHECK(g.note(P(0x100), B));          // dropped, so conservative; replaces entry 1 (0x200)
        CHECK(!g.note(P(0x700), nullptr));   // no workspace: nothing shared; replaces entry 2 (0x300)
        CHECK(g.note(P(0x300), A));          // dropped: conservative; replaces entry 3 (0x400)
        CHECK(!g.note(P(0x700), A));         // present, last launch had no workspace
        CHECK(g.note(P(0x700), A));          // present, the same workspace
        CHECK(!g.note(P(0x500), A));         // present, its last launch used B
        CHECK(g.note(P(0x200), B));          // dropped earlier: conservative
    }
    {
        // many threads on their own streams: every stream ends with the
        // workspace of its own last call
        trfn::StreamWorkspaceGuard<64> g;
        constexpr int T = 8, K = 20000;
        std::vector<std::thread> th;
        std::vector<int> bad(T, 0);
        for (int t = 0; t < T; ++t) {
            th.emplace_back([&, t] {
                void* s = P(0x10000 + 0x100 * (uintptr_t)t);
                void* ws[2] = {P(0x900000 + 0x100 * (uintptr_t)t), P(0xA00000 + 0x100 * (uintptr_t)t)};
                g.note(s, ws[0]);
                for (int k = 1; k < K; ++k)
                    if (g.note(s, ws[k & 1])) ++bad[t];   // alternating workspaces never share
                if (!g.note(s, ws[(K - 1) & 1])) ++bad[t];   // repeating the last one does
            });
        }
        for (auto& x : th) x.join();
        for (int t = 0; t < T; ++t) CHECK(bad[t] == 0);
    }
    if (g_failures == 0) std::printf("stream guard: all checks passed\n");
    return g_failures == 0 ? 0 : 1;
}

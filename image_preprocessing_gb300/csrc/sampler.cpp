// Host sampler of the per-image augmentation records (tr_sample_aug_params).
//
// Follows the random decisions of the FusedNormalization article
// (tech-renaissance.cn/blog/?p=487): the flip draw of execute() (§五), the
// uniform()/randint() helpers over a counter-based Philox generator (§十), and
// generate_erase_rect() (§十二).  Binary32 arithmetic as the article writes it;
// this file is compiled without floating-point contraction so that every
// product and sum is rounded on its own, identically on x86-64 and aarch64.

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace trfn {
namespace {

// Philox4x32-10, Salmon et al., SC'11: ten rounds; each round multiplies
// counter words 0 and 2 by the two round multipliers (64-bit products),
// mixes the high halves with words 1 and 3 and the round key, and the key
// advances by the two Weyl increments between rounds.
class Philox4x32x10 {
 public:
    static void block(uint32_t x[4], uint32_t k0, uint32_t k1) {
        for (int round = 0; round < 10; ++round) {
            const uint64_t a = (uint64_t)x[0] * 0xD2511F53ull;
            const uint64_t b = (uint64_t)x[2] * 0xCD9E8D57ull;
            const uint32_t y0 = (uint32_t)(b >> 32) ^ x[1] ^ k0;
            const uint32_t y1 = (uint32_t)b;
            const uint32_t y2 = (uint32_t)(a >> 32) ^ x[3] ^ k1;
            const uint32_t y3 = (uint32_t)a;
            x[0] = y0; x[1] = y1; x[2] = y2; x[3] = y3;
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
    }
};

// One draw per offset: key = seed, counter = (offset, 0, 0); the top 24 bits
// of the first output word.
class CounterStream {
 public:
    CounterStream(uint64_t seed, uint64_t offset) : seed_(seed), offset_(offset) {}

    uint32_t next24() {
        uint32_t x[4] = {(uint32_t)(offset_ & 0xFFFFFFFFu), (uint32_t)(offset_ >> 32), 0u, 0u};
        Philox4x32x10::block(x, (uint32_t)(seed_ & 0xFFFFFFFFu), (uint32_t)(seed_ >> 32));
        ++offset_;
        return x[0] >> 8;
    }
    // uniform(lo, hi) = lo + u*(hi - lo), u = k / 2^24
    float uniform(float lo, float hi) {
        const float u = (float)next24() * 5.9604644775390625e-8f;   // 2^-24
        return lo + u * (hi - lo);
    }
    // randint(lo, hi), inclusive: lo + floor(u*(hi - lo + 1)), exact in integers
    int randint(int lo, int hi) {
        const uint64_t k = next24();
        const uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
        return (int)((int64_t)lo + (int64_t)((k * span) >> 24));
    }
    uint64_t offset() const { return offset_; }

 private:
    uint64_t seed_;
    uint64_t offset_;
};

struct EraseRule {
    float p, scale_lo, scale_hi, log_ratio_lo, log_ratio_hi;
};

// generate_erase_rect: gate, then up to ten area/aspect attempts.
bool sample_rect(CounterStream& g, const EraseRule& r, int H, int W, tr_aug_param& out) {
    if (g.uniform(0.0f, 1.0f) >= r.p) return false;
    const float area_img = (float)H * (float)W;
    for (int attempt = 0; attempt < 10; ++attempt) {
        const float frac = r.scale_lo + g.uniform(0.0f, 1.0f) * (r.scale_hi - r.scale_lo);
        const float area = frac * area_img;
        const float log_ar = r.log_ratio_lo + g.uniform(0.0f, 1.0f) * (r.log_ratio_hi - r.log_ratio_lo);
        const float ar = std::exp(log_ar);
        const int h = (int)std::round(std::sqrt(area * ar));
        const int w = (int)std::round(std::sqrt(area / ar));
        if (h > 0 && w > 0 && h < H && w < W) {
            out.y0 = g.randint(0, H - h);
            out.x0 = g.randint(0, W - w);
            out.h = h;
            out.w = w;
            return true;
        }
    }
    return false;
}

}  // namespace
}  // namespace trfn

extern "C" int tr_sample_aug_params(uint64_t seed, uint64_t offset, int N, int H, int W,
                                    int flip_enabled, float flip_p, int erase_enabled, float erase_p,
                                    float scale_lo, float scale_hi, float ratio_lo, float ratio_hi,
                                    tr_aug_param* out_host, uint64_t* next_offset) {
    using namespace trfn;
    if (N < 0 || H < 1 || W < 1) return TR_ERR_INVALID_ARGUMENT;
    if (N > 0 && out_host == nullptr) return TR_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(flip_p) || !std::isfinite(erase_p)) return TR_ERR_INVALID_ARGUMENT;
    const bool erase = erase_enabled && erase_p > 0.0f;
    if (erase) {
        if (!std::isfinite(scale_lo) || !std::isfinite(scale_hi) || !std::isfinite(ratio_lo) ||
            !std::isfinite(ratio_hi) || scale_lo > scale_hi || ratio_lo <= 0.0f || ratio_lo > ratio_hi)
            return TR_ERR_INVALID_ARGUMENT;
    }
    CounterStream g(seed, offset);
    const EraseRule rule{erase_p, scale_lo, scale_hi, erase ? std::log(ratio_lo) : 0.0f,
                         erase ? std::log(ratio_hi) : 0.0f};
    for (int n = 0; n < N; ++n) {
        tr_aug_param rec{0, 0, 0, 0, 0};
        if (flip_enabled) rec.flip = (g.uniform(0.0f, 1.0f) < flip_p) ? 1 : 0;
        if (erase) sample_rect(g, rule, H, W, rec);
        out_host[n] = rec;
    }
    if (next_offset) *next_offset = g.offset();
    return TR_OK;
}

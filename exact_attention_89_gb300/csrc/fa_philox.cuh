// fa_philox.cuh -- counter-based random numbers for dropout: Philox4x32-10.
//
// Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11): a
// 4 x 32-bit counter is mixed with a 2 x 32-bit key by ten rounds; each round forms the 64-bit
// products of counter words 0 and 2 with two fixed multipliers and recombines their halves with
// words 1 and 3 and the key, and the key advances by two fixed (Weyl) increments between rounds.
// Being a pure function of (counter, key), the same keep decision is recomputed wherever it is
// needed (forward, backward, mask dump) with no state.
//
// Dropout keep rule of this library: the element (query i, key j) of head bh = b * Hq + hq is
// kept iff word (j mod 4) of Philox4x32-10(counter = (j / 4, i, bh, offset),
// key = (seed mod 2^32, seed / 2^32)) is below floor((1 - p) 2^32).
#pragma once

#include <cstdint>

namespace fa {

constexpr uint32_t kPhiloxMulA = 0xD2511F53u, kPhiloxMulB = 0xCD9E8D57u;
constexpr uint32_t kPhiloxBumpA = 0x9E3779B9u, kPhiloxBumpB = 0xBB67AE85u;

struct DropoutArgs {
    // The key of each of the ten rounds, (k0 + r bumpA, k1 + r bumpB) for the key (k0, k1) =
    // (seed mod 2^32, seed / 2^32): identical for every thread, so they travel in the kernel's
    // parameters instead of being recomputed per call.
    uint32_t round_key[10][2] = {};
    uint32_t offset = 0;                 // counter word 3
    uint32_t thresh = 0;                 // keep iff word < thresh
    float rscale = 1.f;                  // 1 / (1 - p)
};

// Host side: the round keys of a 64-bit seed.
inline void set_round_keys(DropoutArgs *dr, unsigned long long seed) {
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        dr->round_key[r][0] = k0;
        dr->round_key[r][1] = k1;
        k0 += kPhiloxBumpA;
        k1 += kPhiloxBumpB;
    }
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 x, const DropoutArgs &dr) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        // one widening multiply per product: both halves at once
        const uint64_t pA = static_cast<uint64_t>(kPhiloxMulA) * x.x;
        const uint64_t pB = static_cast<uint64_t>(kPhiloxMulB) * x.z;
        x = make_uint4(static_cast<uint32_t>(pB >> 32) ^ x.y ^ dr.round_key[round][0],
                       static_cast<uint32_t>(pB),
                       static_cast<uint32_t>(pA >> 32) ^ x.w ^ dr.round_key[round][1],
                       static_cast<uint32_t>(pA));
    }
    return x;
}

// The four keep words of keys 4m .. 4m+3 at query i of head bh.
__device__ __forceinline__ uint4 dropout_words(const DropoutArgs &dr, uint32_t m, uint32_t i,
                                               uint32_t bh) {
    return philox4x32_10(make_uint4(m, i, bh, dr.offset), dr);
}

}  // namespace fa

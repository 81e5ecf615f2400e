// Dropout keep masks from Philox-4x32-10 (Salmon, Moraes, Dror and Shaw,
// "Parallel random numbers: as easy as 1, 2, 3", SC 2011), written from the
// paper's definition of the round function and key schedule.
//
// Element (b, h, query i, key j) of the attention matrix takes its random
// byte from the call with counter (i / 4, j / 4, h, b) and key = the 64-bit
// seed: output word i % 4, byte j % 4 (least significant first). It is kept
// iff the byte is >= t = round(256 p). A call thus covers a 4 x 4 block, so
// both the forward pass (a thread per query row) and the backward pass (a
// thread per key) use all sixteen bytes of every call: the four lanes that
// share a block each compute one of four calls and swap words with a
// 4 x 4 transpose through shuffles.
#pragma once

#include <stdint.h>

namespace fa {

struct DropoutArgs {
    uint32_t seed_lo, seed_hi;
    uint32_t t4;      // threshold byte replicated into the four bytes
    float inv_keep;   // 1 / (1 - t / 256)
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// 4 x 4 word transpose across the four lanes of an aligned lane quad:
// on entry lane s (s = lane % 4) holds words A[s][0..3]; on exit it holds
// A[0..3][s].
__device__ __forceinline__ uint4 quad_transpose(uint4 w, int s) {
    uint32_t a = w.x, b = w.y, c = w.z, d = w.w;
    uint32_t r = __shfl_xor_sync(0xffffffffu, (s & 1) ? a : b, 1);
    if (s & 1) a = r; else b = r;
    r = __shfl_xor_sync(0xffffffffu, (s & 1) ? c : d, 1);
    if (s & 1) c = r; else d = r;
    r = __shfl_xor_sync(0xffffffffu, (s & 2) ? a : c, 2);
    if (s & 2) a = r; else c = r;
    r = __shfl_xor_sync(0xffffffffu, (s & 2) ? b : d, 2);
    if (s & 2) b = r; else d = r;
    return make_uint4(a, b, c, d);
}

// 4 x 4 byte transpose within four words: byte k of output word n is byte n
// of input word k.
__device__ __forceinline__ uint4 byte_transpose(uint4 w) {
    const uint32_t x = __byte_perm(w.x, w.y, 0x5140), y = __byte_perm(w.z, w.w, 0x5140);
    const uint32_t x2 = __byte_perm(w.x, w.y, 0x7362), y2 = __byte_perm(w.z, w.w, 0x7362);
    return make_uint4(__byte_perm(x, y, 0x5410), __byte_perm(x, y, 0x7632), __byte_perm(x2, y2, 0x5410),
                      __byte_perm(x2, y2, 0x7632));
}

// Keep flags of the four bytes of a word (0xFF where kept, 0 where dropped)
// expanded to two 16-bit lane masks: lo for bytes 0-1, hi for bytes 2-3.
__device__ __forceinline__ void keep_masks16(uint32_t word, uint32_t t4, uint32_t& lo, uint32_t& hi) {
    const uint32_t f = __vcmpgeu4(word, t4);
    lo = __byte_perm(f, 0, 0x1100);
    hi = __byte_perm(f, 0, 0x3322);
}

}  // namespace fa

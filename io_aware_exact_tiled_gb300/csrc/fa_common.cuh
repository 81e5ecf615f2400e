// Shared definitions of the attention kernels: tile sizes, mask tests and the
// per-work-item key-tile enumeration (the tile scheduler's skip rules).
#pragma once

#include <stdint.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kTile = 128;  // query rows per Q tile == keys per K/V tile

struct MaskArgs {
    const uint8_t* blockmask;  // [T][T] or null
    const int32_t* kv_len;     // [B] or null
    int causal;
    int T;  // tiles per sequence (N / 128)
};

// Number of valid keys of batch element b (N when there is no padding).
__device__ __forceinline__ int keys_valid(const MaskArgs& m, int b, int N) {
    if (!m.kv_len) return N;
    int k = m.kv_len[b];
    return k < 0 ? 0 : (k > N ? N : k);
}

// Whether the tile (query block qb, key block kb) has any visible entry:
// causal keeps kb <= qb (tiles above the diagonal are skipped), key padding
// keeps key blocks that start below the valid length, and the tile mask keeps
// the tiles it marks.
__device__ __forceinline__ bool tile_visible(const MaskArgs& m, int qb, int kb, int kvalid) {
    if (m.causal && kb > qb) return false;
    if (kb * kTile >= kvalid) return false;
    if (m.blockmask && m.blockmask[qb * m.T + kb] == 0) return false;
    return true;
}

// Whether entries inside a visible tile still need masking.
__device__ __forceinline__ bool tile_partial(const MaskArgs& m, int qb, int kb, int kvalid) {
    return (m.causal && kb == qb) || (kb * kTile + kTile > kvalid);
}

}  // namespace fa

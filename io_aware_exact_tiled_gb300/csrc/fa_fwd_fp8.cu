// FP8 forward pass with block scales and a Hadamard rotation of Q and K.
//
// What it computes ("FlashAttention: making attention IO-aware", section
// "FlashAttention-3", FP8 with incoherent processing: FP8 doubles the tensor
// rate but is fragile with outliers, so Q and K are multiplied by a random
// orthogonal Hadamard matrix first and every block is quantised with its own
// scale):
//   1. Q' = Q diag(s) H_d and K' = K diag(s) H_d (s random signs, H_d the
//      Sylvester Hadamard matrix; diag(s) H_d / sqrt(d) is orthogonal, and
//      the 1/d this leaves in Q' K'^T is folded into the score scale);
//   2. every 128-row block of Q' and K' is divided by its own power-of-two
//      scale 2^ceil(log2(amax / 448)) and rounded to E4M3 (nearest even,
//      saturating), V likewise with one scale per head, stored transposed;
//   3. S = scale / d * 2^(e_q + e_k) * (Q8 K8^T) on the tensor cores
//      (kind::f8f6f4, fp32 accumulator in TMEM);
//   4. online softmax with an integer reference exponent m: the weights
//      p = 2^(x - m) (x = S log2 e) are rounded to E4M3 and stored four per
//      TMEM column as the A operand of O += P8 V8; the row sum l of the fp32
//      weights gives L = ln 2 (m + log2 l), the sum lw of the rounded weights
//      normalises O = 2^e_v o / lw.
// Because m is an integer and every scale a power of two, the rounded weights
// do not depend on when the running maximum was last moved: rounding to E4M3
// commutes with multiplication by powers of two (away from the subnormals).
//
// Kernels: fa_fp8_prep_kernel (persistent, three CTAs per SM walking the
// 128-row blocks of Q, K and V through double-buffered bulk copies: rotates
// and quantises the Q and K blocks and takes the maximum |v| of each V block,
// in one launch), fa_fp8_v_kernel (the head's V scale from its
// block maxima, then V quantised and transposed), fa_fwd_fp8_kernel
// (attention; two 128-row query tiles per CTA, warp 0 TMA, warp 1 MMA, two
// softmax warpgroups, as in the bf16 kernel). d = 128. Without signs (a null
// pointer) step 1 is skipped: Q and K are quantised as they are and the 1/d
// is not folded into the score scale.
#include <math_constants.h>

#include <algorithm>

#include "fa_common.cuh"
#include "fa_fp8.h"
#include "tmap.h"

namespace fa {

constexpr int kD8 = 128;               // head dimension of the FP8 path
constexpr float kE4M3Max = 448.0f;

// Exponent e of the smallest power of two with amax / 2^e <= 448 (0 for 0).
__device__ __forceinline__ int pow2_scale_exp(float amax) {
    if (!(amax > 0.f)) return 0;
    const float r = amax / kE4M3Max;
    const int bits = __float_as_int(r);
    int e = ((bits >> 23) & 0xFF) - 127;       // floor(log2 r) for normal r
    if ((bits & 0x7FFFFF) != 0) e += 1;        // not a power of two: round up
    if (((bits >> 23) & 0xFF) == 0) e = -126;  // subnormal ratio
    return max(-126, min(127, e));
}

// ---------------------------------------------------------------------------
// Q and K rotation and quantisation, V block maxima: one thread per row of a
// 128-row block. The block arrives by two tiled bulk copies in the 128-byte
// swizzled layout (16-byte chunk c of row r at chunk c ^ (r mod 8) of its
// 128-byte line), so 32 threads reading the same chunk of 32 rows touch all
// 32 banks. A row's 128 values are 64 (even, odd) column pairs, one f32x2
// register each; the Walsh-Hadamard butterflies over column bit 0 combine
// the two halves of a pair, and those over bits 1-6 combine whole pairs, two
// columns per f32x2 instruction. The seven stages commute (the Sylvester
// matrix is the Kronecker power of H_2), so their order is free, and every
// stage stays in the thread.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Persistent: each CTA walks the 128-row blocks j = blockIdx.x, + gridDim.x,
// ... of the three tensors in the order Q, K, V (V's blocks last, so that
// V is still partly in L2 when fa_fp8_v_kernel reads it again). Q and K
// blocks are rotated (when ROT), scaled and rounded to E4M3; a V block only
// gets its maximum |v| (for the head's V scale). Two shared-memory buffers:
// the block after next is requested as soon as every thread has read the
// current one into registers, so every SM keeps loads in flight while it
// computes.
constexpr int kPrepThreads = 128;
constexpr int kPrepBlockBytes = kTile * kD8 * 2;  // 128 rows of bf16
constexpr int kPrepCtasPerSm = 3;
constexpr int kPrepSmem = 2 * kPrepBlockBytes + 1024 + 64;  // two buffers, alignment, four mbarriers, abort flag

template <bool ROT>
__global__ void __launch_bounds__(kPrepThreads, kPrepCtasPerSm)
    fa_fp8_prep_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const float* __restrict__ signs,
                       uint8_t* __restrict__ q8, uint8_t* __restrict__ k8, int* __restrict__ qexp,
                       int* __restrict__ kexp, float* __restrict__ vblk_max, int N, int BH, int* status) {
    extern __shared__ __align__(1024) uint8_t prep_raw[];
    // 1024-byte aligned base: the swizzle pattern follows address bits 4-9
    uint8_t* sm = prep_raw + ((1024u - (smem_u32(prep_raw) & 1023u)) & 1023u);
    __shared__ float wmax[kPrepThreads / 32];
    __shared__ __align__(16) float sg_sh[kD8];
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + 2 * kPrepBlockBytes);  // [2] copy landed
    uint64_t* empty = full + 2;                                                 // [2] every thread has read it
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 4);
    const WaitCtx cx{abort_flag, status};
    const int T = N / kTile;
    const int per_tensor = T * BH;
    const int nblocks = 3 * per_tensor;
    const int r = threadIdx.x, warp = r >> 5, lane = r & 31;
    // block j: tensor j / per_tensor (Q, K, V), rows (j mod per_tensor) * 128 ..
    // of its [B * H * N, 128] view, as two [128 x 64] swizzled boxes
    auto request = [&](int j, int buf) {
        const int which = j / per_tensor, rem = j - which * per_tensor;
        const CUtensorMap* m = which == 0 ? &tmQ : (which == 1 ? &tmK : &tmV);
        mbar_arrive_expect_tx(&full[buf], kPrepBlockBytes);
        tma_load_2d(sm + buf * kPrepBlockBytes, m, 0, rem * kTile, &full[buf]);
        tma_load_2d(sm + buf * kPrepBlockBytes + kPrepBlockBytes / 2, m, 64, rem * kTile, &full[buf]);
    };
    if ((sm - prep_raw) + 2 * kPrepBlockBytes + 64 > kPrepSmem) {
        if (r == 0 && status) atomicCAS(status, 0, FA_DEV_TIMEOUT | (94 << 8));
        return;
    }
    if (r == 0) {
        *abort_flag = 0;
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&empty[0], kPrepThreads);
        mbar_init(&empty[1], kPrepThreads);
        fence_barrier_init();
    }
    if (ROT) sg_sh[r] = signs[r];
    __syncthreads();
    // thread 0: copies issued into each buffer, and which buffers still have
    // one outstanding (issued, not yet consumed)
    int n_issued0 = 0, n_issued1 = 0;
    uint32_t issued = 0;
    if (r == 0) {
        for (int i = 0; i < 2; ++i) {
            const int j = blockIdx.x + i * gridDim.x;
            if (j < nblocks) {
                request(j, i);
                issued |= 1u << i;
                if (i) ++n_issued1; else ++n_issued0;
            }
        }
    }
    int it = 0;
    bool refill_ok = true;
    for (int j = blockIdx.x; j < nblocks; j += gridDim.x, ++it) {
        const int buf = it & 1;
        if (!__syncthreads_and(refill_ok && mbar_wait(&full[buf], (it >> 1) & 1, cx, 31))) break;
        if (r == 0) issued &= ~(1u << buf);
        // this thread's row: 16 chunks of 8 columns (chunk c: columns 8 c ..)
        uint32_t raw[64];
        {
            const uint32_t base = smem_u32(sm + buf * kPrepBlockBytes) + r * 128;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                uint4 w;  // a shared load the compiler keeps ahead of the release below
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                             : "r"(base + (c >> 3) * (kPrepBlockBytes / 2) + (((c & 7) ^ (r & 7)) << 4))
                             : "memory");
                raw[4 * c] = w.x;
                raw[4 * c + 1] = w.y;
                raw[4 * c + 2] = w.z;
                raw[4 * c + 3] = w.w;
            }
        }
        // The refill is a bulk copy, a write by the async proxy: it may start
        // only once every thread's reads of the buffer have been performed.
        // A CTA barrier does not order them with it (the values are used only
        // after the barrier, so loads can still be in flight there, and runs
        // raced: a few rows of Q8 / K8 changed from call to call); each
        // thread's arrival on the buffer's "empty" barrier (release
        // semantics) does, and thread 0 waits for all of them and fences the
        // proxies before it requests the block after next.
        mbar_arrive(&empty[buf]);
        if (r == 0) refill_ok = mbar_wait(&empty[buf], (it >> 1) & 1, cx, 33);
        if (r == 0 && refill_ok) {
            fence_proxy_async_smem();
            const int j2 = j + 2 * gridDim.x;
            if (j2 < nblocks) {
                request(j2, buf);
                issued |= 1u << buf;
                if (buf) ++n_issued1; else ++n_issued0;
            }
        }
        const int which = j / per_tensor, rem = j - which * per_tensor;  // rem = bh * T + blk
        if (which == 2) {  // V: the block's maximum |v| only (uniform branch per CTA)
            uint32_t m2 = 0;  // two 16-bit magnitudes; bf16 magnitudes order like integers
#pragma unroll
            for (int i = 0; i < 64; ++i) m2 = __vmaxu2(m2, raw[i] & 0x7FFF7FFFu);
            float m = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (lane == 0) wmax[warp] = m;
            __syncthreads();
            if (r == 0) vblk_max[rem] = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
            continue;
        }
        // y[i]: columns 2 i and 2 i + 1 as an f32x2 pair
        uint64_t y[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) y[i] = f2_from_bf16x2(raw[i]);
        if (ROT) {
            const uint64_t* sg2 = reinterpret_cast<const uint64_t*>(sg_sh);
#pragma unroll
            for (int i = 0; i < 64; ++i) y[i] = f2_mul(y[i], sg2[i]);
            // column bit 0: the two halves of a pair
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                float a, b;
                f2_split(y[i], a, b);
                y[i] = f2_make(a + b, a - b);
            }
            // column bits 1-6: pairs i and i + M, M = 1 .. 32
#pragma unroll
            for (int M = 1; M < 64; M <<= 1)
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    if (!(i & M)) {
                        const uint64_t u = y[i], v = y[i + M];
                        y[i] = f2_add(u, v);
                        y[i + M] = f2_sub(u, v);
                    }
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            float a, b;
            f2_split(y[i], a, b);
            amax = fmax3(amax, fabsf(a), fabsf(b));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) wmax[warp] = amax;
        __syncthreads();
        // every thread takes the block's scale from the four warp maxima (the
        // next write of wmax follows the next block's first barrier)
        const int e = pow2_scale_exp(fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3])));
        if (r == 0) (which == 0 ? qexp : kexp)[rem] = e;
        const float inv = exp2i(-e);
        const uint64_t inv2 = f2_make(inv, inv);
        uint8_t* dst = (which == 0 ? q8 : k8) + (static_cast<size_t>(rem) * kTile + r) * kD8;
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 16 columns = 8 pairs per 16-byte store
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float a0, b0, a1, b1;
                f2_split(f2_mul(y[8 * c + 2 * h], inv2), a0, b0);
                f2_split(f2_mul(y[8 * c + 2 * h + 1], inv2), a1, b1);
                w[h] = pack_e4m3x2(a0, b0) | (pack_e4m3x2(a1, b1) << 16);
            }
            *reinterpret_cast<uint4*>(dst + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    // after a give-up, copies still in flight must land before the CTA exits
    if (r == 0) {
        // copies into buffer b complete its phases in order; the outstanding
        // one is the last issued there
        if (issued & 1u) mbar_wait_teardown(&full[0], (n_issued0 - 1) & 1, 200000000ull);
        if (issued & 2u) mbar_wait_teardown(&full[1], (n_issued1 - 1) & 1, 200000000ull);
    }
}

// V -> E4M3 with the head's scale, transposed to [d][keys] (the P V product
// needs K-major operands): one CTA per (128-key block, head), one warp per
// 16 of its columns. Lane l converts keys 4 l .. 4 l + 3, so a column's four
// key bytes form one 32-bit word, and the warp's 32 words of a column are
// 128 contiguous bytes of a row of V^T: one full line per store instruction,
// with no shared memory and no barrier. The prep kernel read V last, so much
// of it is still in L2.
__global__ void __launch_bounds__(256) fa_fp8_v_kernel(const uint16_t* __restrict__ v,
                                                       const float* __restrict__ vblk_max, uint8_t* __restrict__ vt8,
                                                       int* __restrict__ vexp, int N) {
    const int blk = blockIdx.x, bh = blockIdx.y;
    const int T = N / kTile;
    const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;  // columns 16 g .. 16 g + 15
    const size_t row0 = static_cast<size_t>(bh) * N + static_cast<size_t>(blk) * kTile;
    uint4 w[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint4* src = reinterpret_cast<const uint4*>(v + (row0 + 4 * lane + r) * kD8 + 16 * g);
        w[r][0] = src[0];
        w[r][1] = src[1];
    }
    // the head's max |v| from its blocks' maxima
    float hm = 0.f;
    for (int i = lane; i < T; i += 32) hm = fmaxf(hm, vblk_max[static_cast<size_t>(bh) * T + i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, off));
    const int e = pow2_scale_exp(hm);
    if (blk == 0 && threadIdx.x == 0) vexp[bh] = e;
    const float inv = exp2i(-e);
    uint8_t* dst = vt8 + (static_cast<size_t>(bh) * kD8 + 16 * g) * N + static_cast<size_t>(blk) * kTile + 4 * lane;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t u[4][4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            u[r][0] = w[r][h].x;
            u[r][1] = w[r][h].y;
            u[r][2] = w[r][h].z;
            u[r][3] = w[r][h].w;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                // column 16 g + 8 h + 2 q + half of keys 4 lane .. 4 lane + 3
                float x[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    x[r] = __uint_as_float(half ? (u[r][q] & 0xFFFF0000u) : (u[r][q] << 16)) * inv;
                *reinterpret_cast<uint32_t*>(dst + static_cast<size_t>(8 * h + 2 * q + half) * N) =
                    pack_e4m3x2(x[0], x[1]) | (pack_e4m3x2(x[2], x[3]) << 16);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Attention kernel
// ---------------------------------------------------------------------------
struct Fp8Cfg {
    static constexpr int TILE_BYTES = kTile * kD8;   // 128 rows x 128 bytes
    static constexpr int KSTAGES = 5, VSTAGES = 4;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + 2 * TILE_BYTES;
    static constexpr int V_OFF = K_OFF + KSTAGES * TILE_BYTES;
    static constexpr int BAR_OFF = V_OFF + VSTAGES * TILE_BYTES;
    static constexpr int SMEM = BAR_OFF + 512 + 1024;
    static constexpr int THREADS = 384;
    static constexpr uint32_t ID_S = idesc_make(128, 128, kFmtE4M3, false, false);
    static constexpr uint32_t ID_PV = idesc_make(128, kD8, kFmtE4M3, false, false);
    static_assert((1 + 2 * KSTAGES + 2 * VSTAGES + 9) * 8 + 8 <= 512, "barrier area");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Fp8Params {
    int B, H, N;
    float c2;  // scale * log2(e) / d
    MaskArgs mask;
    const int* qexp;  // [B*H*T] block scale exponents of Q
    const int* kexp;  // [B*H*T]
    const int* vexp;  // [B*H]
    void* o;
    float* lse;
    int* status;
};

constexpr float kFp8Rescale = 7.0f;  // log2 units: keeps every weight <= 2^7, inside E4M3

struct Fp8Mma {
    int pend_stage[2] = {-1, -1};
    uint32_t pend_ph[2] = {0, 0};
    int pend_u[2] = {0, 0};
    int nP[2] = {0, 0};
    int nPV[2] = {0, 0};
    uint32_t rem = 0;
};

// O_s += P_s V in two halves of 64 keys, the first as soon as the softmax
// warps have stored P of keys 0-63 (p_half), the second after p_full.
__device__ __forceinline__ bool fp8_issue_pv(uint32_t leader, int s, Fp8Mma& st, uint32_t tm, uint64_t dV0,
                                             uint64_t* p_half, uint64_t* p_full, uint64_t* v_full,
                                             uint64_t* kv_empty, const WaitCtx& cx) {
    using C = Fp8Cfg;
    const int ps = st.pend_stage[s];
    const uint32_t php = st.nP[s] & 1;
    if (!mbar_wait_warp(&p_half[s], php, cx, 12)) return false;
    if (!mbar_wait_warp(&v_full[ps], st.pend_ph[s], cx, 4)) return false;
    tc_fence_after();
    const uint64_t vst = sdesc_advance(dV0, ps * C::TILE_BYTES);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {  // 32 keys (8 TMEM columns of P8) per instruction
        if (kk == 2) {
            if (!mbar_wait_warp(&p_full[s], php, cx, 3)) return false;
            tc_fence_after();
        }
        umma_ts_f8(leader, tm + s * 256 + 128, tm + s * 256 + kk * 8, sdesc_advance(vst, kk * 32), C::ID_PV,
                   (st.nPV[s] > 0 || kk > 0) ? 1u : 0u);
    }
    ++st.nP[s];
    ++st.nPV[s];
    uint32_t r = (st.rem >> (2 * ps)) & 3u;
    r -= 1;
    st.rem = (st.rem & ~(3u << (2 * ps))) | (r << (2 * ps));
    if (r == 0) umma_commit(leader, &kv_empty[ps]);
    st.pend_stage[s] = -1;
    return true;
}

__global__ void __launch_bounds__(384, 1)
    fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmVt, const __grid_constant__ CUtensorMap tmO,
                      const __grid_constant__ Fp8Params p) {
    using C = Fp8Cfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    uint64_t* bar_q = bars + 0;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + C::KSTAGES;
    uint64_t* v_full = k_empty + C::KSTAGES;
    uint64_t* kv_empty = v_full + C::VSTAGES;
    uint64_t* s_full = kv_empty + C::VSTAGES;  // [2]
    uint64_t* p_full = s_full + 2;             // [2]
    uint64_t* o_done = p_full + 2;             // [2]
    uint64_t* drain = o_done + 2;
    uint64_t* p_half = drain + 1;              // [2] P of keys 0-63 stored
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_half + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const WaitCtx cx{abort_flag, p.status};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, b = blockIdx.y;
    const int T = p.mask.T;
    const int npairs = (T + 1) >> 1;
    const int qp = npairs - 1 - static_cast<int>(blockIdx.z);
    const int qb0 = 2 * qp, qb1 = 2 * qp + 1;
    const bool act1 = qb1 < T;
    const int N = p.N;
    const int bh = b * p.H + h;
    const int kvalid = keys_valid(p.mask, b, N);
    int hi = T;
    if (p.mask.causal) hi = min(hi, (act1 ? qb1 : qb0) + 1);
    hi = min(hi, (kvalid + kTile - 1) / kTile);

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int i = 0; i < C::KSTAGES; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < C::VSTAGES; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&p_half[i], 128);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
        // both Q tiles are requested before TMEM allocation and the CTA-wide
        // barrier (the producer lets them land before the CTA exits)
        mbar_arrive_expect_tx(bar_q, (act1 ? 2 : 1) * C::TILE_BYTES);
        for (int s = 0; s < (act1 ? 2 : 1); ++s)
            tma_load_2d(sm + C::Q_OFF + s * C::TILE_BYTES, &tmQ, 0, bh * N + (qb0 + s) * kTile, bar_q);
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmVt);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;
    const MaskArgs mk = p.mask;
    auto need_of = [=](int t) -> uint32_t {
        uint32_t nd = tile_visible(mk, qb0, t, kvalid) ? 1u : 0u;
        if (act1 && tile_visible(mk, qb1, t, kvalid)) nd |= 2u;
        return nd;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int nk = 0, nv = 0;
            for (int t = 0; t < hi; ++t) {
                if (!need_of(t)) continue;
                const int kst = nk % C::KSTAGES;
                if (!mbar_wait(&k_empty[kst], ((nk / C::KSTAGES) & 1) ^ 1, cx, 1)) break;
                mbar_arrive_expect_tx(&k_full[kst], C::TILE_BYTES);
                tma_load_2d(sm + C::K_OFF + kst * C::TILE_BYTES, &tmK, 0, bh * N + t * kTile, &k_full[kst]);
                ++nk;
                const int vst = nv % C::VSTAGES;
                if (!mbar_wait(&kv_empty[vst], ((nv / C::VSTAGES) & 1) ^ 1, cx, 9)) break;
                mbar_arrive_expect_tx(&v_full[vst], C::TILE_BYTES);
                // V^T [d][keys]: 128 rows of d, 128 keys of this tile
                tma_load_2d(sm + C::V_OFF + vst * C::TILE_BYTES, &tmVt, t * kTile, bh * kD8, &v_full[vst]);
                ++nv;
            }
            mbar_wait_teardown(bar_q, 0, 200000000ull);
            for (int i = 0; i < C::KSTAGES && i < nk; ++i) {
                const int last = i + ((nk - 1 - i) / C::KSTAGES) * C::KSTAGES;
                mbar_wait_teardown(&k_full[i], (last / C::KSTAGES) & 1, 200000000ull);
            }
            for (int i = 0; i < C::VSTAGES && i < nv; ++i) {
                const int last = i + ((nv - 1 - i) / C::VSTAGES) * C::VSTAGES;
                mbar_wait_teardown(&v_full[i], (last / C::VSTAGES) & 1, 200000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (whole warp, one lane issues)
        const uint32_t leader = elect_one_sync();
        bool ok = mbar_wait_warp(bar_q, 0, cx, 2);
        if (ok) tc_fence_after();
        Fp8Mma st;
        const uint64_t dQ0 = sdesc_sw128(smem_u32(sm + C::Q_OFF), 16, 1024);
        const uint64_t dK0 = sdesc_sw128(smem_u32(sm + C::K_OFF), 16, 1024);
        const uint64_t dV0 = sdesc_sw128(smem_u32(sm + C::V_OFF), 16, 1024);
#define issue_pv8(S) fp8_issue_pv(leader, (S), st, tm, dV0, p_half, p_full, v_full, kv_empty, cx)
        int u = 0;
        for (int t = 0; ok && t < hi; ++t) {
            const uint32_t nd = need_of(t);
            if (!nd) continue;
            const int kst = u % C::KSTAGES;
            const int vst = u % C::VSTAGES;
            const uint32_t vph = (u / C::VSTAGES) & 1;
            // a P V still pending for a tile as old as u - VSTAGES holds the V
            // stage (and its reader count) that tile u reuses: issue it first
#pragma unroll
            for (int s = 0; s < 2; ++s)
                if (ok && st.pend_stage[s] >= 0 && st.pend_u[s] <= u - C::VSTAGES && !issue_pv8(s)) ok = false;
            if (!ok) break;
            if (!mbar_wait_warp(&k_full[kst], (u / C::KSTAGES) & 1, cx, 5)) { ok = false; break; }
            tc_fence_after();
            st.rem = (st.rem & ~(3u << (2 * vst))) | ((uint32_t)__popc(nd) << (2 * vst));
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                if (!(nd & (1u << s))) continue;
                if (st.pend_stage[s] >= 0 && !issue_pv8(s)) { ok = false; break; }
                const uint64_t qs = sdesc_advance(dQ0, s * C::TILE_BYTES);
                const uint64_t ks = sdesc_advance(dK0, kst * C::TILE_BYTES);
#pragma unroll
                for (int kk = 0; kk < kD8 / 32; ++kk)  // 32 bytes of K per instruction
                    umma_ss_f8(leader, tm + s * 256, sdesc_advance(qs, kk * 32), sdesc_advance(ks, kk * 32), C::ID_S,
                               kk > 0 ? 1u : 0u);
                umma_commit(leader, &s_full[s]);
                st.pend_stage[s] = vst;
                st.pend_ph[s] = vph;
                st.pend_u[s] = u;
            }
            if (!ok) break;
            umma_commit(leader, &k_empty[kst]);
            ++u;
        }
        for (int s = 0; ok && s < 2; ++s)
            if (st.pend_stage[s] >= 0 && !issue_pv8(s)) ok = false;
#undef issue_pv8
        if (ok) {
            umma_commit(leader, &o_done[0]);
            umma_commit(leader, &o_done[1]);
        }
        umma_commit(leader, drain);
        mbar_wait_teardown(drain, 0, 200000000ull);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax (thread = query row)
        const int s = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const bool active = (s == 0) || act1;
        const int qb = s == 0 ? qb0 : qb1;
        const int grow = qb * kTile + r;
        const uint32_t tl = tm + (static_cast<uint32_t>(wq * 32) << 16) + s * 256;
        const int T_ = p.mask.T;
        const int eq = p.qexp[static_cast<size_t>(bh) * T_ + min(qb, T_ - 1)];
        // m: integer reference exponent (log2 units); l: fp32 weights; lw: E4M3 weights
        float m_hat = -CUDART_INF_F, l = 0.f, lw = 0.f;
        int n = 0;
        bool ok = true;
        if (active) {
            for (int t = 0; t < hi; ++t) {
                const uint32_t nd = need_of(t);
                if (!(nd & (1u << s))) continue;
                const float c2t = p.c2 * exp2i(eq + p.kexp[static_cast<size_t>(bh) * T_ + t]);
                ok = mbar_wait(&s_full[s], n & 1, cx, 6);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tl + c * 32, sr[c]);
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
                if (tile_partial(p.mask, qb, t, kvalid)) {
                    const int lim = min(kvalid - t * kTile, p.mask.causal && t == qb ? r + 1 : kTile);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c * 32 + i >= lim) sr[c][i] = __float_as_uint(-CUDART_INF_F);
                }
                // row maximum as eight independent chains (one dependent chain
                // of 64 three-input maxima would sit on the softmax's
                // critical path), combined at the end
                float mc[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mc[k] = -CUDART_INF_F;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const int k = 2 * c + ((i >> 2) & 1);
                        mc[k] = fmax3(mc[k], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
                        mc[k] = fmax3(mc[k], __uint_as_float(sr[c][i + 2]), __uint_as_float(sr[c][i + 3]));
                    }
                const float mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), fmaxf(fmax3(mc[3], mc[4], mc[5]), fmax3(mc[6], mc[7], mc[7])));
                const float xmax = mx * c2t;
                float alpha = 1.f;
                bool resc = false;
                if (xmax > -CUDART_INF_F && (m_hat == -CUDART_INF_F || xmax - m_hat > kFp8Rescale)) {
                    const float m_new = floorf(xmax);
                    const float dm = m_hat - m_new;  // an integer <= 0
                    alpha = (m_hat == -CUDART_INF_F || dm < -126.f) ? 0.f : exp2i(static_cast<int>(dm));
                    m_hat = m_new;
                    l *= alpha;
                    lw *= alpha;
                    resc = true;
                }
                const float mu = (m_hat == -CUDART_INF_F) ? 0.f : m_hat;
                const uint64_t cc = f2_make(c2t, c2t), nmu2 = f2_make(-mu, -mu);
                uint64_t rs2 = 0ull, rr2 = 0ull;
                // O is rescaled (below) before any P V of this tile may run
                const bool resc_any = __any_sync(0xffffffffu, resc) && n > 0;
                uint32_t pk[2][16];  // keys 0-63 and 64-127, four E4M3 weights per word
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float x0, x1, x2, x3;
                        f2_split(f2_fma(f2_make(__uint_as_float(sr[c][4 * i]), __uint_as_float(sr[c][4 * i + 1])), cc,
                                        nmu2), x0, x1);
                        f2_split(f2_fma(f2_make(__uint_as_float(sr[c][4 * i + 2]), __uint_as_float(sr[c][4 * i + 3])),
                                        cc, nmu2), x2, x3);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
                        rs2 = f2_add(rs2, f2_add(f2_make(p0, p1), f2_make(p2, p3)));
                        const uint32_t lo = pack_e4m3x2(p0, p1), hi2 = pack_e4m3x2(p2, p3);
                        pk[c >> 1][(c & 1) * 8 + i] = lo | (hi2 << 16);
                        rr2 = f2_add(rr2, f2_add(f2_from_e4m3x2(lo), f2_from_e4m3x2(hi2)));
                    }
                    if (c == 1) {
                        tmem_st16(tl, pk[0]);
                        if (!resc_any) {
                            tmem_st_wait();
                            tc_fence_before();
                            mbar_arrive(&p_half[s]);
                        }
                    }
                }
                tmem_st16(tl + 16, pk[1]);
                {
                    float a_, b_;
                    f2_split(rs2, a_, b_);
                    l += a_ + b_;
                    f2_split(rr2, a_, b_);
                    lw += a_ + b_;
                }
                tmem_st_wait();
                if (resc_any) {
                    // O holds the previous tiles' sum (their P V was issued
                    // before this tile's S): bring it to the new reference
#pragma unroll
                    for (int c = 0; c < kD8 / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(tl + 128 + c * 32, ov);
                        tmem_ld_wait(ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st32(tl + 128 + c * 32, ov);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                if (resc_any) mbar_arrive(&p_half[s]);
                if (!FA_DROP_THIS_ARRIVE(n == 0)) mbar_arrive(&p_full[s]);
                ++n;
            }
            // ------------------------------------------------------------ epilogue
            if (ok && n > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(&o_done[s], 0, cx, 8));
                if (ok) tc_fence_after();
            }
            if (ok) {
                const float inv = lw > 0.f ? exp2i(p.vexp[bh]) / lw : 0.f;
                const size_t orow = (static_cast<size_t>(bh) * N + grow) * kD8;
                // A warp whose query tile saw a key tile stages its 32 rows,
                // as [32 x 64] swizzled bf16 boxes, in two stages of the K
                // ring (free once o_done has landed: every GEMM is complete)
                // and writes them with bulk tensor stores; a tile that saw no
                // key tile stores its (zero) rows directly.
                const bool tma_rows = n > 0;
                uint8_t* ob = sm + C::K_OFF + s * 2 * C::TILE_BYTES + wq * 8192;
                uint32_t oa[kD8 / 32][32];
                if (n > 0) {
#pragma unroll
                    for (int c = 0; c < kD8 / 32; ++c) tmem_ld32(tl + 128 + c * 32, oa[c]);
#pragma unroll
                    for (int c = 0; c < kD8 / 32; ++c) tmem_ld_wait(oa[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < kD8 / 32; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i) oa[c][i] = 0u;
                }
#pragma unroll
                for (int c = 0; c < kD8 / 32; ++c) {
                    const uint32_t* ov = oa[c];
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow + c * 32);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(ov[8 * j + 0]) * inv, __uint_as_float(ov[8 * j + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(ov[8 * j + 2]) * inv, __uint_as_float(ov[8 * j + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(ov[8 * j + 4]) * inv, __uint_as_float(ov[8 * j + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(ov[8 * j + 6]) * inv, __uint_as_float(ov[8 * j + 7]) * inv);
                        if (tma_rows) {
                            const int ch = ((c & 1) << 2) + j;  // 16-byte chunk within the 128-byte row
                            sts128(smem_u32(ob + (c >> 1) * 4096 + lane * 128 + ((ch ^ (lane & 7)) << 4)), w.x, w.y,
                                   w.z, w.w);
                        } else {
                            dst[j] = w;
                        }
                    }
                }
                if (tma_rows) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int wrow = bh * N + qb * kTile + wq * 32;
                        tma_store_2d(&tmO, 0, wrow, ob);
                        tma_store_2d(&tmO, 64, wrow, ob + 4096);
                        bulk_commit_group();
                        bulk_wait_group_read0();  // read out before the CTA exits
                    }
                }
                p.lse[static_cast<size_t>(bh) * N + grow] =
                    l > 0.f ? (m_hat + log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

cudaError_t launch_fwd_fp8(const Fp8Args& a, cudaStream_t stream, int* nlaunch) {
    using C = Fp8Cfg;
    const int T = a.N / kTile;
    const int BH = a.B * a.H;
    const uint64_t rows = static_cast<uint64_t>(BH) * a.N;
    // quantisation: Q, K and the V block maxima in one persistent launch, then V
    static int nsm = 0;
    static bool prep_attr = false;
    if (nsm == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0)
            return cudaErrorUnknown;
    }
    if (!prep_attr) {
        cudaError_t e0 = cudaFuncSetAttribute(fa_fp8_prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              kPrepSmem);
        if (e0 == cudaSuccess)
            e0 = cudaFuncSetAttribute(fa_fp8_prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      kPrepSmem);
        if (e0 != cudaSuccess) return e0;
        prep_attr = true;
    }
    const long long nblocks = 3LL * T * BH;
    const unsigned pgrid = static_cast<unsigned>(std::min<long long>(nblocks, static_cast<long long>(nsm) * kPrepCtasPerSm));
    CUtensorMap tq16, tk16, tv16;
    if (!make_tmap_2d_sw128(&tq16, a.q, rows, kD8, 2, kTile, 64) || !make_tmap_2d_sw128(&tk16, a.k, rows, kD8, 2, kTile, 64) ||
        !make_tmap_2d_sw128(&tv16, a.v, rows, kD8, 2, kTile, 64))
        return cudaErrorInvalidValue;
    const uint16_t* v16 = static_cast<const uint16_t*>(a.v);
    if (a.signs)
        fa_fp8_prep_kernel<true><<<pgrid, kPrepThreads, kPrepSmem, stream>>>(
            tq16, tk16, tv16, a.signs, a.q8, a.k8, a.qexp, a.kexp, a.vblk_max, a.N, BH, a.status);
    else
        fa_fp8_prep_kernel<false><<<pgrid, kPrepThreads, kPrepSmem, stream>>>(
            tq16, tk16, tv16, nullptr, a.q8, a.k8, a.qexp, a.kexp, a.vblk_max, a.N, BH, a.status);
    fa_fp8_v_kernel<<<dim3(T, BH), 256, 0, stream>>>(v16, a.vblk_max, a.vt8, a.vexp, a.N);
    cudaError_t e;
    CUtensorMap tq, tk, tv, to;
    if (!make_tmap_2d_sw128(&to, a.o, rows, kD8, 2, 32, 64) ||
        !make_tmap_2d_sw128(&tq, a.q8, rows, kD8, 1, kTile, 128) ||
        !make_tmap_2d_sw128(&tk, a.k8, rows, kD8, 1, kTile, 128) ||
        !make_tmap_2d_sw128(&tv, a.vt8, static_cast<uint64_t>(BH) * kD8, a.N, 1, kD8, 128))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        e = cudaFuncSetAttribute(fa_fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    Fp8Params p;
    p.B = a.B;
    p.H = a.H;
    p.N = a.N;
    // the rotation leaves a factor d in Q' K'^T (diag(s) H_d is sqrt(d) times an orthogonal matrix)
    p.c2 = a.scale * 1.4426950408889634f / (a.signs ? static_cast<float>(kD8) : 1.f);
    p.mask.blockmask = nullptr;
    p.mask.kv_len = a.kv_len;
    p.mask.causal = a.causal;
    p.mask.T = T;
    p.qexp = a.qexp;
    p.kexp = a.kexp;
    p.vexp = a.vexp;
    p.o = a.o;
    p.lse = a.lse;
    p.status = a.status;
    dim3 grid(a.H, a.B, (T + 1) / 2);
    if (a.ev_begin) cudaEventRecord(a.ev_begin, stream);
    fa_fwd_fp8_kernel<<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, to, p);
    if (a.ev_end) cudaEventRecord(a.ev_end, stream);
    *nlaunch = 3;
    return cudaGetLastError();
}

}  // namespace fa

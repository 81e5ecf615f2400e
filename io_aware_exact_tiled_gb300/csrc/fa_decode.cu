// Decoding: a few query rows against a long key/value cache, split over the
// keys (Flash-Decoding).
//
// What it computes ("FlashAttention: making attention IO-aware", section "In
// practice", the note on decoding; "Why is FlashAttention faster?", section
// "FlashAttention is not KV-cache compression"): for each (batch, head),
// O = softmax(scale * q K^T) V over the cache_len[b] valid keys, and
// L = m + log l per query row. With one query row there are no query blocks
// to spread over the GPU, so the keys are: split c of a head takes a run of
// consecutive keys and produces the partial maximum m_c, sum l_c of
// exp(s - m_c) and unnormalised output o_c; a second kernel merges the
// splits with the logsumexp rescaling of the online softmax,
//   M = max m_c, l = sum exp(m_c - M) l_c, O = sum exp(m_c - M) o_c / l,
//   L = M + log l.
//
// GB300 design: the step reads every valid cache byte once and does about
// one flop per byte, so it is bound by HBM bandwidth, not by arithmetic; it
// runs on the CUDA cores (a 1-row product would waste 127/128 of a tensor-
// core tile) and is built to keep enough bytes in flight:
//   * 64-key K and V tiles come through a 3-stage TMA ring (128-byte
//     swizzle); with about 100 KB of shared memory two CTAs share an SM;
//   * scores: thread (key j, half h) dots its half of k_j with every query
//     (q held in shared memory as fp32, read as broadcasts), the two halves
//     combine through one shuffle;
//   * softmax: warp w keeps the running maximum and sum of queries w and
//     w + 4 (exp2 of pre-scaled scores);
//   * P V: thread (8-column chunk, key group) accumulates fp32 partial
//     outputs over its keys; the key groups are summed once at the end.
// The swizzle makes both the row-per-thread reads of K and the
// column-per-thread reads of V free of shared-memory bank conflicts.
#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_decode.h"
#include "tmap.h"

namespace fa {

template <int D, int NQ>
struct DecCfg {
    static constexpr int KT = 64;                      // keys per tile
    static constexpr int STAGES = D == 64 ? 6 : 3;
    static constexpr int NREG = D / 64;                // 128-byte regions per row
    static constexpr int TILE_BYTES = KT * D * 2;      // one bf16 K or V tile
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
    static constexpr int QS_OFF = V_OFF + STAGES * TILE_BYTES;  // fp32 [NQ][D]
    static constexpr int PS_OFF = QS_OFF + NQ * D * 4;          // fp32 [NQ][KT]
    static constexpr int AL_OFF = PS_OFF + NQ * KT * 4;         // fp32 [NQ] rescale factors
    static constexpr int BAR_OFF = AL_OFF + 64;
    static constexpr int USED = BAR_OFF + 8 * STAGES + 64;
    static constexpr int SMEM = USED + 1024;
    static constexpr int THREADS = 128;
    static constexpr int CHUNKS = D / 8;               // 16-byte chunks per row
    static constexpr int GROUPS = THREADS / CHUNKS;    // key groups of the P V step
    static constexpr int KG = KT / GROUPS;             // keys per group per tile
    // the end-of-split reduction of the key groups reuses the ring
    static_assert(GROUPS * NQ * D * 4 <= 2 * STAGES * TILE_BYTES, "reduction buffer");
    static_assert(NQ <= 8, "at most two queries per softmax warp");
};

// Byte offset of 16-byte chunk `c` (0 .. D/8 - 1) of row `r` in a tile stored
// as NREG regions of [KT rows x 128 bytes] with the 128-byte swizzle.
template <int D>
__device__ __forceinline__ uint32_t dec_chunk_off(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * (64 * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void bf16x8_to_f32(uint4 w, float (&f)[8]) {
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xFFFF0000u);
    f[4] = __uint_as_float(w.z << 16);
    f[5] = __uint_as_float(w.z & 0xFFFF0000u);
    f[6] = __uint_as_float(w.w << 16);
    f[7] = __uint_as_float(w.w & 0xFFFF0000u);
}

template <int D, int NQ>
__global__ void __launch_bounds__(128) fa_decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                                                              const __grid_constant__ CUtensorMap tmV,
                                                              const __grid_constant__ DecodeParams p) {
    using C = DecCfg<D, NQ>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int bh = b * p.H + h;
    int len = p.Nk;
    if (p.cache_len) len = min(max(p.cache_len[b], 0), p.Nk);
    const int k0 = c * p.split;
    const int k1 = min(k0 + p.split, len);
    const int ntiles = k1 > k0 ? (k1 - k0 + C::KT - 1) / C::KT : 0;
    // partial results: m, l [B,H,Nq,S]; o [B,H,Nq,S,D]
    const size_t prow = (static_cast<size_t>(bh) * p.Nq) * p.S;
    if (ntiles == 0) {
        // no valid key in this split: a neutral partial (m = -inf, l = 0, o = 0)
        for (int i = tid; i < p.Nq * D; i += C::THREADS) {
            const int qi = i / D, dd = i % D;
            p.po[((prow + static_cast<size_t>(qi) * p.S + c) * D) + dd] = 0.f;
        }
        if (tid < p.Nq) {
            p.pm[prow + static_cast<size_t>(tid) * p.S + c] = -CUDART_INF_F;
            p.pl[prow + static_cast<size_t>(tid) * p.S + c] = 0.f;
        }
        return;
    }
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(full + C::STAGES);
    const WaitCtx cx{abort_flag, p.status};
    float* qs = reinterpret_cast<float*>(sm + C::QS_OFF);
    float* ps = reinterpret_cast<float*>(sm + C::PS_OFF);
    float* al = reinterpret_cast<float*>(sm + C::AL_OFF);
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < C::STAGES; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    // queries as fp32 (rows past Nq are zero and never read back)
    const uint16_t* q = static_cast<const uint16_t*>(p.q) + static_cast<size_t>(bh) * p.Nq * D;
    for (int i = tid; i < NQ * D; i += C::THREADS)
        qs[i] = i < p.Nq * D ? __uint_as_float(static_cast<uint32_t>(q[i]) << 16) : 0.f;
    __syncthreads();
    const int row0 = bh * p.Nk + k0;  // first cache row of this split
    auto issue = [&](int t) {
        const int st = t % C::STAGES;
        mbar_arrive_expect_tx(&full[st], 2 * C::TILE_BYTES);
        for (int r = 0; r < C::NREG; ++r) {
            tma_load_2d(sm + C::K_OFF + st * C::TILE_BYTES + r * (C::KT * 128), &tmK, r * 64, row0 + t * C::KT,
                        &full[st]);
            tma_load_2d(sm + C::V_OFF + st * C::TILE_BYTES + r * (C::KT * 128), &tmV, r * 64, row0 + t * C::KT,
                        &full[st]);
        }
    };
    if (tid == 0)
        for (int t = 0; t < C::STAGES && t < ntiles; ++t) issue(t);

    // running softmax state of queries warp and warp + 4 (replicated in the lanes)
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F}, l_run[2] = {0.f, 0.f};
    // P V partials: thread (chunk cc, key group g)
    const int cc = tid % C::CHUNKS, g = tid / C::CHUNKS;
    float o[NQ][8];
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
        for (int e = 0; e < 8; ++e) o[qi][e] = 0.f;
    // scores: thread (key j, half hf)
    const int j = tid >> 1, hf = tid & 1;
    bool ok = true;
    int t = 0;
    for (; t < ntiles; ++t) {
        const int st = t % C::STAGES;
        ok = mbar_wait(&full[st], (t / C::STAGES) & 1, cx, 60);
        if (__syncthreads_or(!ok)) { ok = false; break; }
        const uint32_t kb = smem_u32(sm + C::K_OFF + st * C::TILE_BYTES);
        const uint32_t vb = smem_u32(sm + C::V_OFF + st * C::TILE_BYTES);
        // ---- scores of key j against every query
        float s[NQ];
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) s[qi] = 0.f;
#pragma unroll
        for (int ci = 0; ci < C::CHUNKS / 2; ++ci) {
            const int ch = hf * (C::CHUNKS / 2) + ci;
            const uint4 w = lds128_u4(kb + dec_chunk_off<D>(j, ch));
            float kf[8];
            bf16x8_to_f32(w, kf);
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                const float4 qa = *reinterpret_cast<const float4*>(qs + qi * D + ch * 8);
                const float4 qb = *reinterpret_cast<const float4*>(qs + qi * D + ch * 8 + 4);
                s[qi] = fmaf(kf[0], qa.x, s[qi]);
                s[qi] = fmaf(kf[1], qa.y, s[qi]);
                s[qi] = fmaf(kf[2], qa.z, s[qi]);
                s[qi] = fmaf(kf[3], qa.w, s[qi]);
                s[qi] = fmaf(kf[4], qb.x, s[qi]);
                s[qi] = fmaf(kf[5], qb.y, s[qi]);
                s[qi] = fmaf(kf[6], qb.z, s[qi]);
                s[qi] = fmaf(kf[7], qb.w, s[qi]);
            }
        }
        const bool valid = k0 + t * C::KT + j < k1;
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            s[qi] += __shfl_xor_sync(0xffffffffu, s[qi], 1);
            if (hf == 0) ps[qi * C::KT + j] = valid ? s[qi] * p.scale_log2 : -CUDART_INF_F;
        }
        __syncthreads();
        // ---- online softmax: warp w owns queries w and w + 4
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int qi = warp + 4 * k;
            if (qi >= NQ || qi >= p.Nq) continue;
            const float a0 = ps[qi * C::KT + lane], a1 = ps[qi * C::KT + 32 + lane];
            float mx = fmaxf(a0, a1);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m_run[k], mx);  // finite: every tile holds a valid key
            const float alpha = ex2_approx(m_run[k] - m_new);
            const float e0 = ex2_approx(a0 - m_new), e1 = ex2_approx(a1 - m_new);
            ps[qi * C::KT + lane] = e0;
            ps[qi * C::KT + 32 + lane] = e1;
            float sum = e0 + e1;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            l_run[k] = l_run[k] * alpha + sum;
            m_run[k] = m_new;
            if (lane == 0) al[qi] = alpha;
        }
        __syncthreads();
        // ---- O += P V over this thread's keys and columns
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
            const float a = al[qi];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[qi][e] *= a;
        }
#pragma unroll
        for (int i = 0; i < C::KG; ++i) {
            const int jj = g * C::KG + i;
            const uint4 w = lds128_u4(vb + dec_chunk_off<D>(jj, cc));
            float vf[8];
            bf16x8_to_f32(w, vf);
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
                const float pj = ps[qi * C::KT + jj];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[qi][e] = fmaf(pj, vf[e], o[qi][e]);
            }
        }
        __syncthreads();  // stage st and the score buffer are free again
        if (tid == 0 && t + C::STAGES < ntiles) issue(t + C::STAGES);
    }
    if (!ok) {
        // a wait gave up: let the copies still in flight land before leaving
        if (tid == 0)
            for (int u = t; u < ntiles && u < t + C::STAGES; ++u)
                mbar_wait_teardown(&full[u % C::STAGES], (u / C::STAGES) & 1, 200000000ull);
        return;
    }
    // ---- sum the key groups' partial outputs (through the now idle ring)
    float* red = reinterpret_cast<float*>(sm + C::K_OFF);  // [GROUPS][NQ][D]
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi)
#pragma unroll
        for (int e = 0; e < 8; ++e) red[(g * NQ + qi) * D + cc * 8 + e] = o[qi][e];
    __syncthreads();
    for (int i = tid; i < p.Nq * D; i += C::THREADS) {
        const int qi = i / D, dd = i % D;
        float acc = 0.f;
#pragma unroll
        for (int gg = 0; gg < C::GROUPS; ++gg) acc += red[(gg * NQ + qi) * D + dd];
        p.po[((prow + static_cast<size_t>(qi) * p.S + c) * D) + dd] = acc;
    }
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int qi = warp + 4 * k;
            if (qi < NQ && qi < p.Nq) {
                p.pm[prow + static_cast<size_t>(qi) * p.S + c] = m_run[k];  // log2 units, scale applied
                p.pl[prow + static_cast<size_t>(qi) * p.S + c] = l_run[k];
            }
        }
    }
}

// Merge of the splits of one query row: thread = output column.
template <int D>
__global__ void __launch_bounds__(D) fa_decode_merge_kernel(const __grid_constant__ DecodeParams p) {
    const size_t row = blockIdx.x;  // (b * H + h) * Nq + qi
    const int dd = threadIdx.x;
    const float* pm = p.pm + row * p.S;
    const float* pl = p.pl + row * p.S;
    const float* po = p.po + row * p.S * D;
    float M = -CUDART_INF_F;
    for (int c = 0; c < p.S; ++c) M = fmaxf(M, pm[c]);
    const float shift = M == -CUDART_INF_F ? 0.f : M;
    float l = 0.f, acc = 0.f;
    for (int c = 0; c < p.S; ++c) {
        const float w = ex2_approx(pm[c] - shift);  // 0 for an empty split
        l = fmaf(w, pl[c], l);
        acc = fmaf(w, po[static_cast<size_t>(c) * D + dd], acc);
    }
    const float out = l > 0.f ? acc / l : 0.f;
    static_cast<uint16_t*>(p.o)[row * D + dd] = static_cast<uint16_t>(pack_bf16x2(out, 0.f) & 0xFFFFu);
    if (dd == 0)
        p.lse[row] = l > 0.f ? (shift + log2f(l)) * 0.69314718055994530942f : -CUDART_INF_F;
}

template <int D, int NQ>
static cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t stream, int* nlaunch) {
    using C = DecCfg<D, NQ>;
    const uint64_t rows = static_cast<uint64_t>(a.B) * a.H * a.Nk;
    CUtensorMap tk, tv;
    if (!make_tmap_2d_sw128(&tk, a.k, rows, D, 2, C::KT, 64) || !make_tmap_2d_sw128(&tv, a.v, rows, D, 2, C::KT, 64))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(fa_decode_split_kernel<D, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    DecodeParams p;
    p.q = a.q;
    p.o = a.o;
    p.lse = a.lse;
    p.cache_len = a.cache_len;
    p.B = a.B;
    p.H = a.H;
    p.Nq = a.Nq;
    p.Nk = a.Nk;
    p.S = a.splits;
    p.split = a.split_keys;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.pm = a.pm;
    p.pl = a.pl;
    p.po = a.po;
    p.status = a.status;
    dim3 grid(a.splits, a.H, a.B);
    if (a.ev_begin) cudaEventRecord(a.ev_begin, stream);
    fa_decode_split_kernel<D, NQ><<<grid, C::THREADS, C::SMEM, stream>>>(tk, tv, p);
    if (a.ev_end) cudaEventRecord(a.ev_end, stream);
    fa_decode_merge_kernel<D><<<static_cast<unsigned>(static_cast<size_t>(a.B) * a.H * a.Nq), D, 0, stream>>>(p);
    *nlaunch = 2;
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t stream, int* nlaunch) {
    if (a.Nq == 1) return launch_decode_t<D, 1>(a, stream, nlaunch);
    if (a.Nq == 2) return launch_decode_t<D, 2>(a, stream, nlaunch);
    if (a.Nq <= 4) return launch_decode_t<D, 4>(a, stream, nlaunch);
    return launch_decode_t<D, 8>(a, stream, nlaunch);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream, int* nlaunch) {
    if (a.d == 64) return launch_decode_d<64>(a, stream, nlaunch);
    return launch_decode_d<128>(a, stream, nlaunch);
}

}  // namespace fa

// Forward pass for bf16 inputs: one 128-row query tile per CTA.
//
// Same computation as fa_fwd.cu ("FlashAttention: making attention
// IO-aware", sections "Tiling: never materialise S" and "Online softmax"):
// stream the key/value tiles the masks keep, form S = scale * Q K^T on the
// tensor cores, keep the running maximum m, the running sum l of exp(S - m)
// and the unnormalised output o, rescale o and l by exp(m_old - m_new) when
// the maximum grows, and write O = o / l and L = m + log l at the end.
//
// Layout of the work on one SM (384 threads):
//   thread 0    sets up the mbarriers and requests the Q tile
//   warp 0      TMA producer: K and V tiles through a ring of STAGES (>= 3)
//               shared-memory stages, one mbarrier per stage
//   warp 1      TMEM allocation; the whole warp runs the issue loop and one
//               elected lane issues all MMAs
//   warps 2-3   turn the mask row into a bitmap (tile-masked calls)
//   warps 4-7   softmax group 0: thread r owns row r, key columns 0-63
//   warps 8-11  softmax group 1: row r, key columns 64-127
// TMEM: two S buffers (columns 0-127 and 128-255, so that S for tile u+2 is
// computed while tile u's probabilities are produced) and the O accumulator
// (columns 256 .. 256+d). P (bf16) overwrites S in place: group 0 writes its
// 64 keys to the buffer's columns 0-31, group 1 to columns 64-95, so neither
// overwrites scores the other has not read yet.
// The two groups agree on the row maximum through a small shared-memory
// exchange each tile; each keeps partial row sums, which are added at the end.
// The running maximum is only moved (and O rescaled) when it grows by more
// than 2^8 in the exp2 domain (exact: o and l always share the reference).
#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_launch.h"
#include "tmap.h"

namespace fa {

template <int D>
struct Q1Cfg {
    static constexpr int TILE_BYTES = kTile * D * 2;  // one 128-row bf16 tile
    static constexpr int NREG = D / 64;               // 128-byte swizzle regions per row
    static constexpr int STAGES = D == 64 ? 6 : 3;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + TILE_BYTES;
    static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
    static constexpr int X_OFF = V_OFF + STAGES * TILE_BYTES;  // [2 parities][2 groups][128] fp32
    static constexpr int BAR_OFF = X_OFF + 2048;
    // visible key tiles of the query tile as a bitmap (tile-masked calls);
    // longer rows than it holds read the mask tile by tile
    static constexpr int VIS_OFF = BAR_OFF + 256;
    static constexpr int VIS_WORDS = (D == 64 ? 4096 : 1024) / 32;
    static constexpr int USED = VIS_OFF + VIS_WORDS * 4;
    static constexpr int SMEM = USED + 1024 <= 232448 ? USED + 1024 : 232448;
    static constexpr int COL_O = 256;
    static constexpr uint32_t ID_S = idesc_make(128, 128, kFmtBF16, false, false);
    static constexpr uint32_t ID_PV = idesc_make(128, D, kFmtBF16, false, true);
};

struct Q1Params {
    int B, H, N;
    float scale_log2;
    MaskArgs mask;
    void* o;
    float* lse;
    int* status;
};

constexpr float kQ1RescaleThreshold = 8.0f;  // log2 units
constexpr float kQ1Ln2 = 0.69314718055994530942f;

template <int D>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_q1_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ Q1Params p) {
    using C = Q1Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, kept in the shared address space
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((sm - smem_raw) + C::USED > C::SMEM) {
        if (tid == 0 && p.status) atomicCAS(p.status, 0, FA_DEV_TIMEOUT | (98 << 8));
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    uint64_t* bar_q = bars;
    uint64_t* kv_full = bars + 1;               // [STAGES]
    uint64_t* kv_empty = kv_full + C::STAGES;   // [STAGES]
    uint64_t* s_full = kv_empty + C::STAGES;    // [2] S buffer computed
    uint64_t* p_full = s_full + 2;              // [2] P written (both groups)
    uint64_t* xch = p_full + 2;                 // [2] row-max exchange, by tile parity
    uint64_t* sum_x = xch + 2;                  // final row-sum exchange
    uint64_t* o_done = sum_x + 1;               // every P V complete
    uint64_t* drain = o_done + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const WaitCtx cx{abort_flag, p.status};

    // Causal: longest rows first across all heads (grid (H, B, T)). Otherwise
    // the work per query tile is even and the grid is head-major (T, H, B),
    // so that the CTAs running together share one head's K and V in L2.
    const int T = p.mask.T;
    const bool lpt = p.mask.causal != 0;
    const int h = lpt ? blockIdx.x : blockIdx.y, b = lpt ? blockIdx.y : blockIdx.z;
    const int qb = lpt ? T - 1 - static_cast<int>(blockIdx.z) : static_cast<int>(blockIdx.x);
    const int N = p.N;
    const int bh = b * p.H + h;
    const MaskArgs mk = p.mask;
    const int kvalid = keys_valid(mk, b, N);
    int hi = mk.causal ? min(T, qb + 1) : T;
    hi = min(hi, (kvalid + kTile - 1) / kTile);
    // With a tile mask, warps 2 and 3 (otherwise idle) first turn the mask
    // row into a bitmap in shared memory: counting the visible tiles and
    // finding the next one then take a popcount and a find-first-set instead
    // of a dependent load of the mask per tile in every role.
    const bool use_vis = mk.blockmask != nullptr && hi <= C::VIS_WORDS * 32;
    uint32_t* vis = reinterpret_cast<uint32_t*>(sm + C::VIS_OFF);
    if (use_vis && (warp == 2 || warp == 3)) {
        const int nw = (hi + 31) >> 5;
        for (int w = warp - 2; w < nw; w += 2) {
            const int t = w * 32 + lane;
            const uint32_t word = __ballot_sync(0xffffffffu, t < hi && tile_visible(mk, qb, t, kvalid));
            if (lane == 0) vis[w] = word;
        }
    }
    // first visible key tile >= t, or hi (the same enumeration in every role)
    auto next_vis = [=](int t) -> int {
        if (use_vis) {
            while (t < hi) {
                const uint32_t w = vis[t >> 5] >> (t & 31);
                if (w) return t + __ffs(w) - 1;
                t = (t | 31) + 1;
            }
            return hi;
        }
        while (t < hi && !tile_visible(mk, qb, t, kvalid)) ++t;
        return t;
    };

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 256);
            mbar_init(&xch[i], 256);
        }
        mbar_init(sum_x, 256);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
        // the Q tile is requested before TMEM allocation and the CTA-wide
        // barrier (a query tile with no visible key tile never waits for it,
        // and the producer lets it land before the CTA exits)
        mbar_arrive_expect_tx(bar_q, C::TILE_BYTES);
        for (int r = 0; r < C::NREG; ++r)
            tma_load_2d(sm + C::Q_OFF + r * 16384, &tmQ, r * 64, bh * N + qb * kTile, bar_q);
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;
    // number of key tiles this query tile visits
    int ntiles = 0;
    if (use_vis) {
        for (int w = 0; w < ((hi + 31) >> 5); ++w) ntiles += __popc(vis[w]);
    } else {
        for (int t = 0; t < hi; ++t) ntiles += tile_visible(mk, qb, t, kvalid) ? 1 : 0;
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int u = 0;
            for (int t = next_vis(0); t < hi; t = next_vis(t + 1)) {
                const int st = u % C::STAGES;
                const uint32_t ph = (u / C::STAGES) & 1;
                if (!mbar_wait(&kv_empty[st], ph ^ 1, cx, 31)) break;
                uint8_t* sk = sm + C::K_OFF + st * C::TILE_BYTES;
                uint8_t* sv = sm + C::V_OFF + st * C::TILE_BYTES;
                mbar_arrive_expect_tx(&kv_full[st], 2 * C::TILE_BYTES);
                for (int r = 0; r < C::NREG; ++r) {
                    tma_load_2d(sk + r * 16384, &tmK, r * 64, bh * N + t * kTile, &kv_full[st]);
                    tma_load_2d(sv + r * 16384, &tmV, r * 64, bh * N + t * kTile, &kv_full[st]);
                }
                ++u;
            }
            // let every copy in flight land before the CTA can exit
            mbar_wait_teardown(bar_q, 0, 200000000ull);
            for (int i = 0; i < C::STAGES && i < u; ++i) {
                const int last = i + ((u - 1 - i) / C::STAGES) * C::STAGES;
                mbar_wait_teardown(&kv_full[i], (last / C::STAGES) & 1, 200000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs the loop; one elected lane issues
        if (ntiles > 0) {
            const uint32_t leader = elect_one_sync();
            bool ok = mbar_wait_warp(bar_q, 0, cx, 32);
            const uint64_t dQ = sdesc_sw128(smem_u32(sm + C::Q_OFF), 16, 1024);
            const uint64_t dK0 = sdesc_sw128(smem_u32(sm + C::K_OFF), 16, 1024);
            const uint64_t dV0 = sdesc_sw128(smem_u32(sm + C::V_OFF), 16384, 1024);  // MN-major
            // S(j) = scale-free Q K_j^T into buffer j % 2
            auto issue_s = [=](int j) -> bool {
                const int st = j % C::STAGES;
                if (!mbar_wait_warp(&kv_full[st], (j / C::STAGES) & 1, cx, 33)) return false;
                tc_fence_after();
                const uint64_t ks = sdesc_advance(dK0, st * C::TILE_BYTES);
                const uint32_t sbuf = tm + (j & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                    umma_ss<false>(leader, sbuf, sdesc_advance(dQ, off), sdesc_advance(ks, off), C::ID_S, kk > 0 ? 1u : 0u);
                }
                umma_commit(leader, &s_full[j & 1]);
                return true;
            };
            if (ok) tc_fence_after();
            for (int j = 0; ok && j < 2 && j < ntiles; ++j) ok = issue_s(j);
            for (int u = 0; ok && u < ntiles; ++u) {
                // O += P(u) V(u); P of keys 0-63 in columns 0-31, keys 64-127 in 64-95
                if (!(ok = mbar_wait_warp(&p_full[u & 1], (u >> 1) & 1, cx, 34))) break;
                tc_fence_after();
                const int st = u % C::STAGES;
                const uint64_t vs = sdesc_advance(dV0, st * C::TILE_BYTES);
                const uint32_t pbuf = tm + (u & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts<false>(leader, tm + C::COL_O, pbuf + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_advance(vs, kk * 2048),
                                   C::ID_PV, (u > 0 || kk > 0) ? 1u : 0u);
                umma_commit(leader, &kv_empty[st]);  // K and V of tile u consumed
                if (u + 2 < ntiles) ok = issue_s(u + 2);
            }
            if (ok) umma_commit(leader, o_done);
            umma_commit(leader, drain);
            mbar_wait_teardown(drain, 0, 200000000ull);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax
        const int g = (warp - 4) >> 2;  // key columns 64 g .. 64 g + 63
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const int grow = qb * kTile + r;
        const uint32_t tl = tm + (static_cast<uint32_t>(wq * 32) << 16);
        const float c2 = p.scale_log2;
        float* xbuf = reinterpret_cast<float*>(sm + C::X_OFF);  // [parity][group][row]
        float m_hat = -CUDART_INF_F, l = 0.f, lw = 0.f;  // l: fp32 sum; lw: sum of bf16 weights
        bool ok = true;
        int u = 0;
        for (int t = next_vis(0); t < hi; t = next_vis(t + 1)) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[u & 1], (u >> 1) & 1, cx, 35));
            if (!ok) break;
            tc_fence_after();
            const uint32_t sb = tl + (u & 1) * 128;
            uint32_t sr[2][32];
            tmem_ld32(sb + 64 * g, sr[0]);
            tmem_ld32(sb + 64 * g + 32, sr[1]);
            tmem_ld_wait(sr[0]);
            tmem_ld_wait(sr[1]);
            if (tile_partial(mk, qb, t, kvalid)) {
                const int lim = min(kvalid - t * kTile, mk.causal && t == qb ? r + 1 : kTile) - 64 * g;
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c * 32 + i >= lim) sr[c][i] = __float_as_uint(-CUDART_INF_F);
            }
            // row maximum of this group's 64 columns as four independent
            // chains (one chain of 32 dependent maxima would sit on the
            // critical path), combined at the end
            float mc[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) mc[k] = -CUDART_INF_F;
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const int k = 2 * c + ((i >> 2) & 1);
                    mc[k] = fmax3(mc[k], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
                    mc[k] = fmax3(mc[k], __uint_as_float(sr[c][i + 2]), __uint_as_float(sr[c][i + 3]));
                }
            float mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), mc[3]);
            // agree on the row maximum with the other column group
            xbuf[(u & 1) * 256 + g * 128 + r] = mx;
            mbar_arrive(&xch[u & 1]);
            ok = __all_sync(0xffffffffu, mbar_wait(&xch[u & 1], (u >> 1) & 1, cx, 36));
            if (!ok) break;
            mx = fmaxf(mx, xbuf[(u & 1) * 256 + (g ^ 1) * 128 + r]);
            const float m_new = fmaxf(m_hat, mx * c2);
            const bool resc = (m_new - m_hat) > kQ1RescaleThreshold;
            float alpha = 1.f;
            if (resc) {
                alpha = ex2_approx(m_hat - m_new);
                m_hat = m_new;
                l *= alpha;
                lw *= alpha;
            }
            const float mu = (m_hat == -CUDART_INF_F) ? 0.f : m_hat;
            const uint64_t c2c2 = f2_make(c2, c2), nmu2 = f2_make(-mu, -mu);
            uint64_t rs2 = 0ull, rr2 = 0ull;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    f2_split(f2_fma(f2_make(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), c2c2,
                                    nmu2),
                             x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    pk[i] = pack_bf16x2(p0, p1);
                    rs2 = f2_add(rs2, f2_make(p0, p1));
                    rr2 = f2_add(rr2, f2_from_bf16x2(pk[i]));
                }
                tmem_st16(sb + 64 * g + c * 16, pk);
            }
            {
                float a0, a1;
                f2_split(rs2, a0, a1);
                l += a0 + a1;
                f2_split(rr2, a0, a1);
                lw += a0 + a1;
            }
            tmem_st_wait();
            if (__any_sync(0xffffffffu, resc) && u > 0) {
                // bring O (this group's half of the columns) to the new
                // reference maximum once the previous P V has completed
                const int pst = (u - 1) % C::STAGES;
                ok = __all_sync(0xffffffffu, mbar_wait(&kv_empty[pst], ((u - 1) / C::STAGES) & 1, cx, 37));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    uint32_t ov[32];
                    const uint32_t oc = tl + C::COL_O + g * (D / 2) + c * 32;
                    tmem_ld32(oc, ov);
                    tmem_ld_wait(ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    tmem_st32(oc, ov);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            if (!FA_DROP_THIS_ARRIVE(u == 0)) mbar_arrive(&p_full[u & 1]);
            ++u;
        }
        // ------------------------------------------------------------ epilogue
        // Add the two groups' partial row sums through the exchange buffer:
        // l in the half of parity u (last read two tiles ago), then lw in the
        // other half (its last reader, the partner's final tile, has since
        // arrived at the first exchange).
        float l_other = 0.f, lw_other = 0.f;
        if (ok) {
            xbuf[(u & 1) * 256 + g * 128 + r] = l;
            mbar_arrive(sum_x);
            ok = __all_sync(0xffffffffu, mbar_wait(sum_x, 0, cx, 38));
            if (ok) l_other = xbuf[(u & 1) * 256 + (g ^ 1) * 128 + r];
        }
        if (ok) {
            xbuf[((u + 1) & 1) * 256 + g * 128 + r] = lw;
            mbar_arrive(sum_x);
            ok = __all_sync(0xffffffffu, mbar_wait(sum_x, 1, cx, 40));
            if (ok) lw_other = xbuf[((u + 1) & 1) * 256 + (g ^ 1) * 128 + r];
        }
        if (ok && u > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(o_done, 0, cx, 39));
            if (ok) tc_fence_after();
        }
        if (ok) {
            const float lt = l + l_other;
            const float lwt = lw + lw_other;
            const float inv = lwt > 0.f ? 1.f / lwt : 0.f;
            uint16_t* orow = static_cast<uint16_t*>(p.o) + (static_cast<size_t>(bh) * N + grow) * D + g * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t ov[32];
                if (u > 0) {
                    tmem_ld32(tl + C::COL_O + g * (D / 2) + c * 32, ov);
                    tmem_ld_wait(ov);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = 0u;
                }
                uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_uint4(pack_bf16x2(__uint_as_float(ov[8 * j]) * inv, __uint_as_float(ov[8 * j + 1]) * inv),
                                        pack_bf16x2(__uint_as_float(ov[8 * j + 2]) * inv, __uint_as_float(ov[8 * j + 3]) * inv),
                                        pack_bf16x2(__uint_as_float(ov[8 * j + 4]) * inv, __uint_as_float(ov[8 * j + 5]) * inv),
                                        pack_bf16x2(__uint_as_float(ov[8 * j + 6]) * inv, __uint_as_float(ov[8 * j + 7]) * inv));
            }
            if (g == 0)
                p.lse[static_cast<size_t>(bh) * N + grow] = lt > 0.f ? (m_hat + log2f(lt)) * kQ1Ln2 : -CUDART_INF_F;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

template <int D>
static cudaError_t launch_q1(const FwdArgs& a, cudaStream_t stream, int* nlaunch) {
    using C = Q1Cfg<D>;
    const uint64_t rows = static_cast<uint64_t>(a.B) * a.H * a.N;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_2d_sw128(&tq, a.q, rows, D, 2, kTile, 64) || !make_tmap_2d_sw128(&tk, a.k, rows, D, 2, kTile, 64) ||
        !make_tmap_2d_sw128(&tv, a.v, rows, D, 2, kTile, 64))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(fa_fwd_q1_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    Q1Params p;
    p.B = a.B;
    p.H = a.H;
    p.N = a.N;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.mask.blockmask = a.blockmask;
    p.mask.kv_len = a.kv_len;
    p.mask.causal = a.causal;
    p.mask.T = a.N / kTile;
    p.o = a.o;
    p.lse = a.lse;
    p.status = a.status;
    const dim3 grid = a.causal ? dim3(a.H, a.B, a.N / kTile) : dim3(a.N / kTile, a.H, a.B);
    if (a.ev_begin) cudaEventRecord(a.ev_begin, stream);
    fa_fwd_q1_kernel<D><<<grid, 384, C::SMEM, stream>>>(tq, tk, tv, p);
    if (a.ev_end) cudaEventRecord(a.ev_end, stream);
    *nlaunch = 1;
    return cudaGetLastError();
}

cudaError_t launch_fwd_bf16_q1(const FwdArgs& a, cudaStream_t stream, int* nlaunch) {
    if (a.d == 64) return launch_q1<64>(a, stream, nlaunch);
    return launch_q1<128>(a, stream, nlaunch);
}

}  // namespace fa

// Forward pass for bf16 calls without dropout ([B, H, N, d] tensors or packed
// variable-length batches): one 128-row query tile per CTA and two CTAs per
// SM.
//
// Same computation as fa_fwd.cu ("FlashAttention: making attention
// IO-aware", sections "Tiling: never materialise S" and "Online softmax";
// masked tiles are never loaded or computed, section "Counting the IO",
// block-sparse attention): for the query tile Q_i, stream the key / value
// tiles the mask keeps, form S = scale * Q_i K_j^T on the tensor cores, keep
// the running maximum m, the running sum l of exp(S - m) and the unnormalised
// output o (rescaled by exp(m_old - m_new) when the maximum grows), and write
// O = o / l and L = m + log l at the end.
//
// Why one query tile per CTA: in a CTA that holds two query tiles, one
// in-order MMA issuer serves both, and a key tile that only one of them needs
// (the usual case under a random tile mask) waits on that tile's chain
// S -> softmax -> P V -> next S. Here each CTA owns one query tile with its
// own producer, issuer and softmax warps, and two CTAs share an SM (256 TMEM
// columns and under half of the shared memory each): while one CTA's softmax
// forms P, the other's GEMMs run, and no issue order ties them together. The
// price is that each K and V tile is loaded once per query tile instead of
// once per pair: twice the L2-to-shared-memory traffic, well within what TMA
// sustains from L2.
//
// Layout of one CTA (192 threads):
//   thread 0    sets up the mbarriers and requests Q and the first K / V
//   warp 0      TMA producer: K tiles through KSTAGES stages and V in half
//               tiles (64 keys) through NVH slots, so that the first half of
//               the next V loads while the second half of the current one
//               is still being read
//   warp 1      allocates TMEM (256 columns); one elected lane issues the MMAs
//   warps 2-5   softmax: thread r owns row r (TMEM lane r, r = 32 (warp % 4)
//               + lane); before the loop they turn the mask row into a bitmap
// TMEM: S in columns [0, 128) (P overwrites it as bf16), O in [128, 128 + d).
// The reference maximum is only moved (and O rescaled) when the row maximum
// grows by more than 2^8 in the exp2 domain (exact: o and l always share it).
// Two running sums: l over the fp32 probabilities (gives L) and lw over their
// bf16 roundings, the weights P V multiplies (normalises O).
#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_launch.h"
#include "tmap.h"

namespace fa {

// Key tiles per sequence up to which the visible tiles are kept as a bitmap
// in shared memory (N <= 524,288); longer rows read the mask tile by tile.
constexpr int kT1VisMaxTiles = 4096;

template <int D>
struct T1Cfg {
    static constexpr int TILE_BYTES = kTile * D * 2;   // 128 rows of Q or K
    static constexpr int HALF_BYTES = TILE_BYTES / 2;  // 64 rows of V
    static constexpr int NREG = D / 64;                // 128-byte swizzle regions per row
    static constexpr int KSTAGES = D == 64 ? 2 : 1;
    static constexpr int NVH = D == 64 ? 4 : 2;         // V half-tile slots
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + TILE_BYTES;
    static constexpr int V_OFF = K_OFF + KSTAGES * TILE_BYTES;
    static constexpr int BAR_OFF = V_OFF + NVH * HALF_BYTES;
    static constexpr int VIS_OFF = BAR_OFF + 256;
    static constexpr int VIS_WORDS = kT1VisMaxTiles / 32;
    static constexpr int USED = VIS_OFF + VIS_WORDS * 4;
    static constexpr int SMEM = USED + 1024;  // + alignment slack
    static constexpr int THREADS = 192;
    static constexpr int COL_O = 128;
    static constexpr int S_KSTEPS = D / 16;
    static constexpr uint32_t ID_S = idesc_make(128, 128, kFmtBF16, false, false);
    // V is read MN-major straight from its [keys][d] layout
    static constexpr uint32_t ID_PV = idesc_make(128, D, kFmtBF16, false, true);
    // two CTAs per SM: 228 KiB per SM, 1 KiB of it reserved per CTA
    static_assert(2 * (SMEM + 1024) <= 233472, "two CTAs per SM");
    static_assert((1 + 2 * KSTAGES + 2 * NVH + 5) * 8 + 8 <= 256, "barrier area");
};

struct T1Params {
    int B, H, N;
    float scale_log2;  // scale * log2(e)
    MaskArgs mask;
    void* o;
    float* lse;
    int* status;
    int group;  // > 0 (causal): 1D grid of head groups, longest query tile first in each
    const int32_t* cu_seqlens;  // packed variable-length batch, else null
    int total;                  // tokens of the packed batch
};

constexpr float kT1RescaleThreshold = 8.0f;  // log2 units
constexpr float kT1Ln2 = 0.69314718055994530942f;

// VARLEN: packed variable-length batch ([total, H, d] tensors, sequence b at
// tokens cu_seqlens[b] .. cu_seqlens[b + 1] - 1, L as [H, total]); a separate
// instantiation so that the [B, H, N, d] kernel carries none of its branches.
template <int D, bool VARLEN>
__global__ void __launch_bounds__(192, 2)
    fa_fwd_t1_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmVh, const __grid_constant__ CUtensorMap tmO,
                     const __grid_constant__ T1Params p) {
    using C = T1Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base for the swizzled tiles, kept in the shared
    // address space
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((sm - smem_raw) + C::USED > C::SMEM) {
        if (tid == 0 && p.status) atomicCAS(p.status, 0, FA_DEV_TIMEOUT | (96 << 8));
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    uint64_t* bar_q = bars + 0;
    uint64_t* k_full = bars + 1;               // [KSTAGES] K of a stage landed
    uint64_t* k_empty = k_full + C::KSTAGES;   // [KSTAGES] the S GEMM reading it is done
    uint64_t* v_full = k_empty + C::KSTAGES;   // [NVH] V half of a slot landed
    uint64_t* v_empty = v_full + C::NVH;       // [NVH] the P V GEMMs reading it are done
    uint64_t* s_full = v_empty + C::NVH;
    uint64_t* p_half = s_full + 1;             // P of keys 0-63 stored
    uint64_t* p_full = p_half + 1;             // P of all keys stored
    uint64_t* o_done = p_full + 1;
    uint64_t* drain = o_done + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const WaitCtx cx{abort_flag, p.status};

    // Without a causal mask every query tile of a head costs about the same:
    // query tile fastest, so that the CTAs running together read the K and V
    // of one or two heads, which stay in L2. With a causal mask query tile qb
    // reads qb + 1 key tiles: a 1D grid runs groups of p.group heads in turn
    // (sized so that a group's K and V stay in L2), longest tile first across
    // the heads of a group, so that the kernel ends on short CTAs.
    // A packed batch runs a (query tile, H, B) grid over its longest
    // sequence, query tile fastest so that the CTAs running together share a
    // head's K and V in L2: CTAs past the end of a shorter sequence leave at
    // once, and with a causal mask z = 0 is the sequence's last (longest)
    // query tile.
    int qb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    int N = p.N, T = p.mask.T, seq0 = 0;
    if constexpr (VARLEN) {
        h = blockIdx.y;
        b = blockIdx.z;
        const int s0 = min(max(p.cu_seqlens[b], 0), p.total);
        const int s1 = min(max(p.cu_seqlens[b + 1], s0), p.total);
        if (s1 - s0 > p.N && tid == 0 && h == 0 && blockIdx.x == 0 && p.status)
            atomicCAS(p.status, 0, FA_DEV_INVALID | (95 << 8));
        seq0 = s0;
        N = min(s1 - s0, p.N);
        T = (N + kTile - 1) / kTile;
        const int z = static_cast<int>(blockIdx.x);
        if (z >= T) return;  // uniform over the CTA, before any barrier or TMEM use
        qb = p.mask.causal ? T - 1 - z : z;
    } else if (p.group > 0) {
        const int nb = p.B * p.H, L = static_cast<int>(blockIdx.x);
        const int gi = L / (p.group * T), rr = L - gi * p.group * T;
        const int g0 = gi * p.group, gsz = min(p.group, nb - g0);
        const int zq = rr / gsz, bhx = g0 + (rr - zq * gsz);
        qb = T - 1 - zq;
        b = bhx / p.H;
        h = bhx - b * p.H;
    }
    const int bh = b * p.H + h;
    const int kvalid = VARLEN ? N : keys_valid(p.mask, b, N);
    int hi = min(T, (kvalid + kTile - 1) / kTile);
    if (p.mask.causal) hi = min(hi, qb + 1);
    const MaskArgs mk = p.mask;
    const bool use_vis = mk.blockmask != nullptr && hi <= kT1VisMaxTiles;
    uint32_t* vis = reinterpret_cast<uint32_t*>(sm + C::VIS_OFF);
    auto visible_t = [=](int t) -> bool {
        if (use_vis) return (vis[t >> 5] >> (t & 31)) & 1u;
        return tile_visible(mk, qb, t, kvalid);
    };
    // first key tile >= t that the walk visits: with the bitmap the next
    // visible one (or hi); otherwise t itself, and the walk tests each tile
    auto next_tile = [=](int t) -> int {
        if (use_vis) {
            while (t < hi) {
                const uint32_t w = vis[t >> 5] >> (t & 31);
                if (w) return t + __ffs(w) - 1;
                t = (t | 31) + 1;
            }
            return hi;
        }
        return t;
    };

    // rows row .. of this head ([B, H, N, d]) or of this sequence (packed)
    auto load_rows = [&](void* dst, const CUtensorMap* m, int x, int row, uint64_t* bar) {
        if constexpr (VARLEN)
            tma_load_3d(dst, m, x, h, seq0 + row, bar);
        else
            tma_load_2d(dst, m, x, bh * N + row, bar);
    };
    auto load_k = [&](int t, int kst) {
        uint8_t* sk = sm + C::K_OFF + kst * C::TILE_BYTES;
        mbar_arrive_expect_tx(&k_full[kst], C::TILE_BYTES);
        for (int r = 0; r < C::NREG; ++r) load_rows(sk + r * 16384, &tmK, r * 64, t * kTile, &k_full[kst]);
    };
    // V half hf (keys 64 hf .. 64 hf + 63) of key tile t into slot vs: NREG
    // swizzled boxes of [64 keys x 64 columns], 8 KiB apart
    auto load_vh = [&](int t, int hf, int vs) {
        uint8_t* sv = sm + C::V_OFF + vs * C::HALF_BYTES;
        mbar_arrive_expect_tx(&v_full[vs], C::HALF_BYTES);
        for (int r = 0; r < C::NREG; ++r)
            load_rows(sv + r * 8192, &tmVh, r * 64, t * kTile + hf * 64, &v_full[vs]);
    };

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(bar_q, 1);
        for (int i = 0; i < C::KSTAGES; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < C::NVH; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_half, 128);
        mbar_init(p_full, 128);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
        // the Q load is the CTA's start-up latency: requested first, before
        // TMEM allocation and the CTA-wide barrier
        mbar_arrive_expect_tx(bar_q, C::TILE_BYTES);
        for (int r = 0; r < C::NREG; ++r)
            load_rows(sm + C::Q_OFF + r * 16384, &tmQ, r * 64, qb * kTile, bar_q);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmVh);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    if (use_vis && warp >= 2) {
        const int nw = (hi + 31) >> 5;
#pragma unroll 4
        for (int w = warp - 2; w < nw; w += 4) {
            const int t = w * 32 + lane;
            const uint32_t word = __ballot_sync(0xffffffffu, t < hi && tile_visible(mk, qb, t, kvalid));
            if (lane == 0) vis[w] = word;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // tile u of the walk: K into stage u % KSTAGES, its V halves into
            // slots (2u + hf) % NVH; each waits for the GEMMs that last read
            // the buffer (the order K, V half 0, V half 1 is the order in which
            // those GEMMs complete)
            int u = 0;
            for (int t = next_tile(0); t < hi; t = next_tile(t + 1)) {
                if (!visible_t(t)) continue;
                const int kst = u % C::KSTAGES;
                if (!mbar_wait(&k_empty[kst], ((u / C::KSTAGES) & 1) ^ 1, cx, 31)) break;
                load_k(t, kst);
                bool ok = true;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int n = 2 * u + hf, vs = n % C::NVH;
                    if (!(ok = mbar_wait(&v_empty[vs], ((n / C::NVH) & 1) ^ 1, cx, 32))) break;
                    load_vh(t, hf, vs);
                }
                if (!ok) break;
                ++u;
            }
            // let every copy in flight land before the CTA can exit
            mbar_wait_teardown(bar_q, 0, 200000000ull);
            for (int i = 0; i < C::KSTAGES && i < u; ++i) {
                const int last = i + ((u - 1 - i) / C::KSTAGES) * C::KSTAGES;
                mbar_wait_teardown(&k_full[i], (last / C::KSTAGES) & 1, 200000000ull);
            }
            for (int i = 0; i < C::NVH && i < 2 * u; ++i) {
                const int last = i + ((2 * u - 1 - i) / C::NVH) * C::NVH;
                mbar_wait_teardown(&v_full[i], (last / C::NVH) & 1, 200000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs the loop; one elected lane issues
        const uint32_t leader = elect_one_sync();
        bool ok = mbar_wait_warp(bar_q, 0, cx, 33);
        if (ok) tc_fence_after();
        const uint64_t dQ0 = sdesc_sw128(smem_u32(sm + C::Q_OFF), 16, 1024);
        const uint64_t dK0 = sdesc_sw128(smem_u32(sm + C::K_OFF), 16, 1024);
        // V half slots MN-major: the two 64-column regions of a slot are
        // 8 KiB apart
        const uint64_t dV0 = sdesc_sw128(smem_u32(sm + C::V_OFF), 8192, 1024);
        // O += P V of walk tile uu: half hf (keys 64 hf ..) as soon as the
        // softmax has stored P for those keys and V half hf has landed; the
        // commit after each half releases its V slot
        auto issue_pv = [&](int uu) -> bool {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                if (!mbar_wait_warp(hf == 0 ? p_half : p_full, uu & 1, cx, 34)) return false;
                const int n = 2 * uu + hf, vs = n % C::NVH;
                if (!mbar_wait_warp(&v_full[vs], (n / C::NVH) & 1, cx, 35)) return false;
                tc_fence_after();
                const uint64_t vd = sdesc_advance(dV0, vs * C::HALF_BYTES);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_ts<false>(leader, tm + C::COL_O, tm + (hf * 4 + kk) * 8, sdesc_advance(vd, kk * 2048),
                                   C::ID_PV, (uu > 0 || hf > 0 || kk > 0) ? 1u : 0u);
                umma_commit(leader, &v_empty[vs]);
            }
            return true;
        };
        int u = 0;
        for (int t = next_tile(0); ok && t < hi; t = next_tile(t + 1)) {
            if (!visible_t(t)) continue;
            // the previous tile's P V goes first: S below overwrites the
            // columns its P is read from, and MMAs run in issue order
            if (u > 0 && !(ok = issue_pv(u - 1))) break;
            const int kst = u % C::KSTAGES;
            if (!(ok = mbar_wait_warp(&k_full[kst], (u / C::KSTAGES) & 1, cx, 36))) break;
            tc_fence_after();
            const uint64_t ks = sdesc_advance(dK0, kst * C::TILE_BYTES);
#pragma unroll
            for (int kk = 0; kk < C::S_KSTEPS; ++kk) {
                const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                umma_ss<false>(leader, tm, sdesc_advance(dQ0, off), sdesc_advance(ks, off), C::ID_S, kk > 0 ? 1u : 0u);
            }
            umma_commit(leader, s_full);
            umma_commit(leader, &k_empty[kst]);
            ++u;
        }
        if (ok && u > 0) ok = issue_pv(u - 1);
        if (ok) umma_commit(leader, o_done);
        // every MMA issued so far must be complete before TMEM is released
        umma_commit(leader, drain);
        mbar_wait_teardown(drain, 0, 200000000ull);
    } else {
        // ------------------------------------------------------------ softmax
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t tl = tm + (static_cast<uint32_t>(wq * 32) << 16);
        const float c2 = p.scale_log2;
        float m_hat = -CUDART_INF_F, l = 0.f, lw = 0.f;
        int n = 0;
        bool ok = true;
        for (int t = next_tile(0); t < hi; t = next_tile(t + 1)) {
            if (!visible_t(t)) continue;
            ok = mbar_wait(s_full, n & 1, cx, 37);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tl + c * 32, sr[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
            if (tile_partial(mk, qb, t, kvalid)) {
                const int lim = min(kvalid - t * kTile, mk.causal && t == qb ? r + 1 : kTile);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c * 32 + i >= lim) sr[c][i] = __float_as_uint(-CUDART_INF_F);
            }
            // row maximum as eight independent chains, combined at the end
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
            const float mx =
                fmaxf(fmax3(mc[0], mc[1], mc[2]), fmaxf(fmax3(mc[3], mc[4], mc[5]), fmax3(mc[6], mc[7], mc[7])));
            const float m_new = fmaxf(m_hat, mx * c2);
            const bool resc = (m_new - m_hat) > kT1RescaleThreshold;
            float alpha = 1.f;
            if (resc) {
                alpha = ex2_approx(m_hat - m_new);
                m_hat = m_new;
                l *= alpha;
                lw *= alpha;
            }
            const float mu = (m_hat == -CUDART_INF_F) ? 0.f : m_hat;
            const uint64_t c2c2 = f2_make(c2, c2), nmu2 = f2_make(-mu, -mu);
            // O is rescaled (below) before any P V of this tile may run
            const bool resc_any = __any_sync(0xffffffffu, resc) && n > 0;
            uint64_t rs2 = 0ull;
            uint32_t pk[4][16];  // P as bf16 pairs; kept for the bf16-weight sum
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    f2_split(f2_fma(f2_make(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), c2c2,
                                    nmu2),
                             x0, x1);
                    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                    pk[c][i] = pack_bf16x2(p0, p1);
                    rs2 = f2_add(rs2, f2_make(p0, p1));
                }
                tmem_st16(tl + c * 16, pk[c]);
                if (c == 1 && !resc_any) {
                    // keys 0-63 are ready: the first half of P V may start
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(p_half);
                }
            }
            tmem_st_wait();
            {
                float a_, b_;
                f2_split(rs2, a_, b_);
                l += a_ + b_;
            }
            // the sum of the bf16-rounded weights (what P V multiplies) is
            // not needed before the next tile: in the usual case it is formed
            // after P has been handed to the MMA thread
            auto bf16_row_sum = [&]() {
                uint64_t rr2 = 0ull;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 16; ++i) rr2 = f2_add(rr2, f2_from_bf16x2(pk[c][i]));
                float a_, b_;
                f2_split(rr2, a_, b_);
                lw += a_ + b_;
            };
            if (resc_any) {
                bf16_row_sum();
                // O holds the previous tiles' sum; their last P V was issued
                // before this tile's S, and MMAs complete in issue order, so S
                // being complete means O is final: rescale it to the new
                // reference maximum
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld32(tl + C::COL_O + c * 32, ov);
                    tmem_ld_wait(ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    tmem_st32(tl + C::COL_O + c * 32, ov);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(p_half);
                if (!FA_DROP_THIS_ARRIVE(n == 0)) mbar_arrive(p_full);
            } else {
                tc_fence_before();
                if (!FA_DROP_THIS_ARRIVE(n == 0)) mbar_arrive(p_full);
                bf16_row_sum();
            }
            ++n;
        }
        // ------------------------------------------------------------ epilogue
        if (ok && n > 0) {
            ok = mbar_wait(o_done, 0, cx, 38);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) tc_fence_after();
        }
        if (ok) {
            const float inv = lw > 0.f ? 1.f / lw : 0.f;
            const int grow = qb * kTile + r;  // query row within the sequence
            // packed rows past the end of the sequence belong to the next
            // one: computed (the TMEM loads are warp-wide) but not stored
            const bool row_ok = !VARLEN || grow < N;
            const size_t orow = VARLEN ? (static_cast<size_t>(seq0 + grow) * p.H + h) * D
                                       : (static_cast<size_t>(bh) * N + grow) * D;
            // a warp whose 32 rows all lie in the sequence stages them in the
            // Q buffer (every S GEMM is complete once o_done is), as [32 x 64]
            // swizzled boxes, and stores them with one bulk tensor copy per
            // box; other warps, and a tile that saw no key tile (n == 0:
            // nothing waited for its Q load, which may still be landing in the
            // buffer), store their valid rows directly
            const int wrow0 = qb * kTile + wq * 32;
            const bool tma_rows = n > 0 && (!VARLEN || wrow0 + 32 <= N);
            uint8_t* ob = sm + C::Q_OFF + wq * (C::NREG * 4096);
            uint32_t oa[D / 32][32];
            if (n > 0) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) tmem_ld32(tl + C::COL_O + c * 32, oa[c]);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) tmem_ld_wait(oa[c]);
            } else {
#pragma unroll
                for (int c = 0; c < D / 32; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) oa[c][i] = 0u;
            }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
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
                        sts128(smem_u32(ob + (c >> 1) * 4096 + lane * 128 + ((ch ^ (lane & 7)) << 4)), w.x, w.y, w.z,
                               w.w);
                    } else if (row_ok) {
                        dst[j] = w;
                    }
                }
            }
            if (tma_rows) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int rg = 0; rg < C::NREG; ++rg)
                        if constexpr (VARLEN)
                            tma_store_3d(&tmO, rg * 64, h, seq0 + wrow0, ob + rg * 4096);
                        else
                            tma_store_2d(&tmO, rg * 64, bh * N + wrow0, ob + rg * 4096);
                    bulk_commit_group();
                    // the shared buffer must be read out before the CTA exits
                    bulk_wait_group_read0();
                }
            }
            const size_t lrow = VARLEN ? static_cast<size_t>(h) * p.total + seq0 + grow : static_cast<size_t>(bh) * N + grow;
            if (row_ok) p.lse[lrow] = l > 0.f ? (m_hat + log2f(l)) * kT1Ln2 : -CUDART_INF_F;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 256);
    }
}

template <int D>
static cudaError_t launch_t1(const FwdArgs& a, cudaStream_t stream, int* nlaunch) {
    using C = T1Cfg<D>;
    const uint64_t rows = static_cast<uint64_t>(a.B) * a.H * a.N;
    CUtensorMap tq, tk, tvh, to;
    if (a.cu_seqlens) {
        const uint64_t tot = static_cast<uint64_t>(a.total);
        if (!make_tmap_packed_sw128(&tq, a.q, tot, a.H, D, 2, kTile, 64) ||
            !make_tmap_packed_sw128(&tk, a.k, tot, a.H, D, 2, kTile, 64) ||
            !make_tmap_packed_sw128(&tvh, a.v, tot, a.H, D, 2, 64, 64) ||
            !make_tmap_packed_sw128(&to, a.o, tot, a.H, D, 2, 32, 64))
            return cudaErrorInvalidValue;
    } else if (!make_tmap_2d_sw128(&tq, a.q, rows, D, 2, kTile, 64) ||
               !make_tmap_2d_sw128(&tk, a.k, rows, D, 2, kTile, 64) ||
               !make_tmap_2d_sw128(&tvh, a.v, rows, D, 2, 64, 64) ||
               !make_tmap_2d_sw128(&to, a.o, rows, D, 2, 32, 64)) {
        return cudaErrorInvalidValue;
    }
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(fa_fwd_t1_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fa_fwd_t1_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    T1Params p;
    p.B = a.B;
    p.H = a.H;
    p.N = a.N;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.mask.blockmask = a.blockmask;
    p.mask.kv_len = a.kv_len;
    p.mask.causal = a.causal;
    p.mask.T = (a.N + kTile - 1) / kTile;
    p.o = a.o;
    p.lse = a.lse;
    p.status = a.status;
    p.cu_seqlens = a.cu_seqlens;
    p.total = a.total;
    // causal [B, H, N, d] calls: head groups whose K and V take at most 64 MiB
    p.group = 0;
    if (a.causal && !a.cu_seqlens) {
        long long g = (64LL << 20) / (4LL * a.N * D);
        g = g < 1 ? 1 : g;
        p.group = static_cast<int>(g < a.B * a.H ? g : a.B * a.H);
    }
    const unsigned T = static_cast<unsigned>(p.mask.T);
    const dim3 grid = p.group > 0 ? dim3(T * a.H * a.B) : dim3(T, a.H, a.B);
    if (a.ev_begin) cudaEventRecord(a.ev_begin, stream);
    if (a.cu_seqlens)
        fa_fwd_t1_kernel<D, true><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tvh, to, p);
    else
        fa_fwd_t1_kernel<D, false><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tvh, to, p);
    if (a.ev_end) cudaEventRecord(a.ev_end, stream);
    *nlaunch = 1;
    return cudaGetLastError();
}

cudaError_t launch_fwd_bf16_t1(const FwdArgs& a, cudaStream_t stream, int* nlaunch) {
    if (a.d == 64) return launch_t1<64>(a, stream, nlaunch);
    return launch_t1<128>(a, stream, nlaunch);
}

}  // namespace fa

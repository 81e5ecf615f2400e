// Forward pass of fused, tiled, exact softmax attention on sm_103a.
//
// What it computes ("FlashAttention: making attention IO-aware", sections
// "Tiling: never materialise S" and "Online softmax", and the page's tiled
// forward listing): for each query tile Q_i it streams key/value tiles
// (K_j, V_j), forms S_ij = scale * Q_i K_j^T on the tensor cores, updates a
// running row maximum m, a running sum l of exp(S - m) and an unnormalised
// output o (rescaled by exp(m_old - m_new) when the maximum grows), and at the
// end writes O = o / l and L = m + log l. Tiles that the causal mask, the key
// padding or the tile mask remove are never loaded or computed
// ("FlashAttention-2": tiles above the diagonal are skipped; "Counting the
// IO": block-sparse attention skips masked tiles).
//
// This file's kernel serves fp32 inputs and dropout; bf16 calls without
// dropout ([B, H, N, d] or packed) run fa_fwd_t1.cu (one query tile per CTA,
// two CTAs per SM), which is faster on every measured shape.
//
// GB300 design (one CTA per pair of 128-row query tiles of one head):
//   thread 0    sets up the mbarriers and requests both Q tiles and the first
//               K / V tile before the CTA-wide barrier
//   warp 0      TMA producer: the remaining K and V tiles through separate
//               multi-stage shared-memory rings guarded by mbarriers
//   warp 1      allocates TMEM; the whole warp runs the issue loop and one
//               elected lane issues every tcgen05.mma and commit
//   warps 2-3   idle after the set-up
//   warps 4-7   softmax warpgroup of Q tile 0 (thread r owns row r, which is
//               TMEM lane r, so row max and row sum are in-thread)
//   warps 8-11  softmax warpgroup of Q tile 1
// TMEM (512 columns): per Q tile, S (128 fp32 columns, P overwrites it as
// bf16) and the O accumulator (d columns). The MMA warp interleaves the two
// Q tiles so that one tile's softmax overlaps the other tile's GEMMs, and
// issues each P V in slices of the keys as the softmax stores them. The
// epilogue stages O in the Q tile's buffer and writes it with TMA stores.
// The online-softmax reference maximum is only moved (and O rescaled) when
// the row maximum grows by more than 2^8 in the exp2 domain; otherwise the
// stale maximum is kept, which is exact because o and l always share it.
// Two running sums are kept: l over the fp32 probabilities, which gives L,
// and lw over the same probabilities after their rounding to bf16, i.e. the
// weights the P V product actually multiplies, which normalises O so that it
// is a convex combination of rows of V even with bf16 weights.
#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_philox.cuh"
#include "fa_launch.h"
#include "tmap.h"

namespace fa {

template <bool TF32, int D>
struct FwdCfg {
    static constexpr int ELEM = TF32 ? 4 : 2;
    static constexpr int ROWB = D * ELEM;              // bytes per row of Q/K/V
    static constexpr int NREG = ROWB / 128;            // 128-byte swizzle regions per row
    static constexpr int TILE_BYTES = kTile * ROWB;    // one 128-row tile
    // fp32 inputs: S is formed from tf32 high and low parts of Q and K
    // (Qh Kh^T + Qh Kl^T + Ql Kh^T), so Q and K tiles come in two copies.
    static constexpr int SPLIT = TF32 ? 2 : 1;
    // K and V rings: a K stage frees as soon as the S GEMMs reading it
    // complete, so extra K stages let the next K tiles load further ahead
    static constexpr int KSTAGES = TF32 ? 1 : (TILE_BYTES <= 16384 ? 6 : 3);
    static constexpr int VSTAGES = TF32 ? 1 : (TILE_BYTES <= 16384 ? 4 : 2);
    static constexpr int NQ = 2;                       // query tiles per CTA
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + NQ * SPLIT * TILE_BYTES;
    static constexpr int V_OFF = K_OFF + KSTAGES * SPLIT * TILE_BYTES;
    static constexpr int BAR_OFF = V_OFF + VSTAGES * TILE_BYTES;
    static constexpr int SMEM = BAR_OFF + 512 + 1024;  // + alignment slack
    static constexpr int KSTEP = 32 / ELEM;            // K elements per MMA instruction
    static constexpr int S_KSTEPS = D / KSTEP;
    static constexpr int PV_KSTEPS = kTile / KSTEP;
    static constexpr int THREADS = 384;
    static constexpr int BOXC = 128 / ELEM;            // elements per swizzle row
    static constexpr uint32_t ID_S = idesc_make(128, 128, TF32 ? kFmtTF32 : kFmtBF16, false, false);
    // bf16: V is read MN-major straight from its [keys][d] layout;
    // tf32 operands must be K-major, so V arrives transposed ([d][keys]).
    static constexpr uint32_t ID_PV = idesc_make(128, D, TF32 ? kFmtTF32 : kFmtBF16, false, !TF32);
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert((1 + 2 * KSTAGES + 2 * VSTAGES + 13) * 8 + 8 <= 512, "barrier area");
    static_assert(VSTAGES <= 16, "two bits of reader count per V stage");
};

struct FwdParams {
    int B, H, N;
    float scale_log2;  // scale * log2(e)
    MaskArgs mask;
    void* o;
    float* lse;
    int* status;
    DropoutArgs drop;           // dropout on the probabilities (DROPOUT kernels)
    int head_major;             // grid (pairs, H, B) instead of (H, B, pairs)
    int group;                  // > 0: 1D grid of head groups (heads per group), longest pair first in each
};

// Work item L of the head-group order: groups of `group` heads in turn (the
// last one may be smaller), and within a group pair rank zq (0 = longest)
// major, head minor.
__device__ __forceinline__ void fwd_group_item(int L, int group, int np, int nb, int H, int& b, int& h, int& zq) {
    const int gi = L / (group * np), r = L - gi * group * np;
    const int g0 = gi * group, gsz = min(group, nb - g0);
    zq = r / gsz;
    const int bhx = g0 + (r - zq * gsz);
    b = bhx / H;
    h = bhx - b * H;
}

// Issue state of the MMA thread, per Q tile s of the CTA.
struct MmaState {
    int pend_stage[2] = {-1, -1};  // V stage whose P V GEMM is still to be issued
    uint32_t pend_ph[2] = {0, 0};  // V-full phase parity of that stage
    int pend_u[2] = {0, 0};        // index (among loaded tiles) of that tile
    int nP[2] = {0, 0};            // P-ready phases consumed
    int nPV[2] = {0, 0};           // P V GEMMs issued
    uint32_t rem = 0;              // 2 bits per stage: Q tiles still to read its V
};

// O_s += P_s V for Q tile s's pending K/V tile, in PARTS slices of the
// keys: each as soon as the softmax warps have stored P for its keys
// (p_part[s][k] for all slices but the last, p_full for the last), so that
// the product runs while they form P for the later keys.
template <bool TF32, int D, int PARTS>
__device__ __forceinline__ bool fwd_issue_pv(uint32_t leader, int s, MmaState& st, uint32_t tm, uint64_t dV0,
                                             uint64_t* p_half, uint64_t* p_full,
                                             uint64_t* v_full, uint64_t* kv_empty, const WaitCtx& cx) {
    using C = FwdCfg<TF32, D>;
    const int ps = st.pend_stage[s];
    const uint32_t php = st.nP[s] & 1;
    if (!mbar_wait_warp(&p_half[s * 3], php, cx, 12)) return false;  // first slice
    // V comes through its own ring and is normally resident long before P
    if (!mbar_wait_warp(&v_full[ps], st.pend_ph[s], cx, 4)) return false;
    tc_fence_after();
    const uint64_t vst = sdesc_advance(dV0, ps * C::TILE_BYTES);
#pragma unroll
    for (int kk = 0; kk < C::PV_KSTEPS; ++kk) {
        if (kk > 0 && kk % (C::PV_KSTEPS / PARTS) == 0) {
            const int q = kk / (C::PV_KSTEPS / PARTS);
            if (!mbar_wait_warp(q == PARTS - 1 ? &p_full[s] : &p_half[s * 3 + q], php, cx, 3)) return false;
            tc_fence_after();
        }
        const uint32_t off = TF32 ? (kk / 4) * (D * 128) + (kk % 4) * 32 : kk * 2048;
        umma_ts<TF32>(leader, tm + s * 256 + 128, tm + s * 256 + kk * 8, sdesc_advance(vst, off), C::ID_PV,
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

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

// DROPOUT: dropout on the probabilities, with the keep mask regenerated from
// Philox (fa_philox.cuh); a separate instantiation.
template <bool TF32, int D, bool DROPOUT = false>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmQlo,
                  const __grid_constant__ CUtensorMap tmKlo, const __grid_constant__ CUtensorMap tmO,
                  const __grid_constant__ FwdParams p) {
    using C = FwdCfg<TF32, D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base for the swizzled tiles; offsetting the shared
    // array itself (rather than casting through an integer) keeps the pointer
    // in the shared address space, so accesses compile to shared loads/stores
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    uint64_t* bar_q = bars + 0;
    // K and V travel through separate rings with the same number of stages:
    // a K stage is released once the S GEMMs that read it complete, a V stage
    // once its P V GEMMs complete, so the next K tile loads during the
    // current tile's softmax instead of waiting for its P V products.
    uint64_t* k_full = bars + 1;               // K of a stage landed
    uint64_t* k_empty = k_full + C::KSTAGES;   // S GEMMs reading a K stage done
    uint64_t* v_full = k_empty + C::KSTAGES;   // V of a stage landed
    uint64_t* kv_empty = v_full + C::VSTAGES;  // P V GEMMs reading a V stage done
    uint64_t* s_full = kv_empty + C::VSTAGES;  // [2]
    uint64_t* p_full = s_full + 2;            // [2]
    uint64_t* o_done = p_full + 2;            // [2]
    uint64_t* drain = o_done + 2;
    // P V runs in two slices of the keys (more slices cost the softmax warps
    // more in TMEM-store waits than the earlier slices gain):
    // p_half[s][k] = P of slices 0..k stored
    constexpr int PV_PARTS = 2;
    uint64_t* p_half = drain + 1;             // [2][3]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p_half + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const WaitCtx cx{abort_flag, p.status};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Longest-first order (the query-tile pair index is the slowest grid
    // dimension): with causal masks the longest CTAs start first and the
    // short ones fill the tail. Causal [B, H, N, d] calls run it within
    // groups of p.group heads in turn on a 1D grid, the group sized so that
    // its K and V stay in L2 (across all heads the resident CTAs' K and V
    // tiles would span every head and part of them would be read again).
    // Without causal masking every pair of a head costs about the same, and
    // a tile mask (here: fp32 inputs) makes the pairs share few key tiles,
    // so the grid is then head-major instead: the CTAs running together read
    // one head's K and V, which stays in L2.
    int h = p.head_major ? blockIdx.y : blockIdx.x, b = p.head_major ? blockIdx.z : blockIdx.y;
    int zq = static_cast<int>(p.head_major ? blockIdx.x : blockIdx.z);  // pair rank, longest first
    if (p.group > 0)
        fwd_group_item(static_cast<int>(blockIdx.x), p.group, (p.mask.T + 1) >> 1, p.B * p.H, p.H, b, h, zq);
    // head (b, h) is rows bh * N .. of the [B * H * N, d] view
    const int N = p.N, T = p.mask.T;
    const int npairs = (T + 1) >> 1;
    const int qp = npairs - 1 - zq;
    if (qp < 0) return;  // uniform over the CTA, before any barrier or TMEM use
    const int qb0 = 2 * qp, qb1 = 2 * qp + 1;
    const bool act1 = qb1 < T;
    const int bh = b * p.H + h;
    const int kvalid = keys_valid(p.mask, b, N);
    int hi = T;
    if (p.mask.causal) hi = min(hi, (act1 ? qb1 : qb0) + 1);
    hi = min(hi, (kvalid + kTile - 1) / kTile);

    // K and V tile loads (producer thread): rows t * 128 .. of this head
    // into K stage kst / V stage vst
    auto load_rows = [&](void* dst, const CUtensorMap* m, int x, int row, uint64_t* bar) {
        tma_load_2d(dst, m, x, bh * N + row, bar);
    };
    auto load_k = [&](int t, int kst) {
        uint8_t* sk = sm + C::K_OFF + kst * C::SPLIT * C::TILE_BYTES;
        mbar_arrive_expect_tx(&k_full[kst], C::SPLIT * C::TILE_BYTES);
        for (int r = 0; r < C::NREG; ++r) {
            load_rows(sk + r * 16384, &tmK, r * C::BOXC, t * kTile, &k_full[kst]);
            if constexpr (TF32)
                tma_load_2d(sk + C::TILE_BYTES + r * 16384, &tmKlo, r * C::BOXC, bh * N + t * kTile, &k_full[kst]);
        }
    };
    auto load_v = [&](int t, int vst) {
        uint8_t* sv = sm + C::V_OFF + vst * C::TILE_BYTES;
        mbar_arrive_expect_tx(&v_full[vst], C::TILE_BYTES);
        if constexpr (!TF32) {
            for (int r = 0; r < C::NREG; ++r) load_rows(sv + r * 16384, &tmV, r * C::BOXC, t * kTile, &v_full[vst]);
        } else {
            // V^T [d][keys]: four 32-key swizzle regions of [d][32]
            for (int r = 0; r < 4; ++r) tma_load_2d(sv + r * D * 128, &tmV, t * kTile + r * 32, bh * D, &v_full[vst]);
        }
    };
    int t_early = -1;  // key tile whose K and V the set-up thread requested

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
            for (int k = 0; k < 3; ++k) mbar_init(&p_half[i * 3 + k], 128);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(drain, 1);
        fence_barrier_init();
        // Both Q tiles are requested at once, by the thread that set up the
        // barriers (the producer), before TMEM allocation and the CTA-wide
        // barrier: the Q and first K loads are the CTA's start-up latency.
        mbar_arrive_expect_tx(bar_q, (act1 ? 2 : 1) * C::SPLIT * C::TILE_BYTES);
        for (int s = 0; s < (act1 ? 2 : 1); ++s)
            for (int r = 0; r < C::NREG; ++r) {
                uint8_t* dq = sm + C::Q_OFF + s * C::SPLIT * C::TILE_BYTES + r * 16384;
                tma_load_2d(dq, &tmQ, r * C::BOXC, bh * N + (qb0 + s) * kTile, bar_q);
                if constexpr (TF32)
                    tma_load_2d(dq + C::TILE_BYTES, &tmQlo, r * C::BOXC, bh * N + (qb0 + s) * kTile, bar_q);
            }
        // ... and so are the first needed tile's K and V (the rings start
        // empty)
        {
            int t0 = 0;
            while (t0 < hi && !tile_visible(p.mask, qb0, t0, kvalid) && !(act1 && tile_visible(p.mask, qb1, t0, kvalid)))
                ++t0;
            if (t0 < hi) {
                load_k(t0, 0);
                load_v(t0, 0);
                t_early = t0;
            }
        }
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        if constexpr (TF32) {
            tma_prefetch_desc(&tmQlo);
            tma_prefetch_desc(&tmKlo);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    const MaskArgs mk = p.mask;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tmem_slot;

    // which Q tiles of this CTA need key tile t (bit s = Q tile s)
    // (captured by value: a by-reference capture would give these variables
    // addresses and move them to local memory)
    auto need_of = [=](int t) -> uint32_t {
        uint32_t nd = tile_visible(mk, qb0, t, kvalid) ? 1u : 0u;
        if (act1 && tile_visible(mk, qb1, t, kvalid)) nd |= 2u;
        return nd;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // K and V tiles whose loads were issued (the first one possibly
            // by the set-up code above)
            int nk = t_early >= 0 ? 1 : 0, nv = nk;
            for (int t = t_early + 1; t < hi; ++t) {
                if (!need_of(t)) continue;
                const int kst = nk % C::KSTAGES;
                if (!mbar_wait(&k_empty[kst], ((nk / C::KSTAGES) & 1) ^ 1, cx, 1)) break;
                load_k(t, kst);
                ++nk;
                const int vst = nv % C::VSTAGES;
                if (!mbar_wait(&kv_empty[vst], ((nv / C::VSTAGES) & 1) ^ 1, cx, 9)) break;
                load_v(t, vst);
                ++nv;
            }
            // let every copy in flight land before the CTA can exit
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
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs the loop; one elected lane issues
        {
            const uint32_t leader = elect_one_sync();
            bool ok = mbar_wait_warp(bar_q, 0, cx, 2);
            if (ok) tc_fence_after();
            MmaState st;
            // descriptors are built once and advanced by constants per k-step
            const uint64_t dQ0 = sdesc_sw128(smem_u32(sm + C::Q_OFF), 16, 1024);
            const uint64_t dK0 = sdesc_sw128(smem_u32(sm + C::K_OFF), 16, 1024);
            // bf16: V MN-major (LBO = distance between 64-column regions);
            // tf32: V^T K-major
            const uint64_t dV0 = sdesc_sw128(smem_u32(sm + C::V_OFF), TF32 ? 16 : 16384, 1024);
#define issue_pv(S) fwd_issue_pv<TF32, D, PV_PARTS>(leader, (S), st, tm, dV0, p_half, p_full, v_full, kv_empty, cx)
            int (&pend_stage)[2] = st.pend_stage;
            uint32_t(&pend_ph)[2] = st.pend_ph;
            uint32_t& rem = st.rem;

            int u = 0;
            for (int t = 0; ok && t < hi; ++t) {
                const uint32_t nd = need_of(t);
                if (!nd) continue;
                const int kst = u % C::KSTAGES;
                const int vst = u % C::VSTAGES;
                const uint32_t vph = (u / C::VSTAGES) & 1;
                // The producer issues K of tile u only after V of tile u - 1,
                // which waits for every P V reading tile u - 1 - VSTAGES, and
                // tile u reuses the V stage (and its reader count) of tile
                // u - VSTAGES: a P V still pending for a tile that old (its Q
                // tile skipped the tiles since) is issued first.
#pragma unroll
                for (int s = 0; s < 2; ++s)
                    if (ok && pend_stage[s] >= 0 && st.pend_u[s] <= u - C::VSTAGES && !issue_pv(s)) ok = false;
                if (!ok) break;
                if (!mbar_wait_warp(&k_full[kst], (u / C::KSTAGES) & 1, cx, 5)) { ok = false; break; }
                tc_fence_after();
                rem = (rem & ~(3u << (2 * vst))) | ((uint32_t)__popc(nd) << (2 * vst));
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    if (!(nd & (1u << s))) continue;
                    if (pend_stage[s] >= 0 && !issue_pv(s)) { ok = false; break; }
                    const uint64_t qs = sdesc_advance(dQ0, s * C::SPLIT * C::TILE_BYTES);
                    const uint64_t ks = sdesc_advance(dK0, kst * C::SPLIT * C::TILE_BYTES);
                    // bf16: one product; fp32: (Qh, Kh), (Qh, Kl), (Ql, Kh)
#pragma unroll
                    for (int part = 0; part < (TF32 ? 3 : 1); ++part) {
                        const uint64_t qa = sdesc_advance(qs, part == 2 ? C::TILE_BYTES : 0);
                        const uint64_t kb2 = sdesc_advance(ks, part == 1 ? C::TILE_BYTES : 0);
#pragma unroll
                        for (int kk = 0; kk < C::S_KSTEPS; ++kk) {
                            const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                            umma_ss<TF32>(leader, tm + s * 256, sdesc_advance(qa, off), sdesc_advance(kb2, off), C::ID_S,
                                          (part > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit(leader, &s_full[s]);
                    pend_stage[s] = vst;
                    pend_ph[s] = vph;
                    st.pend_u[s] = u;
                }
                if (!ok) break;
                umma_commit(leader, &k_empty[kst]);  // S GEMMs reading this K stage are all issued
                ++u;
            }
            // one commit per Q tile after its last P V: the epilogue waits on
            // it. Q tile 0 usually finishes a tile earlier (with a causal
            // mask Q tile 1 alone sees the last key tile), so its commit goes
            // out before Q tile 1's last P V waits for its probabilities.
            for (int s = 0; ok && s < 2; ++s) {
                if (pend_stage[s] >= 0 && !issue_pv(s)) ok = false;
                if (ok) umma_commit(leader, &o_done[s]);
            }
#undef issue_pv
            // wait for every MMA issued so far before TMEM can be released
            umma_commit(leader, drain);
            mbar_wait_teardown(drain, 0, 200000000ull);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax
        const int s = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int r = wq * 32 + lane;
        const bool active = (s == 0) || act1;
        const int qb = s == 0 ? qb0 : qb1;
        const int grow = qb * kTile + r;  // query row within the sequence
        const uint32_t tl = tm + (static_cast<uint32_t>(wq * 32) << 16) + s * 256;
        const float c2 = p.scale_log2;
        // l: running sum of the fp32 probabilities (gives L); lw: running sum
        // of the same probabilities rounded to the bf16 weights that the P V
        // product multiplies (normalises O)
        float m_hat = -CUDART_INF_F, l = 0.f, lw = 0.f;
        int n = 0;
        bool ok = true;
        if (active) {
            for (int t = 0; t < hi; ++t) {
                const uint32_t nd = need_of(t);
                if (!(nd & (1u << s))) continue;
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
                const float m_new = fmaxf(m_hat, mx * c2);
                const bool resc = (m_new - m_hat) > kRescaleThreshold;
                float alpha = 1.f;
                if (resc) {
                    alpha = ex2_approx(m_hat - m_new);
                    m_hat = m_new;
                    l *= alpha;
                    lw *= alpha;
                }
                const float mu = (m_hat == -CUDART_INF_F) ? 0.f : m_hat;
                float rs = 0.f, rr = 0.f;
                // two elements per f32x2 instruction: x = s * c2 - mu, the
                // fp32 row sum and the sum of the bf16-rounded weights
                const uint64_t c2c2 = f2_make(c2, c2), nmu2 = f2_make(-mu, -mu);
                // O is rescaled (below) before any P V of this tile may run
                const bool resc_any = __any_sync(0xffffffffu, resc) && n > 0;
                uint64_t rs2 = 0ull;
                uint64_t rr2d = 0ull;  // dropout: bf16-weight sum, formed before the weights are masked
                uint32_t pk[4][16];  // P as bf16 pairs; kept for the bf16-weight sum
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if constexpr (!TF32) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float x0, x1;
                            f2_split(f2_fma(f2_make(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])),
                                            c2c2, nmu2),
                                     x0, x1);
                            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                            pk[c][i] = pack_bf16x2(p0, p1);
                            rs2 = f2_add(rs2, f2_make(p0, p1));
                        }
                        if constexpr (DROPOUT) {
                            // the normaliser sums every weight; dropout then
                            // zeroes the dropped ones before the P V product
#pragma unroll
                            for (int i = 0; i < 16; ++i) rr2d = f2_add(rr2d, f2_from_bf16x2(pk[c][i]));
                            const int s4 = lane & 3;
#pragma unroll
                            for (int g4 = 0; g4 < 2; ++g4) {
                                // this lane's call: key block g4 * 4 + s4 of the chunk
                                const uint32_t kb = static_cast<uint32_t>((t * kTile + c * 32) >> 2) + g4 * 4 + s4;
                                const uint4 w = quad_transpose(
                                    philox4x32_10(make_uint4(static_cast<uint32_t>(grow) >> 2, kb,
                                                             static_cast<uint32_t>(h), static_cast<uint32_t>(b)),
                                                  p.drop.seed_lo, p.drop.seed_hi),
                                    s4);
                                const uint32_t kw[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                for (int n4 = 0; n4 < 4; ++n4) {
                                    uint32_t lo, hi;
                                    keep_masks16(kw[n4], p.drop.t4, lo, hi);
                                    pk[c][2 * (g4 * 4 + n4)] &= lo;
                                    pk[c][2 * (g4 * 4 + n4) + 1] &= hi;
                                }
                            }
                        }
                        tmem_st16(tl + c * 16, pk[c]);
                        if (c < 3 && (c + 1) % (4 / PV_PARTS) == 0 && !resc_any) {
                            tmem_st_wait();
                            tc_fence_before();
                            mbar_arrive(&p_half[s * 3 + (c + 1) / (4 / PV_PARTS) - 1]);
                        }
                    } else {
                        uint32_t pk[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c][i]), c2, -mu));
                            rs += p0;
                            pk[i] = __float_as_uint(p0);
                        }
                        rr = rs;
                        tmem_st32(tl + c * 32, pk);
                        if (c < 3 && (c + 1) % (4 / PV_PARTS) == 0 && !resc_any) {
                            tmem_st_wait();
                            tc_fence_before();
                            mbar_arrive(&p_half[s * 3 + (c + 1) / (4 / PV_PARTS) - 1]);
                        }
                    }
                }
                if constexpr (TF32) {
                    l += rs;
                    lw += rr;
                }
                tmem_st_wait();
                // Row sums of this tile: fp32 probabilities (for L) and their
                // bf16 roundings, the weights P V uses (for O). They are not
                // needed before the next tile, so in the usual case they are
                // formed after P has been handed to the MMA thread.
                if constexpr (!TF32) {
                    float a_, b_;
                    f2_split(rs2, a_, b_);
                    l += a_ + b_;
                }
                // The sum of the bf16-rounded weights (what P V multiplies; it
                // normalises O) is not needed before the next tile: in the usual
                // case it is formed after P has been handed to the MMA thread.
#define FA_ROW_SUMS()                                                                                     \
    do {                                                                                                  \
        if constexpr (DROPOUT) {                                                                          \
            float a_, b_;                                                                                 \
            f2_split(rr2d, a_, b_);                                                                       \
            lw += a_ + b_;                                                                                \
        } else if constexpr (!TF32) {                                                                     \
            uint64_t rr2 = 0ull;                                                                          \
            _Pragma("unroll") for (int c = 0; c < 4; ++c) _Pragma("unroll") for (int i = 0; i < 16; ++i)    \
                rr2 = f2_add(rr2, f2_from_bf16x2(pk[c][i]));                                              \
            float a_, b_;                                                                                 \
            f2_split(rr2, a_, b_);                                                                        \
            lw += a_ + b_;                                                                                \
        }                                                                                                 \
    } while (0)
                if (resc_any) {
                    FA_ROW_SUMS();
                    // O holds the previous tiles' sum; their last P V was issued
                    // before this tile's S, and MMAs complete in issue order,
                    // so S being complete means O is final: rescale it to the
                    // new reference maximum.
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(tl + 128 + c * 32, ov);
                        tmem_ld_wait(ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                        tmem_st32(tl + 128 + c * 32, ov);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    for (int k = 0; k < PV_PARTS - 1; ++k) mbar_arrive(&p_half[s * 3 + k]);
                    if (!FA_DROP_THIS_ARRIVE(n == 0)) mbar_arrive(&p_full[s]);
                } else {
                    tc_fence_before();
                    if (!FA_DROP_THIS_ARRIVE(n == 0)) mbar_arrive(&p_full[s]);
                    FA_ROW_SUMS();
                }
#undef FA_ROW_SUMS
                ++n;
            }
            // ------------------------------------------------------------ epilogue
            if (ok && n > 0) {
                ok = mbar_wait(&o_done[s], 0, cx, 8);
                ok = __all_sync(0xffffffffu, ok);
                if (ok) tc_fence_after();
            }
            if (ok) {
                float inv = lw > 0.f ? 1.f / lw : 0.f;
                if constexpr (DROPOUT) inv *= p.drop.inv_keep;
                const size_t orow = (static_cast<size_t>(bh) * N + grow) * D;
                const size_t lrow = static_cast<size_t>(bh) * N + grow;
                // bf16: a warp stages its 32 rows in its Q tile's buffer (every
                // S GEMM is complete once o_done is), in the 128-byte swizzled
                // layout of [32 x 64] boxes, and stores them with one bulk
                // tensor copy per box; a store per thread and row would touch
                // 32 rows (cache lines) per instruction. A Q tile that saw no
                // key tile (n == 0: nothing waited for its Q load, which may
                // still be landing in the buffer) stores its rows directly.
                const int wrow0 = qb * kTile + wq * 32;
                const bool tma_rows = !TF32 && n > 0 && wrow0 + 32 <= N;
                uint8_t* ob = sm + C::Q_OFF + s * C::SPLIT * C::TILE_BYTES + wq * (C::NREG * 4096);
                // all of O's TMEM loads in flight before the first wait
                uint32_t oa[D / 32][32];
                if (n > 0) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) tmem_ld32(tl + 128 + c * 32, oa[c]);
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
                    if constexpr (!TF32) {
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
                    } else {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + orow + c * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(ov[4 * j]) * inv, __uint_as_float(ov[4 * j + 1]) * inv,
                                                 __uint_as_float(ov[4 * j + 2]) * inv,
                                                 __uint_as_float(ov[4 * j + 3]) * inv);
                    }
                }
                if (tma_rows) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int rg = 0; rg < C::NREG; ++rg)
                            tma_store_2d(&tmO, rg * C::BOXC, bh * N + wrow0, ob + rg * 4096);
                        bulk_commit_group();
                        // the shared buffer must be read out before the CTA exits
                        bulk_wait_group_read0();
                    }
                }
                p.lse[lrow] = l > 0.f ? (m_hat + log2f(l)) * kLn2 : -CUDART_INF_F;
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

// fp32 inputs: x = hi + lo with hi = x with its 13 low mantissa bits cleared
// (exactly representable in tf32) and lo = x - hi (exact in fp32, |lo| <
// 2^-10 |x|), so that products of tf32 parts recover S to about fp32 accuracy.
__global__ void fa_split_tf32_kernel(const float4* __restrict__ x, float4* __restrict__ hi, float4* __restrict__ lo,
                                     long long n4) {
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float4 a = x[i];
        float4 h;
        h.x = __uint_as_float(__float_as_uint(a.x) & 0xFFFFE000u);
        h.y = __uint_as_float(__float_as_uint(a.y) & 0xFFFFE000u);
        h.z = __uint_as_float(__float_as_uint(a.z) & 0xFFFFE000u);
        h.w = __uint_as_float(__float_as_uint(a.w) & 0xFFFFE000u);
        hi[i] = h;
        lo[i] = make_float4(a.x - h.x, a.y - h.y, a.z - h.z, a.w - h.w);
    }
}

// V [BH][N][d] fp32 -> V^T [BH][d][N] (tf32 operands of tcgen05 must be K-major)
__global__ void fa_transpose_v_kernel(const float* __restrict__ v, float* __restrict__ vt, int N, int D) {
    __shared__ float tile[32][33];
    const int bh = blockIdx.z;
    const int n0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
    const float* src = v + static_cast<size_t>(bh) * N * D;
    float* dst = vt + static_cast<size_t>(bh) * N * D;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) tile[i][threadIdx.x] = src[(size_t)(n0 + i) * D + d0 + threadIdx.x];
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) dst[(size_t)(d0 + i) * N + n0 + threadIdx.x] = tile[threadIdx.x][i];
}

template <bool TF32, int D>
static cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream, int* nlaunch) {
    using C = FwdCfg<TF32, D>;
    const int elem = TF32 ? 4 : 2;
    const uint64_t rows = static_cast<uint64_t>(a.B) * a.H * a.N;
    CUtensorMap tq, tk, tv, tql, tkl, to;
    int launches = 0;
    if constexpr (TF32) {
        // scratch: V^T, Qh, Ql, Kh, Kl (each [B,H,N,d] fp32)
        const size_t n = rows * D;
        float* vt = static_cast<float*>(a.fp32_scratch);
        float *qh = vt + n, *ql = qh + n, *kh = ql + n, *kl = kh + n;
        dim3 g(a.N / 32, D / 32, a.B * a.H);
        fa_transpose_v_kernel<<<g, dim3(32, 8), 0, stream>>>(static_cast<const float*>(a.v), vt, a.N, D);
        const long long n4 = static_cast<long long>(n / 4);
        const unsigned blocks = static_cast<unsigned>(n4 < 152 * 32 * 256 ? (n4 + 255) / 256 : 152 * 32);
        fa_split_tf32_kernel<<<blocks, 256, 0, stream>>>(static_cast<const float4*>(a.q), reinterpret_cast<float4*>(qh),
                                                         reinterpret_cast<float4*>(ql), n4);
        fa_split_tf32_kernel<<<blocks, 256, 0, stream>>>(static_cast<const float4*>(a.k), reinterpret_cast<float4*>(kh),
                                                         reinterpret_cast<float4*>(kl), n4);
        launches += 3;
        if (!make_tmap_2d_sw128(&tv, vt, static_cast<uint64_t>(a.B) * a.H * D, a.N, elem, D, C::BOXC) ||
            !make_tmap_2d_sw128(&tq, qh, rows, D, elem, kTile, C::BOXC) ||
            !make_tmap_2d_sw128(&tql, ql, rows, D, elem, kTile, C::BOXC) ||
            !make_tmap_2d_sw128(&tk, kh, rows, D, elem, kTile, C::BOXC) ||
            !make_tmap_2d_sw128(&tkl, kl, rows, D, elem, kTile, C::BOXC))
            return cudaErrorInvalidValue;
    } else {
        // O is stored in [32 rows x 64 columns] boxes, one per warp and region
        if (!make_tmap_2d_sw128(&tq, a.q, rows, D, elem, kTile, C::BOXC) ||
            !make_tmap_2d_sw128(&tk, a.k, rows, D, elem, kTile, C::BOXC) ||
            !make_tmap_2d_sw128(&tv, a.v, rows, D, elem, kTile, C::BOXC) ||
            !make_tmap_2d_sw128(&to, a.o, rows, D, elem, 32, C::BOXC))
            return cudaErrorInvalidValue;
        tql = tq;
        tkl = tk;
    }
    if constexpr (TF32) to = tq;  // unused: fp32 O is stored directly
    // bf16 calls reach this kernel only with dropout ([B, H, N, d]); the
    // others run fa_fwd_t1.cu
    if (!TF32 && (a.cu_seqlens || !a.dropout)) return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e;
        if constexpr (TF32) {
            e = cudaFuncSetAttribute(fa_fwd_kernel<true, D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::SMEM);
        } else {
            e = cudaFuncSetAttribute(fa_fwd_kernel<false, D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::SMEM);
        }
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    FwdParams p;
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
    const int T = (a.N + kTile - 1) / kTile;
    p.head_major = (a.blockmask && !a.causal) ? 1 : 0;
    // causal calls: head groups whose K and V take at most 64 MiB
    p.group = 0;
    if (a.causal) {
        const long long per_head = 2LL * a.N * D * elem;
        long long g = (64LL << 20) / per_head;
        g = g < 1 ? 1 : g;
        p.group = static_cast<int>(g < a.B * a.H ? g : a.B * a.H);
    }
    const dim3 grid = p.group > 0     ? dim3(static_cast<unsigned>((T + 1) / 2) * a.H * a.B)
                      : p.head_major ? dim3((T + 1) / 2, a.H, a.B)
                                     : dim3(a.H, a.B, (T + 1) / 2);
    if (a.ev_begin) cudaEventRecord(a.ev_begin, stream);
    p.drop = a.drop;
    if constexpr (TF32)
        fa_fwd_kernel<true, D, false><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tql, tkl, to, p);
    else
        fa_fwd_kernel<false, D, true><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tql, tkl, to, p);
    if (a.ev_end) cudaEventRecord(a.ev_end, stream);
    ++launches;
    *nlaunch = launches;
    return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream, int* nlaunch) {
    // bf16 calls without dropout ([B, H, N, d] or packed): one query tile per
    // CTA, two CTAs per SM (fa_fwd_t1.cu); this file's pair kernel serves
    // fp32 inputs and dropout
    if (!a.fp32 && !a.dropout) return launch_fwd_bf16_t1(a, stream, nlaunch);
    if (a.fp32) {
        if (a.d == 64) return launch_fwd_t<true, 64>(a, stream, nlaunch);
        return cudaErrorInvalidValue;  // fp32 d=128 exceeds the shared-memory budget of this kernel
    }
    if (a.d == 64) return launch_fwd_t<false, 64>(a, stream, nlaunch);
    return launch_fwd_t<false, 128>(a, stream, nlaunch);
}

}  // namespace fa

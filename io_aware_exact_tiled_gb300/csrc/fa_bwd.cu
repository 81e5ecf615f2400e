// Backward pass of fused, tiled, exact softmax attention on sm_103a.
//
// What it computes ("FlashAttention: making attention IO-aware", section
// "The backward pass: recompute, don't store"): the forward pass kept only O
// and L = m + log l. Each score tile is recomputed from Q and K, the
// probabilities come back already normalised as P = exp(S - L), and the
// softmax-gradient row sum is the closed form D = rowsum(dO * O). With these,
// the gradients of <dO, O> are (textbook derivative of the definition):
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q,
// and no N x N matrix is written to device memory.
//
// Kernels (all on the caller's stream):
//   fa_bwd_pre_kernel   D = rowsum(dO * O) (fp32, shuffle reduction over the
//                       threads that share a row) and zeroing of the fp32 dQ
//                       accumulator
//   fa_bwd_kernel       one CTA per (batch, head, 128-key block j): K_j and
//                       V_j stay in shared memory while the query blocks i
//                       stream through a two-stage TMA ring; five tcgen05
//                       GEMMs per tile with dK_j and dV_j accumulated in TMEM;
//                       dQ_i = dS K_j is added into the fp32 accumulator with
//                       TMA bulk reduce-adds staged through shared memory;
//                       dK_j, dV_j are staged in shared memory at the end and
//                       leave through TMA stores (coalesced stores in the
//                       tile-masked instance)
//   fa_bwd_dq_kernel    fp32 dQ accumulator -> dQ in bf16
//
// TMEM columns of fa_bwd_kernel: two 128-column buffers in [0, 256) that
// alternate between query blocks (one holds S^T, then P^T (bf16), then dQ_i;
// the other dP^T); [256, 256+d) dV_j; [256+d, 256+2d) dK_j. The softmax
// scale is applied once, to dK_j in the epilogue and to dQ in the conversion
// kernel, instead of to every element of dS.
#include <math_constants.h>

#include "fa_common.cuh"
#include "fa_philox.cuh"
#include "fa_launch.h"
#include "tmap.h"

namespace fa {

// Query tiles per sequence up to which a tile-masked CTA keeps the visible
// query tiles of its key tile as a bitmap in shared memory (N <= 262,144);
// longer sequences read the tile mask in global memory tile by tile.
constexpr int kBwdVisMaxTiles = 2048;

template <int D>
struct BwdCfg {
    static constexpr int ROWB = D * 2;
    static constexpr int NREG = ROWB / 128;
    static constexpr int TILE_BYTES = kTile * ROWB;  // 128 rows of Q, K, V or dO
    static constexpr int STAGES = 2;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE_BYTES;
    static constexpr int Q_OFF = V_OFF + TILE_BYTES;                  // [STAGES]
    static constexpr int DO_OFF = Q_OFF + STAGES * TILE_BYTES;        // [STAGES]
    static constexpr int DS_OFF = DO_OFF + STAGES * TILE_BYTES;       // dS^T, 128 x 128 bf16
    static constexpr int LSE_OFF = DS_OFF + 32768;                    // [STAGES][128] fp32
    static constexpr int DEL_OFF = LSE_OFF + STAGES * 512;            // [STAGES][128] fp32
    static constexpr int BAR_OFF = DEL_OFF + STAGES * 512;
    static constexpr int VIS_OFF = BAR_OFF + 256;                     // visible query tiles (tile mask)
    static constexpr int VIS_WORDS = kBwdVisMaxTiles / 32;
    static constexpr int USED = VIS_OFF + VIS_WORDS * 4;
    static constexpr int SMEM = USED + 1024 <= 232448 ? USED + 1024 : 232448;
    static constexpr int THREADS = 512;
    static constexpr uint32_t ID_SQ = idesc_make(128, 128, kFmtBF16, false, false);  // S^T, dP^T
    static constexpr uint32_t ID_KN = idesc_make(128, D, kFmtBF16, false, true);     // dV, dK
    static constexpr uint32_t ID_DQ = idesc_make(128, D, kFmtBF16, true, true);      // dQ
    // Columns [0, 256) are two 128-column buffers that trade roles every
    // query block u: S^T (then P^T, then dQ_u) goes to buffer u % 2 and dP^T
    // to the other one (col_s / col_dp below). S^T of block u + 1 can then be
    // issued right after dQ_u, without waiting for the drain to read dQ_u;
    // the wait moves to dP^T of block u + 1, which is needed only later.
    static constexpr int COL_DV = 256, COL_DK = 256 + D;
};

struct BwdParams {
    int B, H, N;
    float scale;
    float scale_log2;
    MaskArgs mask;
    const float* nlse2;   // -L * log2(e) (-inf where L = -inf, so that P = 0)
    const float* ndelta;  // -D = -rowsum(dO * O)
    void* dk;
    void* dv;
    int* status;
    const int32_t* cu_seqlens;  // packed variable-length batch, else null
    const int32_t* cu_tiles;    // [B + 1] running 128-row tile counts (packed)
    int total;                  // tokens of the packed batch
    long long lpad;             // rows per head of nlse2 / ndelta (packed)
    DropoutArgs drop;           // dropout on the probabilities (DROPOUT kernel)
    int group;                  // > 0: causal head-group order on a 1D grid (heads per group)
};

constexpr float kLog2e = 1.4426950408889634f;

// Warp roles (512 threads):
//   thread 0      sets up the mbarriers and requests K_j, V_j and the first
//                 stage before the CTA-wide barrier
//   warp 0        TMA producer (the remaining Q_i, dO_i, L_i, D_i stages)
//   warp 1        TMEM allocation; the whole warp runs the issue loop and one
//                 elected lane issues the MMAs
//   warps 2-3     tile-masked kernel only: gather the mask column into a bitmap
//   warps 4-7     compute group 0: thread r owns key r, queries 0-63 of block i
//   warps 8-11    compute group 1: key r, queries 64-127
//   warps 12-15   dQ drain: thread r owns query r of block i
// Per query block i the MMA thread issues, in this order:
//   S^T  = K_j Q_i^T   (into the buffer that held dP^T of the previous block)
//   dP^T = V_j dO_i^T  (after the drain has read dQ_{i-1} out of its buffer)
//   dV  += P^T dO_i    (P^T from TMEM, written by the compute groups)
//   dK  += dS^T Q_i, dQ_i = dS K_j  (dS^T from shared memory; the d = 128
//                      kernels without tile mask or packing issue dQ_i first)
// VARLEN: packed variable-length batch; a separate instantiation so that the
// [B, H, N, d] kernel carries none of its branches.
// DROPOUT: the keep mask of the forward pass is regenerated (fa_philox.cuh);
// P^T masked by it feeds dV, the unmasked P^T (kept in the free half of the
// buffer's columns) feeds dS.
// TMASK: calls with a tile mask; the visible-tile bitmap and the jumps over
// masked query tiles live only in this instantiation.
template <int D, bool VARLEN, bool DROPOUT = false, bool TMASK = false>
__global__ void __launch_bounds__(512, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQacc, const __grid_constant__ CUtensorMap tmdK,
                  const __grid_constant__ CUtensorMap tmdV, const __grid_constant__ BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base for the swizzled tiles; offsetting the shared
    // array itself (rather than casting through an integer) keeps the pointer
    // in the shared address space, so accesses compile to shared loads/stores
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The carve-up needs the dynamic shared window to start within the slack
    // reserved for alignment; report instead of overrunning if it does not.
    if ((sm - smem_raw) + C::USED > C::SMEM) {
        if (tid == 0 && p.status) atomicCAS(p.status, 0, FA_DEV_TIMEOUT | (99 << 8));
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
    uint64_t* kv_full = bars + 0;
    uint64_t* qd_full = bars + 1;                 // [STAGES]
    uint64_t* qd_empty = qd_full + C::STAGES;     // [STAGES]
    uint64_t* s_full = qd_empty + C::STAGES;
    uint64_t* dp_full = s_full + 1;
    uint64_t* p_ready = dp_full + 1;
    uint64_t* ds_ready = p_ready + 1;
    uint64_t* dq_full = ds_ready + 1;
    uint64_t* dq_free = dq_full + 1;
    uint64_t* dkv_done = dq_free + 1;
    uint64_t* drain = dkv_done + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // barriers of the plain d = 128 kernel only (kSplitStage, kDqFirst), after
    // the others so that every instance keeps the same layout for those
    uint64_t* do_full = reinterpret_cast<uint64_t*>(tmem_slot + 2);  // [STAGES] dO_i and -D of a stage landed
    uint64_t* dk_done = do_full + C::STAGES;                          // dK_j += dS^T Q_i of a block complete
    const WaitCtx cx{abort_flag, p.status};

    // Head-major order: the key blocks of one head are adjacent in the grid
    // (j = 0, the longest causal column, first), so the CTAs running at any
    // time share the Q, dO and dQ-accumulator rows of a few heads in L2.
    // With a causal mask that order ends on the long columns of the last
    // heads; there the grid is 1D and runs groups of p.group heads in turn,
    // longest column first across the heads of a group (sized so that a
    // group's rows still fit in L2), so that the kernel ends on short CTAs.
    int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    if (p.group > 0) {
        const int Tg = p.mask.T, nb = p.B * p.H;
        const int L = static_cast<int>(blockIdx.x);
        const int gi = L / (p.group * Tg), r = L - gi * p.group * Tg;
        const int g0 = gi * p.group, gsz = min(p.group, nb - g0);
        j = r / gsz;
        const int bhx = g0 + (r - j * gsz);
        b = bhx / p.H;
        h = bhx - b * p.H;
    }
    // A packed variable-length batch puts sequence b at tokens seq0 ..
    // seq0 + N - 1 of [total, H, d] tensors; its rows of -L and -D start at
    // lrow0, a multiple of 128 (so that they can be bulk-copied). Key blocks
    // past the end of a shorter sequence leave at once.
    constexpr bool varlen = VARLEN;
    int N = p.N, T = p.mask.T, seq0 = 0;
    long long lrow0 = static_cast<long long>(b * p.H + h) * p.N;
    if (varlen) {
        const int s0 = min(max(p.cu_seqlens[b], 0), p.total);
        const int s1 = min(max(p.cu_seqlens[b + 1], s0), p.total);
        seq0 = s0;
        N = min(s1 - s0, p.N);
        T = (N + kTile - 1) / kTile;
        lrow0 = static_cast<long long>(h) * p.lpad + static_cast<long long>(p.cu_tiles[b]) * kTile;
    }
    if (j >= T) return;  // uniform over the CTA, before any barrier or TMEM use
    const int bh = b * p.H + h;
    const int kvalid = keys_valid(p.mask, b, N);
    const int lo = p.mask.causal ? j : 0;
    // captured by value (a by-reference capture would move them to local memory)
    const MaskArgs mk = p.mask;
    // With a tile mask every role would otherwise find the next visible query
    // tile by reading a column of the mask in global memory, a dependent load
    // (and a new cache line) per skipped tile; warps 2 and 3 (otherwise idle)
    // first gather the column into a bitmap (bit i: query tile i visible), and
    // the roles jump to the next visible tile with a find-first-set.
    constexpr bool kVis = TMASK && !VARLEN && !DROPOUT;
    const bool use_vis = kVis && mk.blockmask != nullptr && T <= kBwdVisMaxTiles;
    uint32_t* vis = reinterpret_cast<uint32_t*>(sm + C::VIS_OFF);
    auto visible_i = [=](int i) -> bool {
        if (kVis && use_vis) return (vis[i >> 5] >> (i & 31)) & 1u;
        return tile_visible(mk, i, j, kvalid);
    };
    // first query tile >= i that the walk visits: i itself except in the
    // tile-masked kernel, which jumps to the next visible one (or T)
    auto next_i = [=](int i) -> int {
        if constexpr (kVis) {
            if (use_vis) {
                while (i < T) {
                    const uint32_t w = vis[i >> 5] >> (i & 31);
                    if (w) return i + __ffs(w) - 1;
                    i = (i | 31) + 1;
                }
                return T;
            }
        }
        return i;
    };

    // K_j, V_j (once) and the Q_i, dO_i, -L, -D stage loads (producer thread)
    auto load_kv = [&]() {
        mbar_arrive_expect_tx(kv_full, 2 * C::TILE_BYTES);
        for (int r = 0; r < C::NREG; ++r) {
            if (varlen) {
                tma_load_3d(sm + C::K_OFF + r * 16384, &tmK, r * 64, h, seq0 + j * kTile, kv_full);
                tma_load_3d(sm + C::V_OFF + r * 16384, &tmV, r * 64, h, seq0 + j * kTile, kv_full);
            } else {
                tma_load_2d(sm + C::K_OFF + r * 16384, &tmK, r * 64, bh * N + j * kTile, kv_full);
                tma_load_2d(sm + C::V_OFF + r * 16384, &tmV, r * 64, bh * N + j * kTile, kv_full);
            }
        }
    };
    // In the plain [B, H, N, d] kernel at d = 128, Q_i and -L land on qd_full
    // and dO_i and -D on a barrier of their own, so that S^T and the P phase
    // can start before dO_i has landed (2.5 % faster on long4k and long8k);
    // the tile-masked (+5 %), packed (+3 %), dropout (+2 %) and d = 64
    // (+1.5-2.6 %) kernels were measured slower that way and keep one barrier
    // per stage.
    constexpr bool kSplitStage = !TMASK && !VARLEN && !DROPOUT && D == 128;
    // That kernel and the dropout one (d = 128) issue dQ_i before dK_i, so
    // that the drain starts one GEMM earlier: it stages the first half of dQ_i
    // in the dO_i tile (free once dV is complete) and the second half in the
    // Q_i tile only after dK_i, which reads Q_i, is complete; and the next
    // dS^T waits for dK_i (3 % faster plain, 1.2 % with dropout; the packed
    // kernel is unchanged by it and the tile-masked one 6 % slower).
    constexpr bool kDqFirst = D == 128 && !TMASK && !VARLEN;
    // The tile-masked kernel writes dK_j and dV_j out of their shared staging
    // with coalesced stores instead of bulk tensor stores (2 % faster there;
    // the other instances were as fast or slower that way).
    constexpr bool kDirectEpi = TMASK;
    auto load_stage = [&](int i, int st) {
        if constexpr (kSplitStage) {
            mbar_arrive_expect_tx(&qd_full[st], C::TILE_BYTES + 512);
            mbar_arrive_expect_tx(&do_full[st], C::TILE_BYTES + 512);
            const int row = bh * N + i * kTile;
            const long long lrow = lrow0 + static_cast<long long>(i) * kTile;
            for (int r = 0; r < C::NREG; ++r) {
                uint8_t* dq_s = sm + C::Q_OFF + st * C::TILE_BYTES + r * 16384;
                if (varlen)
                    tma_load_3d(dq_s, &tmQ, r * 64, h, seq0 + i * kTile, &qd_full[st]);
                else
                    tma_load_2d(dq_s, &tmQ, r * 64, row, &qd_full[st]);
            }
            bulk_load(sm + C::LSE_OFF + st * 512, p.nlse2 + lrow, 512, &qd_full[st]);
            for (int r = 0; r < C::NREG; ++r) {
                uint8_t* ddo_s = sm + C::DO_OFF + st * C::TILE_BYTES + r * 16384;
                if (varlen)
                    tma_load_3d(ddo_s, &tmdO, r * 64, h, seq0 + i * kTile, &do_full[st]);
                else
                    tma_load_2d(ddo_s, &tmdO, r * 64, row, &do_full[st]);
            }
            bulk_load(sm + C::DEL_OFF + st * 512, p.ndelta + lrow, 512, &do_full[st]);
            return;
        }
        mbar_arrive_expect_tx(&qd_full[st], 2 * C::TILE_BYTES + 1024);
        const int row = bh * N + i * kTile;
        for (int r = 0; r < C::NREG; ++r) {
            uint8_t* dq_s = sm + C::Q_OFF + st * C::TILE_BYTES + r * 16384;
            uint8_t* ddo_s = sm + C::DO_OFF + st * C::TILE_BYTES + r * 16384;
            if (varlen) {
                tma_load_3d(dq_s, &tmQ, r * 64, h, seq0 + i * kTile, &qd_full[st]);
                tma_load_3d(ddo_s, &tmdO, r * 64, h, seq0 + i * kTile, &qd_full[st]);
            } else {
                tma_load_2d(dq_s, &tmQ, r * 64, row, &qd_full[st]);
                tma_load_2d(ddo_s, &tmdO, r * 64, row, &qd_full[st]);
            }
        }
        const long long lrow = lrow0 + static_cast<long long>(i) * kTile;
        bulk_load(sm + C::LSE_OFF + st * 512, p.nlse2 + lrow, 512, &qd_full[st]);
        bulk_load(sm + C::DEL_OFF + st * 512, p.ndelta + lrow, 512, &qd_full[st]);
    };
    int i_early = -1;  // query block whose stage the set-up thread requested

    if (tid == 0) {
        *abort_flag = 0;
        mbar_init(kv_full, 1);
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&qd_full[s], 1);
            if constexpr (kSplitStage) mbar_init(&do_full[s], 1);
            mbar_init(&qd_empty[s], 4);  // the four dQ drain warps, done staging through it
        }
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        mbar_init(p_ready, 256);
        mbar_init(ds_ready, 256);
        mbar_init(dq_full, 1);
        mbar_init(dq_free, 128);
        mbar_init(dkv_done, 1);
        if constexpr (kDqFirst) mbar_init(dk_done, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
        // K, V and the first visible query block's stage are requested before
        // TMEM allocation and the CTA-wide barrier (the tile-masked kernel
        // finds its first block in the bitmap built after this)
        if constexpr (!TMASK) {
            int i0 = lo;
            while (i0 < T && !tile_visible(mk, i0, j, kvalid)) ++i0;
            if (i0 < T) {
                load_kv();
                load_stage(i0, 0);
                i_early = i0;
            }
        }
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
        tma_prefetch_desc(&tmdQacc);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    if (use_vis && (warp == 2 || warp == 3)) {
        const int nw = (T + 31) >> 5;
#pragma unroll 4
        for (int w = warp - 2; w < nw; w += 2) {
            const int i = w * 32 + lane;
            const uint32_t word = __ballot_sync(0xffffffffu, i >= lo && i < T && tile_visible(mk, i, j, kvalid));
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
            // the set-up code may have requested K, V and the first stage
            int u = i_early >= 0 ? 1 : 0;
            bool kv_issued = i_early >= 0;
            for (int i = next_i(i_early >= 0 ? i_early + 1 : lo); i < T; i = next_i(i + 1)) {
                if (!visible_i(i)) continue;
                if (!kv_issued) {
                    load_kv();
                    kv_issued = true;
                }
                const int st = u % C::STAGES;
                const uint32_t ph = (u / C::STAGES) & 1;
                if (!mbar_wait(&qd_empty[st], ph ^ 1, cx, 11)) break;
                load_stage(i, st);
                ++u;
            }
            if (kv_issued) mbar_wait_teardown(kv_full, 0, 200000000ull);
            for (int s = 0; s < C::STAGES && s < u; ++s) {
                const int last = s + ((u - 1 - s) / C::STAGES) * C::STAGES;
                mbar_wait_teardown(&qd_full[s], (last / C::STAGES) & 1, 200000000ull);
                if constexpr (kSplitStage) mbar_wait_teardown(&do_full[s], (last / C::STAGES) & 1, 200000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs the loop; one elected lane issues
        {
            const uint32_t leader = elect_one_sync();
            // descriptors are built once and advanced by constants per k-step
            const uint64_t dK_k = sdesc_sw128(smem_u32(sm + C::K_OFF), 16, 1024);        // K_j, K-major
            const uint64_t dV_k = sdesc_sw128(smem_u32(sm + C::V_OFF), 16, 1024);        // V_j, K-major
            const uint64_t dK_mn = sdesc_sw128(smem_u32(sm + C::K_OFF), 16384, 1024);    // K_j, MN-major
            const uint64_t dS_k = sdesc_sw128(smem_u32(sm + C::DS_OFF), 16, 1024);       // dS^T, K-major
            const uint64_t dS_mn = sdesc_sw128(smem_u32(sm + C::DS_OFF), 16384, 1024);   // dS, MN-major
            bool ok = true;
            int u = 0;
            for (int i = next_i(lo); ok && i < T; i = next_i(i + 1)) {
                if (!visible_i(i)) continue;
                if (u == 0) {
                    if (!(ok = mbar_wait_warp(kv_full, 0, cx, 12))) break;
                }
                const int st = u % C::STAGES;
                const uint32_t ph = (u / C::STAGES) & 1;
                if (!(ok = mbar_wait_warp(&qd_full[st], ph, cx, 13))) break;
                tc_fence_after();
                const uint32_t qb = smem_u32(sm + C::Q_OFF + st * C::TILE_BYTES);
                const uint32_t dob = smem_u32(sm + C::DO_OFF + st * C::TILE_BYTES);
                const uint64_t dQ_k = sdesc_sw128(qb, 16, 1024), dQ_mn = sdesc_sw128(qb, 16384, 1024);
                const uint64_t dO_k = sdesc_sw128(dob, 16, 1024), dO_mn = sdesc_sw128(dob, 16384, 1024);
                const uint32_t col_s = (u & 1) ? 128u : 0u, col_dp = col_s ^ 128u;
                // S^T = K_j Q_i^T (its buffer last held dP^T of the previous
                // block, read by the compute groups before they signalled
                // dS^T of that block, which the previous dK / dQ waited for)
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                    umma_ss<false>(leader, tm + col_s, sdesc_advance(dK_k, off), sdesc_advance(dQ_k, off), C::ID_SQ,
                                   kk > 0);
                }
                umma_commit(leader, s_full);
                // dP^T = V_j dO_i^T (its buffer held dQ of the previous block)
                if (u > 0 && !(ok = mbar_wait_warp(dq_free, (u - 1) & 1, cx, 14))) break;
                if (kSplitStage && !(ok = mbar_wait_warp(&do_full[st], ph, cx, 23))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                    umma_ss<false>(leader, tm + col_dp, sdesc_advance(dV_k, off), sdesc_advance(dO_k, off), C::ID_SQ,
                                   kk > 0);
                }
                umma_commit(leader, dp_full);
                // dV_j += P^T dO_i ; P^T of queries 0-63 sits in the buffer's
                // columns 0-31 and that of queries 64-127 in columns 64-95
                if (!(ok = mbar_wait_warp(p_ready, u & 1, cx, 15))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_ts<false>(leader, tm + C::COL_DV, tm + col_s + (kk >> 2) * 64 + (kk & 3) * 8,
                                   sdesc_advance(dO_mn, kk * 2048), C::ID_KN, (u > 0 || kk > 0) ? 1u : 0u);
                // dK_j += dS^T Q_i ; dQ_i = dS K_j
                if (!(ok = mbar_wait_warp(ds_ready, u & 1, cx, 16))) break;
                tc_fence_after();
                if constexpr (kDqFirst) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_ss<false>(leader, tm + col_s, sdesc_advance(dS_mn, kk * 2048), sdesc_advance(dK_mn, kk * 2048),
                                       C::ID_DQ, kk > 0 ? 1u : 0u);
                    umma_commit(leader, dq_full);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                        umma_ss<false>(leader, tm + C::COL_DK, sdesc_advance(dS_k, off), sdesc_advance(dQ_mn, kk * 2048),
                                       C::ID_KN, (u > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(leader, dk_done);
                } else {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk / 4) * 16384 + (kk % 4) * 32;
                        umma_ss<false>(leader, tm + C::COL_DK, sdesc_advance(dS_k, off), sdesc_advance(dQ_mn, kk * 2048), C::ID_KN,
                                       (u > 0 || kk > 0) ? 1u : 0u);
                    }
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        umma_ss<false>(leader, tm + col_s, sdesc_advance(dS_mn, kk * 2048), sdesc_advance(dK_mn, kk * 2048),
                                       C::ID_DQ, kk > 0 ? 1u : 0u);
                    umma_commit(leader, dq_full);
                }
                ++u;
            }
            if (ok && u > 0) umma_commit(leader, dkv_done);
            umma_commit(leader, drain);
            mbar_wait_teardown(drain, 0, 200000000ull);
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ P^T, dS^T (thread = key)
        const int g = (warp - 4) >> 2;       // query half: 64 g .. 64 g + 63
        const int r = (warp & 3) * 32 + lane;
        const uint32_t tl = tm + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const int key = j * kTile + r;
        const bool key_ok = key < kvalid;
        const uint64_t c2c2 = f2_make(p.scale_log2, p.scale_log2);
        const uint32_t ds_row = smem_u32(sm + C::DS_OFF + g * 16384 + r * 128);
        bool ok = true;
        int u = 0;
        for (int i = next_i(lo); i < T; i = next_i(i + 1)) {
            if (!visible_i(i)) continue;
            const int st = u % C::STAGES;
            const uint32_t ph = (u / C::STAGES) & 1;
            // -L log2 e and -D of this group's 64 queries (shared memory; plain
            // loads, so that the compiler may schedule them early)
            const float4* nlse_s = reinterpret_cast<const float4*>(sm + C::LSE_OFF + st * 512 + 256 * g);
            const float4* ndel_s = reinterpret_cast<const float4*>(sm + C::DEL_OFF + st * 512 + 256 * g);
            ok = mbar_wait(&qd_full[st], ph, cx, 17);
            ok = __all_sync(0xffffffffu, ok) && __all_sync(0xffffffffu, mbar_wait(s_full, u & 1, cx, 18));
            if (!ok) break;
            tc_fence_after();
            const uint32_t col_s = (u & 1) ? 128u : 0u, col_dp = col_s ^ 128u;
            // masking is needed only on the diagonal tile (causal), for
            // padded keys, and for the query rows of a packed sequence's last
            // block that lie past its end (they belong to the next sequence)
            const bool diag = p.mask.causal && i == j;
            const int qlim = varlen ? N - i * kTile : kTile;
            const bool masked = diag || !key_ok || qlim < kTile;
            uint32_t pu0[DROPOUT ? 16 : 1];  // dropout: unmasked P^T of the first 32 queries
            // both halves of S^T are requested before either is waited for
            uint32_t srs[2][32];
            tmem_ld32(tl + col_s + 64 * g, srs[0]);
            tmem_ld32(tl + col_s + 64 * g + 32, srs[1]);
            tmem_ld_wait(srs[0]);
            tmem_ld_wait(srs[1]);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t pk[16];  // P^T of 32 queries, bf16 pairs
                uint32_t(&sr)[32] = srs[c];
                uint32_t kw[DROPOUT ? 8 : 1];  // keep bytes of this key for the chunk's 32 queries
                if constexpr (DROPOUT) {
                    const int s4 = lane & 3;
#pragma unroll
                    for (int m4 = 0; m4 < 2; ++m4) {
                        // this lane's call: query block m4 * 4 + s4 of the chunk
                        const uint32_t qblk = static_cast<uint32_t>((i * kTile + 64 * g + c * 32) >> 2) + m4 * 4 + s4;
                        const uint4 w = quad_transpose(
                            byte_transpose(philox4x32_10(make_uint4(qblk, static_cast<uint32_t>(key) >> 2,
                                                                    static_cast<uint32_t>(h), static_cast<uint32_t>(b)),
                                                         p.drop.seed_lo, p.drop.seed_hi)),
                            s4);
                        kw[m4 * 4 + 0] = w.x;
                        kw[m4 * 4 + 1] = w.y;
                        kw[m4 * 4 + 2] = w.z;
                        kw[m4 * 4 + 3] = w.w;
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    // x = S * scale * log2(e) - L * log2(e), two queries per instruction
                    const float4 nL = nlse_s[c * 8 + e];
                    float x0, x1, x2, x3;
                    f2_split(f2_fma(f2_make(__uint_as_float(sr[4 * e]), __uint_as_float(sr[4 * e + 1])), c2c2,
                                    f2_make(nL.x, nL.y)), x0, x1);
                    f2_split(f2_fma(f2_make(__uint_as_float(sr[4 * e + 2]), __uint_as_float(sr[4 * e + 3])), c2c2,
                                    f2_make(nL.z, nL.w)), x2, x3);
                    float pv0 = ex2_approx(x0), pv1 = ex2_approx(x1), pv2 = ex2_approx(x2), pv3 = ex2_approx(x3);
                    if (masked) {
                        const int q = 64 * g + c * 32 + 4 * e;
                        if (!key_ok || (diag && q + 0 < r) || q + 0 >= qlim) pv0 = 0.f;
                        if (!key_ok || (diag && q + 1 < r) || q + 1 >= qlim) pv1 = 0.f;
                        if (!key_ok || (diag && q + 2 < r) || q + 2 >= qlim) pv2 = 0.f;
                        if (!key_ok || (diag && q + 3 < r) || q + 3 >= qlim) pv3 = 0.f;
                    }
                    pk[2 * e] = pack_bf16x2(pv0, pv1);
                    pk[2 * e + 1] = pack_bf16x2(pv2, pv3);
                }
                if constexpr (DROPOUT) {
                    uint32_t pz[16];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        uint32_t lo, hi;
                        keep_masks16(kw[e], p.drop.t4, lo, hi);
                        pz[2 * e] = pk[2 * e] & lo;
                        pz[2 * e + 1] = pk[2 * e + 1] & hi;
                    }
                    tmem_st16(tl + col_s + 64 * g + c * 16, pz);
                    // the unmasked P^T goes to columns 32-63 of the group,
                    // which hold the second chunk's scores until it is read
                    if (c == 0) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) pu0[e] = pk[e];
                    } else {
                        tmem_st16(tl + col_s + 64 * g + 32, pu0);
                        tmem_st16(tl + col_s + 64 * g + 48, pk);
                    }
                } else {
                    tmem_st16(tl + col_s + 64 * g + c * 16, pk);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            if (!FA_DROP_THIS_ARRIVE(u == 0)) mbar_arrive(p_ready);
            // dS^T = P^T * (dP^T - D) (the scale is applied to dK and dQ at
            // the end); P^T is read back from TMEM (bf16). The previous dS^T
            // must have been consumed by its dK / dQ GEMMs before this one is
            // written (long done by now: their completion released dQ_{i-1}
            // to the drain), so each half is stored as soon as it is formed.
            ok = __all_sync(0xffffffffu, mbar_wait(dp_full, u & 1, cx, 19) &&
                                             (!kSplitStage || mbar_wait(&do_full[st], ph, cx, 24)));
            if (ok && u > 0) ok = __all_sync(0xffffffffu, mbar_wait(kDqFirst ? dk_done : dq_full, (u - 1) & 1, cx, 20));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t dr[32], pk[16], pz[DROPOUT ? 16 : 1];
                tmem_ld32(tl + col_dp + 64 * g + c * 32, dr);
                if constexpr (DROPOUT) {
                    tmem_ld16(tl + col_s + 64 * g + 32 + c * 16, pk);  // unmasked P^T
                    tmem_ld16(tl + col_s + 64 * g + c * 16, pz);       // masked P^T (zero where dropped)
                    tmem_ld_wait(pz);
                } else {
                    tmem_ld16(tl + col_s + 64 * g + c * 16, pk);
                }
                tmem_ld_wait(dr);
                tmem_ld_wait(pk);
                if constexpr (DROPOUT) {
                    // dP of a dropped element is 0; a kept one is divided by the keep rate
                    const float ik = p.drop.inv_keep;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        dr[2 * e] = __float_as_uint(__uint_as_float(dr[2 * e]) * ((pz[e] & 0xFFFFu) ? ik : 0.f));
                        dr[2 * e + 1] = __float_as_uint(__uint_as_float(dr[2 * e + 1]) * ((pz[e] >> 16) ? ik : 0.f));
                    }
                }
                uint32_t dsw[16];
#pragma unroll
                for (int e = 0; e < 8; ++e) {  // 4 queries
                    const float4 nD = ndel_s[c * 8 + e];
                    const uint64_t t01 = f2_add(f2_make(__uint_as_float(dr[4 * e]), __uint_as_float(dr[4 * e + 1])),
                                                f2_make(nD.x, nD.y));
                    const uint64_t t23 = f2_add(f2_make(__uint_as_float(dr[4 * e + 2]), __uint_as_float(dr[4 * e + 3])),
                                                f2_make(nD.z, nD.w));
                    dsw[2 * e] = bf16x2_from_f2(f2_mul(t01, f2_from_bf16x2(pk[2 * e])));
                    dsw[2 * e + 1] = bf16x2_from_f2(f2_mul(t23, f2_from_bf16x2(pk[2 * e + 1])));
                }
#pragma unroll
                for (int chunk = 0; chunk < 4; ++chunk)  // 8 queries per 16-byte chunk
                    sts128(ds_row + (((c * 4 + chunk) ^ (r & 7)) * 16), dsw[4 * chunk], dsw[4 * chunk + 1],
                           dsw[4 * chunk + 2], dsw[4 * chunk + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(ds_ready);
            ++u;
        }
        // ------------------------------------------------------------ dK, dV epilogue
        // group 0 writes dV_j, group 1 writes dK_j = scale * (dS^T Q)
        if (ok && u > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(dkv_done, 0, cx, 21));
            if (ok) tc_fence_after();
        }
        if (ok) {
            // packed keys past the end of the sequence: read (the TMEM loads
            // are warp-wide) but not stored
            const bool row_ok = !varlen || key < N;
            const size_t orow = varlen ? (static_cast<size_t>(seq0 + key) * p.H + h) * D
                                       : (static_cast<size_t>(bh) * N + key) * D;
            uint16_t* out = static_cast<uint16_t*>(g == 0 ? p.dv : p.dk) + orow;
            const uint32_t col = g == 0 ? C::COL_DV : C::COL_DK;
            const float mul = g == 0 ? (DROPOUT ? p.drop.inv_keep : 1.f) : p.scale;
            // A warp whose 32 keys all lie in the sequence stages its rows in
            // the V (dV) or K (dK) tile buffer, free once every GEMM is
            // complete, as [32 x 64] swizzled boxes, and writes them with one
            // bulk tensor store per box (kDirectEpi: with coalesced stores of
            // its own); other warps (and a key tile that saw no query tile)
            // store their valid rows directly.
            const int wkey0 = j * kTile + (warp & 3) * 32;
            const bool tma_rows = u > 0 && wkey0 + 32 <= N;
            uint8_t* ob = sm + (g == 0 ? C::V_OFF : C::K_OFF) + (warp & 3) * (C::NREG * 4096);
            // two 32-column TMEM loads in flight at a time (128 registers a
            // thread at 512 threads leave no room for all of them)
#pragma unroll
            for (int c2 = 0; c2 < D / 64; ++c2) {
                uint32_t va[2][32];
                if (u > 0) {
                    tmem_ld32(tl + col + c2 * 64, va[0]);
                    tmem_ld32(tl + col + c2 * 64 + 32, va[1]);
                    tmem_ld_wait(va[0]);
                    tmem_ld_wait(va[1]);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) va[0][e] = va[1][e] = 0u;
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int c = 2 * c2 + half;
                    const uint32_t* v = va[half];
                    uint4* dst = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 w = make_uint4(
                            pack_bf16x2(__uint_as_float(v[8 * q]) * mul, __uint_as_float(v[8 * q + 1]) * mul),
                            pack_bf16x2(__uint_as_float(v[8 * q + 2]) * mul, __uint_as_float(v[8 * q + 3]) * mul),
                            pack_bf16x2(__uint_as_float(v[8 * q + 4]) * mul, __uint_as_float(v[8 * q + 5]) * mul),
                            pack_bf16x2(__uint_as_float(v[8 * q + 6]) * mul, __uint_as_float(v[8 * q + 7]) * mul));
                        if (tma_rows) {
                            const int ch = (half << 2) + q;  // 16-byte chunk within the 128-byte row
                            sts128(smem_u32(ob + c2 * 4096 + lane * 128 + ((ch ^ (lane & 7)) << 4)), w.x, w.y, w.z,
                                   w.w);
                        } else if (row_ok) {
                            dst[q] = w;
                        }
                    }
                }
            }
            if (kDirectEpi && tma_rows) {
                // the warp copies its boxes out itself, four full 128-byte
                // rows per store instruction, instead of queueing bulk tensor
                // stores behind the last block's dQ reduce-adds in the SM's
                // bulk-copy unit (which drain at the L2 reduction rate)
                __syncwarp();
                uint16_t* obase = static_cast<uint16_t*>(g == 0 ? p.dv : p.dk);
#pragma unroll
                for (int rg = 0; rg < C::NREG; ++rg)
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int row = it * 4 + (lane >> 3), ch = lane & 7;
                        const uint4 w = lds128_u4(smem_u32(ob + rg * 4096 + row * 128 + ((ch ^ (row & 7)) << 4)));
                        const size_t grow_ = varlen ? (static_cast<size_t>(seq0 + wkey0 + row) * p.H + h) * D
                                                    : (static_cast<size_t>(bh) * N + wkey0 + row) * D;
                        *reinterpret_cast<uint4*>(obase + grow_ + rg * 64 + ch * 8) = w;
                    }
            } else if (tma_rows) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const CUtensorMap* m = g == 0 ? &tmdV : &tmdK;
#pragma unroll
                    for (int rg = 0; rg < C::NREG; ++rg) {
                        if (varlen)
                            tma_store_3d(m, rg * 64, h, seq0 + wkey0, ob + rg * 4096);
                        else
                            tma_store_2d(m, rg * 64, bh * N + wkey0, ob + rg * 4096);
                    }
                    bulk_commit_group();
                    // the shared buffer must be read out before the CTA exits
                    bulk_wait_group_read0();
                }
            }
        }
    } else if (warp >= 12) {
        // ------------------------------------------------------------ dQ drain (thread = query)
        // dQ_i is staged through the Q_i and dO_i stage of its own block:
        // its GEMMs are complete once dQ_i is, and the producer reloads the
        // stage only after the four drain warps release it. Warp wq's rows
        // form D / 32 boxes of [32 x 32] fp32 (4 KiB); box k sits in the Q
        // tile for the first half of the boxes and in the dO tile for the
        // rest, so every reduce-add of the block is issued before any wait.
        constexpr int NB = D / 32, NBH = NB / 2;
        const int wq = warp & 3;
        const uint32_t tl = tm + (static_cast<uint32_t>(wq * 32) << 16);
        int u = 0;
        for (int i = next_i(lo); i < T; i = next_i(i + 1)) {
            if (!visible_i(i)) continue;
            bool ok = mbar_wait(dq_full, u & 1, cx, 22);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int grow = bh * N + i * kTile + wq * 32;  // first accumulator row of this warp
            const int st = u % C::STAGES;
            uint8_t* box_q = sm + C::Q_OFF + st * C::TILE_BYTES + wq * (NBH * 4096);
            uint8_t* box_do = sm + C::DO_OFF + st * C::TILE_BYTES + wq * (NBH * 4096);
#pragma unroll
            for (int half = 0; half < D / 64; ++half) {
                if (kDqFirst && half == 1) {
                    // the second half goes to the Q_i tile, which dK_i reads
                    ok = __all_sync(0xffffffffu, mbar_wait(dk_done, u & 1, cx, 25));
                    if (!ok) break;
                }
                uint32_t v[2][32];
                const uint32_t col_q = (u & 1) ? 128u : 0u;  // dQ_u shares the buffer of S^T_u
                tmem_ld32(tl + col_q + half * 64, v[0]);
                tmem_ld32(tl + col_q + half * 64 + 32, v[1]);
                tmem_ld_wait(v[0]);
                tmem_ld_wait(v[1]);
                if (half == D / 64 - 1) {
                    // every TMEM read of dQ_i is done: its columns may be reused
                    tc_fence_before();
                    mbar_arrive(dq_free);
                }
#pragma unroll
                for (int bx = 0; bx < 2; ++bx) {
                    const int k = half * 2 + bx;
                    uint8_t* box = kDqFirst ? (half == 1 ? box_q : box_do) + bx * 4096
                                            : (k < NBH ? box_q + k * 4096 : box_do + (k - NBH) * 4096);
                    const uint32_t sb = smem_u32(box);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t* w = &v[bx][4 * c];
                        sts128(sb + lane * 128 + ((c ^ (lane & 7)) * 16), w[0], w[1], w[2], w[3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx) {
                        const int k = half * 2 + bx;
                        const uint8_t* box = kDqFirst ? (half == 1 ? box_q : box_do) + bx * 4096
                                                      : (k < NBH ? box_q + k * 4096 : box_do + (k - NBH) * 4096);
                        if (varlen)
                            tma_reduce_add_3d(&tmdQacc, k * 32, h, seq0 + i * kTile + wq * 32, box);
                        else
                            tma_reduce_add_2d(&tmdQacc, k * 32, grow, box);
                    }
                    bulk_commit_group();
                }
            }
            if (kDqFirst && !ok) break;  // gave up waiting for dK_i (the reduce-adds in flight land below)
            if (lane == 0) {
                // the stage may be refilled once the reduce-adds have read it
                bulk_wait_group_read0();
                mbar_arrive(&qd_empty[st]);
            }
            __syncwarp();
            ++u;
        }
        if (lane == 0) bulk_wait_group0();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

// D[row] = sum_k dO[row, k] * O[row, k] in fp32, stored negated (-D); also
// zeroes dQ_accum[row, :] and writes -L in log2 units (-L * log2 e; -inf for
// a row that saw no key, so that its recomputed probabilities are 0). D/8
// threads share a row (16 bytes of O and of dO each) and reduce with warp
// shuffles.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                                         const float* __restrict__ lse, float* __restrict__ ndelta,
                                                         float* __restrict__ nlse2, float* __restrict__ dq_accum,
                                                         long long rows) {
    constexpr int TPR = D / 8;  // threads per row
    const long long row = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) / TPR;
    const int part = threadIdx.x % TPR;
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + part * 8);
        const uint4 g = *reinterpret_cast<const uint4*>(dout + row * D + part * 8);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(__uint_as_float(av[e] << 16), __uint_as_float(gv[e] << 16), acc);
            acc = fmaf(__uint_as_float(av[e] & 0xFFFF0000u), __uint_as_float(gv[e] & 0xFFFF0000u), acc);
        }
        float4* z = reinterpret_cast<float4*>(dq_accum + row * D + part * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && part == 0) {
        ndelta[row] = -acc;
        const float L = lse[row];
        nlse2[row] = L == -CUDART_INF_F ? -CUDART_INF_F : -L * kLog2e;
    }
}

// Packed batches: cu_tiles[b] = number of 128-row tiles of the sequences
// before b (each sequence clamped as the attention kernels clamp it), so that
// sequence b's rows of -L and -D can start at the aligned row cu_tiles[b] *
// 128 of a per-head block. One block; a scan over chunks of 1024 sequences.
__global__ void __launch_bounds__(1024) fa_varlen_tiles_kernel(const int32_t* __restrict__ cu, int B, int total,
                                                               int max_seqlen, int32_t* __restrict__ cu_tiles) {
    __shared__ int warp_sums[32];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int base = 0; base < B; base += 1024) {
        const int bi = base + threadIdx.x;
        int tiles = 0;
        if (bi < B) {
            const int s0 = min(max(cu[bi], 0), total);
            const int s1 = min(max(cu[bi + 1], s0), total);
            tiles = (min(s1 - s0, max_seqlen) + kTile - 1) / kTile;
        }
        int x = tiles;  // inclusive scan within the warp
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) warp_sums[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            warp_sums[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int before = carry + (wid > 0 ? warp_sums[wid - 1] : 0) + x - tiles;
        if (bi < B) cu_tiles[bi] = before;
        __syncthreads();
        if (threadIdx.x == 1023) carry = before + tiles;
        __syncthreads();
    }
    if (threadIdx.x == 0) cu_tiles[B] = carry;
}

// Packed-batch version of fa_bwd_pre_kernel: row = token * H + head of the
// [total, H, d] tensors; -D and -L * log2 e go to the aligned per-sequence
// rows of the scratch; tokens not covered by any (clamped) sequence only get
// their dQ accumulator row zeroed.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_varlen_kernel(
    const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout, const float* __restrict__ lse,
    const int32_t* __restrict__ cu, const int32_t* __restrict__ cu_tiles, int B, int H, int total, int max_seqlen,
    long long lpad, float* __restrict__ ndelta, float* __restrict__ nlse2, float* __restrict__ dq_accum) {
    constexpr int TPR = D / 8;
    const long long rows = static_cast<long long>(total) * H;
    const long long row = (static_cast<long long>(blockIdx.x) * 256 + threadIdx.x) / TPR;
    const int part = threadIdx.x % TPR;
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + part * 8);
        const uint4 g = *reinterpret_cast<const uint4*>(dout + row * D + part * 8);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(__uint_as_float(av[e] << 16), __uint_as_float(gv[e] << 16), acc);
            acc = fmaf(__uint_as_float(av[e] & 0xFFFF0000u), __uint_as_float(gv[e] & 0xFFFF0000u), acc);
        }
        float4* z = reinterpret_cast<float4*>(dq_accum + row * D + part * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && part == 0) {
        const int t = static_cast<int>(row / H), h = static_cast<int>(row % H);
        // the sequence holding token t: the last b with cu[b] <= t
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (min(max(cu[mid], 0), total) <= t) lo = mid; else hi = mid - 1;
        }
        const int s0 = min(max(cu[lo], 0), total);
        const int s1 = min(max(cu[lo + 1], s0), total);
        const int len = min(s1 - s0, max_seqlen);
        const int local = t - s0;
        if (local >= 0 && local < len) {
            const long long dst = static_cast<long long>(h) * lpad + static_cast<long long>(cu_tiles[lo]) * kTile + local;
            ndelta[dst] = -acc;
            const float L = lse[static_cast<long long>(h) * total + t];
            nlse2[dst] = L == -CUDART_INF_F ? -CUDART_INF_F : -L * kLog2e;
        }
    }
}

// dQ (bf16) <- scale * dQ_accum (fp32), 8 elements per thread.
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                        long long n8, float scale) {
    for (long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; i < n8;
         i += static_cast<long long>(gridDim.x) * 256) {
        const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
        const float4 c = reinterpret_cast<const float4*>(acc)[2 * i + 1];
        reinterpret_cast<uint4*>(dq)[i] = make_uint4(pack_bf16x2(a.x * scale, a.y * scale),
                                                     pack_bf16x2(a.z * scale, a.w * scale),
                                                     pack_bf16x2(c.x * scale, c.y * scale),
                                                     pack_bf16x2(c.z * scale, c.w * scale));
    }
}

template <int D>
static cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t stream, int* nlaunch) {
    using C = BwdCfg<D>;
    const bool varlen = a.cu_seqlens != nullptr;
    // rows of the [rows, d] views: B * H * N, or total * H for a packed batch
    const uint64_t rows = varlen ? static_cast<uint64_t>(a.total) * a.H : static_cast<uint64_t>(a.B) * a.H * a.N;
    CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
    if (varlen) {
        const uint64_t tot = static_cast<uint64_t>(a.total);
        if (!make_tmap_packed_sw128(&tq, a.q, tot, a.H, D, 2, kTile, 64) ||
            !make_tmap_packed_sw128(&tk, a.k, tot, a.H, D, 2, kTile, 64) ||
            !make_tmap_packed_sw128(&tv, a.v, tot, a.H, D, 2, kTile, 64) ||
            !make_tmap_packed_sw128(&tdo, a.dout, tot, a.H, D, 2, kTile, 64) ||
            !make_tmap_packed_sw128(&tdq, a.dq_accum, tot, a.H, D, 4, 32, 32) ||
            !make_tmap_packed_sw128(&tdk, a.dk, tot, a.H, D, 2, 32, 64) ||
            !make_tmap_packed_sw128(&tdv, a.dv, tot, a.H, D, 2, 32, 64))
            return cudaErrorInvalidValue;
    } else if (!make_tmap_2d_sw128(&tq, a.q, rows, D, 2, kTile, 64) ||
               !make_tmap_2d_sw128(&tk, a.k, rows, D, 2, kTile, 64) ||
               !make_tmap_2d_sw128(&tv, a.v, rows, D, 2, kTile, 64) ||
               !make_tmap_2d_sw128(&tdo, a.dout, rows, D, 2, kTile, 64) ||
               !make_tmap_2d_sw128(&tdq, a.dq_accum, rows, D, 4, 32, 32) ||
               !make_tmap_2d_sw128(&tdk, a.dk, rows, D, 2, 32, 64) ||
               !make_tmap_2d_sw128(&tdv, a.dv, rows, D, 2, 32, 64))
        return cudaErrorInvalidValue;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(fa_bwd_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fa_bwd_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fa_bwd_kernel<D, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     C::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(fa_bwd_kernel<D, false, false, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const long long nrows = static_cast<long long>(rows);
    const long long pre_threads = nrows * (D / 8);
    int launches = 0;
    if (varlen) {
        fa_varlen_tiles_kernel<<<1, 1024, 0, stream>>>(a.cu_seqlens, a.B, a.total, a.N, a.cu_tiles);
        // rows of the -L / -D blocks that no token fills stay finite (zero)
        const size_t lbytes = static_cast<size_t>(a.H) * a.lpad * sizeof(float);
        cudaError_t e = cudaMemsetAsync(a.delta, 0, lbytes, stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(a.lse2, 0, lbytes, stream);
        if (e != cudaSuccess) return e;
        fa_bwd_pre_varlen_kernel<D><<<static_cast<unsigned>((pre_threads + 255) / 256), 256, 0, stream>>>(
            static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.lse, a.cu_seqlens, a.cu_tiles,
            a.B, a.H, a.total, a.N, a.lpad, a.delta, a.lse2, a.dq_accum);
        launches += 2;
    } else {
        fa_bwd_pre_kernel<D><<<static_cast<unsigned>((pre_threads + 255) / 256), 256, 0, stream>>>(
            static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.lse, a.delta, a.lse2,
            a.dq_accum, nrows);
        launches += 1;
    }
    BwdParams p;
    p.B = a.B;
    p.H = a.H;
    p.N = a.N;
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.mask.blockmask = a.blockmask;
    p.mask.kv_len = a.kv_len;
    p.mask.causal = a.causal;
    p.mask.T = (a.N + kTile - 1) / kTile;
    p.nlse2 = a.lse2;
    p.ndelta = a.delta;
    p.dk = a.dk;
    p.dv = a.dv;
    p.status = a.status;
    p.cu_seqlens = a.cu_seqlens;
    p.cu_tiles = a.cu_tiles;
    p.total = a.total;
    p.lpad = a.lpad;
    // causal [B, H, N, d] calls: head groups whose Q, dO (bf16) and dQ
    // accumulator (fp32) rows take at most 64 MiB of L2
    const int Tn = (a.N + kTile - 1) / kTile;
    p.group = 0;
    if (a.causal && !varlen) {
        const long long per_head = 8LL * a.N * D;
        long long g = (64LL << 20) / per_head;
        g = g < 1 ? 1 : g;
        p.group = static_cast<int>(g < a.B * a.H ? g : a.B * a.H);
    }
    const dim3 grid = p.group > 0 ? dim3(static_cast<unsigned>(Tn) * a.H * a.B) : dim3(Tn, a.H, a.B);
    if (a.ev_begin) cudaEventRecord(a.ev_begin, stream);
    p.drop = a.drop;
    if (varlen)
        fa_bwd_kernel<D, true><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
    else if (a.dropout)
        fa_bwd_kernel<D, false, true><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
    else if (a.blockmask)
        fa_bwd_kernel<D, false, false, true><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
    else
        fa_bwd_kernel<D, false><<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, tdk, tdv, p);
    if (a.ev_end) cudaEventRecord(a.ev_end, stream);
    const long long n8 = nrows * D / 8;
    long long blocks = (n8 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    fa_bwd_dq_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a.dq_accum, static_cast<uint16_t*>(a.dq), n8,
                                                                        a.scale);
    *nlaunch = launches + 2;
    return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream, int* nlaunch) {
    if (a.d == 64) return launch_bwd_t<64>(a, stream, nlaunch);
    return launch_bwd_t<128>(a, stream, nlaunch);
}

}  // namespace fa

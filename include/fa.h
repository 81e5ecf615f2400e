/*
 * fa.h -- C ABI of libfa.so: fused, tiled, exact softmax attention on GB300
 * (sm_103a), forward and backward.
 *
 * What is computed ("FlashAttention: making attention IO-aware", sections
 * "Attention is memory-bound", "Tiling: never materialise S", "Online
 * softmax", "The backward pass: recompute, don't store"):
 *
 *   S = scale * Q K^T (+ mask),  P = softmax(S) row-wise,  O = P V,
 *   L = m + log(l) per query row (natural log; m = row max, l = sum exp(S - m))
 *
 * and, for the backward pass, the gradients of <dO, O>:
 *
 *   D = rowsum(dO * O),  dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
 *   dQ = scale * dS K,  dK = scale * dS^T Q,
 *
 * with P recomputed tile by tile from Q, K and L. No N x N matrix is ever
 * written to device memory.
 *
 * Masks (all optional, combined with AND): causal (key j visible to query i
 * iff j <= i; "FlashAttention-2" section: tiles above the diagonal are
 * skipped), key padding (key j visible iff j < kv_len[b]; "Why is
 * FlashAttention faster?", "Extra computation can still finish sooner"), and
 * a 128 x 128 tile mask shared by every (batch, head) (block-sparse
 * attention, "Counting the IO": masked tiles are skipped entirely). A query
 * row that sees no key gets O = 0, L = -inf and contributes no gradient.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout: Q, K, V, O, dO, dQ, dK, dV are contiguous [B, H, N, d] row-major
 *   arrays in device memory, all of the element type `dtype`; lse is a
 *   contiguous float32 [B, H, N] array. Base pointers must be 16-byte aligned.
 * Types: FA_BF16 (bfloat16 in and out, bf16 tensor-core products with fp32
 *   accumulation) or FA_FP32 (float32 in and out; S from three tf32
 *   tensor-core products of high/low parts, P V in tf32, fp32 accumulation;
 *   forward pass with d = 64 only).
 * Supported sizes: d in {64, 128}; N a positive multiple of 128;
 *   B * H * N < 2^31. Other sizes return FA_ERR_UNSUPPORTED.
 * blockmask: NULL or a device uint8 array [N/128, N/128]; entry [i][j] != 0
 *   keeps the tile of query block i and key block j.
 * kv_len: NULL or a device int32 array [B] with 0 <= kv_len[b] <= N.
 * Ownership: the caller allocates and frees every buffer, including the
 *   workspace; the library allocates no device memory and keeps no pointer
 *   after a call returns. The one exception is fa_bwd_noalloc (and its status
 *   reader), which uses a fixed device array inside the library and caches
 *   its address per device; its own comment below gives the rules.
 * Device: kernels run on the calling thread's current CUDA device
 *   (cudaGetDevice); every buffer must be memory of that device and `stream`
 *   one of its streams. Buffers of another device are not detected here.
 * Streams: `stream` is a cudaStream_t (NULL = legacy default stream). Calls
 *   are asynchronous with respect to the host: argument checks run on the host
 *   and return an error before anything is launched; launch failures return
 *   FA_ERR_CUDA; a device-side wait that gives up (a bounded wait that expired)
 *   is reported by fa_get_status on the workspace of that call.
 * Workspace: a device buffer of at least the size the matching
 *   *_workspace_size function returns, 256-byte aligned. Its contents need not
 *   be initialised. Two calls in flight at the same time need two workspaces.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null pointer, bad alignment, negative size, ... */
    FA_ERR_UNSUPPORTED = 2, /* valid request outside the supported sizes/types */
    FA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    FA_ERR_TIMEOUT = 4      /* a device-side bounded wait gave up */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP32 = 1 } fa_dtype;

/* Bytes of workspace fa_fwd needs for these sizes: the status word, plus,
 * for FA_FP32 calls, a transposed copy of V (tf32 tensor-core operands must
 * be K-major) and the tf32 high and low parts of Q and K (S is formed from
 * three tf32 products to keep fp32 accuracy). FA_BF16 calls need only 256
 * bytes but accept the full size. */
size_t fa_fwd_workspace_size(int B, int H, int N, int d);

/* Bytes of workspace fa_bwd needs: D = rowsum(dO * O) and L in log2 units
 * (fp32 [B,H,N] each), the fp32 dQ accumulator [B,H,N,d] and the status
 * word. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Forward pass ("Online softmax"; the tiled forward of "FlashAttention:
 * making attention IO-aware"): writes O [B,H,N,d] and lse = L [B,H,N].
 *   q, k, v   in,  device, [B,H,N,d] of `dtype`
 *   o         out, device, [B,H,N,d] of `dtype`
 *   lse       out, device, float32 [B,H,N], natural-log logsumexp of the
 *             scaled, masked scores of each row
 *   scale     multiplies Q K^T before the softmax (usually 1/sqrt(d))
 *   causal    0 or 1
 *   blockmask, kv_len  optional masks (see above)
 *   workspace, ws_bytes  device scratch of fa_fwd_workspace_size bytes
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (nothing launched),
 *         FA_ERR_CUDA (launch failed).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, const uint8_t* blockmask, const int32_t* kv_len, fa_dtype dtype,
                 void* workspace, size_t ws_bytes, void* stream);

/*
 * Packed variable-length batches ("FlashAttention: making attention
 * IO-aware", section "In practice": a packed kernel takes one flat batch of
 * concatenated sequences plus their offsets, so padding costs nothing).
 * Self-attention within each sequence: sequence b is tokens
 * cu_seqlens[b] .. cu_seqlens[b+1]-1, it attends only to its own tokens, and
 * the causal mask is aligned at the start of each sequence.
 *   q, k, v     in,  device, token-major [total, H, d] bf16 (FA_BF16 only)
 *   o           out, device, [total, H, d] bf16
 *   lse         out, device, float32 [H, total] (natural log)
 *   cu_seqlens  in,  device, int32 [B + 1]: 0 = cu_seqlens[0] <= ... <=
 *               cu_seqlens[B] = total
 *   max_seqlen  host, the longest cu_seqlens[b+1] - cu_seqlens[b] (sizes the
 *               grid); 1 <= max_seqlen <= total
 *   scale, causal, workspace as for fa_fwd (workspace of
 *               fa_fwd_varlen_workspace_size bytes)
 * Any sequence lengths are allowed (no multiple of 128 needed; empty
 * sequences produce nothing). The offsets live in device memory, so they are
 * checked on the device: values outside [0, total] are clamped, and a
 * sequence longer than max_seqlen is cut to max_seqlen tokens and reported
 * as FA_ERR_INVALID_ARG by fa_get_status (rows outside the cut are not
 * written). Errors otherwise as for fa_fwd.
 */
size_t fa_fwd_varlen_workspace_size(int H, int total, int d);
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens,
                        int B, int H, int total, int max_seqlen, int d, float scale, int causal, fa_dtype dtype,
                        void* workspace, size_t ws_bytes, void* stream);

/*
 * Decoding: a few new query rows against a long key/value cache
 * ("FlashAttention: making attention IO-aware", section "In practice": with
 * one query row there is no query block to parallelise over, so
 * Flash-Decoding splits the keys across thread blocks and merges the partial
 * results with logsumexp rescaling). Every query row of batch element b sees
 * the first cache_len[b] cache entries.
 *   q           in,  device, [B, H, Nq, d] bf16, 1 <= Nq <= 8
 *   k, v        in,  device, the cache, [B, H, Nk, d] bf16 (any Nk >= 1)
 *   o           out, device, [B, H, Nq, d] bf16
 *   lse         out, device, float32 [B, H, Nq] (natural log; -inf for a row
 *               with no valid key, whose o row is 0)
 *   cache_len   NULL (all Nk entries valid) or device int32 [B]; values are
 *               clamped to [0, Nk] on the device
 *   num_splits  key splits per (b, h): 0 picks a count from the sizes;
 *               otherwise at most one split per 64 keys is used
 *   workspace   fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits) bytes
 *               (partial maxima, sums and outputs of the splits)
 * Runs two kernels (the splits, then the merge). FA_BF16 only; d in {64, 128}.
 */
size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits);
fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                    int d, float scale, const int32_t* cache_len, int num_splits, fa_dtype dtype, void* workspace,
                    size_t ws_bytes, void* stream);

/*
 * FP8 forward pass ("FlashAttention: making attention IO-aware", section
 * "FlashAttention-3": FP8 doubles the tensor rate but is fragile with
 * outliers, so Q and K are multiplied by a random orthogonal Hadamard matrix
 * first and quantised per block). An approximation of attention:
 *   1. Q' = Q diag(signs) H_128 and K' = K diag(signs) H_128 (Sylvester
 *      Hadamard matrix; the 1/128 left in Q' K'^T joins the score scale);
 *   2. each 128-row block of Q' and of K', and V (one block per head), is
 *      divided by the power of two 2^ceil(log2(amax / 448)) and rounded to
 *      E4M3 (nearest even, saturating);
 *   3. S and O = softmax(S) V on the FP8 tensor cores; the weights are
 *      rounded to E4M3 relative to a running integer exponent (a weight
 *      below 2^-6 of the row's final maximum can therefore round differently
 *      than relative to that maximum), O is normalised by the sum of the
 *      rounded weights and L comes from the unrounded ones.
 *   q, k, v   in,  device, [B, H, N, 128] bf16
 *   o         out, device, [B, H, N, 128] bf16
 *   lse       out, device, float32 [B, H, N]
 *   signs     in,  device, float32 [128], each +1 or -1 (drawn by the
 *             caller), or NULL: no rotation (step 1 skipped, Q and K are
 *             quantised as they are; for measuring what the rotation buys)
 *   causal, kv_len  masks as for fa_fwd (no tile mask)
 *   workspace fa_fwd_fp8_workspace_size(B, H, N, d) bytes: the quantised
 *             Q, K and V^T, their scale exponents and V's block maxima
 * d = 128, N a multiple of 128 and B * H <= 65535 only (FA_ERR_UNSUPPORTED
 * otherwise). Runs three kernels: quantisation of Q and K together with the
 * block maxima of V, V's quantisation, and the attention kernel.
 */
size_t fa_fwd_fp8_workspace_size(int B, int H, int N, int d);
fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                     float scale, int causal, const int32_t* kv_len, const float* signs, void* workspace,
                     size_t ws_bytes, void* stream);

/*
 * Attention with dropout on the probabilities, fused into the kernels ("Why
 * is FlashAttention faster?", "Kernel fusion removes stage boundaries":
 * masking, softmax and dropout become stages of one kernel). The forward
 * computes O = (softmax(S) * Z / (1 - p)) V and L = logsumexp(S); the
 * backward regenerates the same keep mask Z instead of storing it.
 * Z for (b, h, query i, key j): byte (j mod 4) of word (i mod 4) of
 * Philox-4x32-10 (Salmon et al., SC 2011) with counter (i/4, j/4, h, b) and
 * key (seed mod 2^32, seed / 2^32); kept iff the byte >= t = round(256 p),
 * so the effective rate is t / 256 (0 <= p < 1, t capped at 255).
 * Arguments as for fa_fwd / fa_bwd with FA_BF16 tensors and no tile mask,
 * plus dropout_p and seed; the backward must get the forward's p and seed.
 */
fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                         float scale, int causal, const int32_t* kv_len, float dropout_p, unsigned long long seed,
                         void* workspace, size_t ws_bytes, void* stream);
fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, const int32_t* kv_len, float dropout_p, unsigned long long seed, void* workspace,
                         size_t ws_bytes, void* stream);

/*
 * Backward pass of a packed variable-length batch: the gradients of
 * <dO, O> for fa_fwd_varlen.
 *   q, k, v, o, dout  in,  device, [total, H, d] bf16
 *   lse               in,  device, float32 [H, total] from fa_fwd_varlen
 *   dq, dk, dv        out, device, [total, H, d] bf16
 *   cu_seqlens, B, max_seqlen, scale, causal as for fa_fwd_varlen
 *   workspace         fa_bwd_varlen_workspace_size(B, H, total, d) bytes:
 *                     the status word, the running tile counts of the
 *                     sequences, -L and -D with every sequence starting on a
 *                     128-row boundary, and the fp32 dQ accumulator
 * Launches four kernels: the tile counts, D = rowsum(dO * O), the fused
 * key-block kernel, and the dQ conversion (plus three memsets: the status
 * word and the -L and -D blocks).
 */
size_t fa_bwd_varlen_workspace_size(int B, int H, int total, int d);
fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, const int32_t* cu_seqlens, int B, int H,
                        int total, int max_seqlen, int d, float scale, int causal, fa_dtype dtype, void* workspace,
                        size_t ws_bytes, void* stream);

/*
 * Backward pass ("The backward pass: recompute, don't store"): given the
 * forward inputs, its outputs O and lse, and dO, writes dQ, dK, dV.
 *   q, k, v, o, dout  in,  device, [B,H,N,d] of `dtype` (FA_BF16 only)
 *   lse               in,  device, float32 [B,H,N] from fa_fwd
 *   dq, dk, dv        out, device, [B,H,N,d] of `dtype`
 *   the remaining arguments as for fa_fwd; the masks must be the ones the
 *   forward pass used.
 * Runs three kernels on `stream`: D = rowsum(dO * O) (and zeroing of the dQ
 * accumulator), the fused key-block kernel, and the dQ conversion.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                 const uint8_t* blockmask, const int32_t* kv_len, fa_dtype dtype, void* workspace, size_t ws_bytes,
                 void* stream);

/*
 * Backward pass without a caller-supplied workspace. The pages describe no
 * counterpart of this call; it exists for callers that cannot allocate
 * device memory when they run the backward pass (for example a plug-in whose
 * host runtime gives it tensors but no allocator, or a latency-critical loop
 * that must not call cudaMalloc / cudaFree because they can synchronise the
 * device). Arguments and results are those of fa_bwd minus the workspace:
 * the scratch fa_bwd would take from the workspace comes from a fixed 32 MiB
 * device array inside the library, which every GPU that loads the library
 * keeps until the process exits. Nothing is allocated.
 *   - Requests with fa_bwd_workspace_size(B, H, N, d) > 32 MiB return
 *     FA_ERR_UNSUPPORTED without launching anything.
 *   - All calls on a device share that array and it keeps the previous call's
 *     contents; each call re-zeroes what must start at zero. Calls that can
 *     overlap on the GPU (other streams, unordered host threads) race on it:
 *     serialise them on one stream.
 *   - The first call on each device (with that device current) looks up the
 *     array's device address; make that first call before any stream capture.
 *     The address stays cached until the process exits; cudaDeviceReset
 *     unloads the library's device code, so do not call this entry point on a
 *     device after resetting it.
 *   - Device-side wait time-outs are recorded in the array's status word and
 *     returned by fa_bwd_noalloc_get_status. Each call clears the word when
 *     it starts, so read it before the next call on that device.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, const uint8_t* blockmask, const int32_t* kv_len, fa_dtype dtype, void* stream);

/* Status of the last fa_bwd_noalloc call on the current device, like
 * fa_get_status for a workspace: synchronises `stream` (the stream of that
 * call), then reads and clears the status word of the library's fixed
 * scratch array. Returns FA_OK, FA_ERR_TIMEOUT (a device-side wait gave up;
 * that call's dQ, dK, dV are invalid) or FA_ERR_CUDA. The pages have no
 * counterpart of this call. */
fa_status fa_bwd_noalloc_get_status(void* stream);

/* Synchronises `stream`, then reads and clears the device status word of
 * `workspace` (of the fa_fwd or fa_bwd call that used it). Returns FA_OK or
 * FA_ERR_TIMEOUT (a device-side wait gave up; the outputs are then invalid),
 * or FA_ERR_CUDA if the stream reported an error. */
fa_status fa_get_status(void* workspace, void* stream);

/* Static, human-readable name of a status code. */
const char* fa_status_string(fa_status s);

/* Number of kernels that the last successful call made by this host thread
 * to an entry point that launches work (fa_fwd, fa_bwd, their packed,
 * decoding, FP8 and dropout forms, fa_bwd_noalloc) launched, for accounting
 * in benchmarks. */
int fa_last_launch_count(void);

/* Profiling hook: for the following calls made by this host thread to the
 * entry points that launch work, record the CUDA event `begin` (a
 * cudaEvent_t) on the call's stream immediately before the main attention
 * kernel and `end` immediately after it, so that a caller can time that
 * kernel alone. Passing NULL for both
 * turns the hook off. The events are owned by the caller. Returns
 * FA_ERR_INVALID_ARG if exactly one of them is NULL. */
fa_status fa_set_timing_events(void* begin, void* end);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */

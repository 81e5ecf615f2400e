// C ABI of libfa.so (declared in include/fa.h): argument checks, workspace
// carving, status word handling and dispatch to the kernel launchers.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "fa.h"
#include "fa_decode.h"
#include "fa_fp8.h"
#include "fa_launch.h"

namespace {

constexpr size_t kStatusBytes = 256;
thread_local int g_last_launches = 0;
thread_local cudaEvent_t g_ev_begin = nullptr, g_ev_end = nullptr;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape checks shared by both passes.
fa_status check_shape(int B, int H, int N, int d, float scale) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (N % 128 != 0) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * H * N >= (1LL << 31)) return FA_ERR_UNSUPPORTED;
    // grid limits: forward (H, B, pairs of query tiles), backward (N/128, H, B)
    if (B > 65535 || H > 65535 || (N / 128 + 1) / 2 > 65535) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// Shape checks of the packed variable-length entry points.
fa_status check_varlen_shape(int B, int H, int total, int max_seqlen, int d, float scale) {
    if (B <= 0 || H <= 0 || total <= 0 || max_seqlen <= 0 || d <= 0) return FA_ERR_INVALID_ARG;
    if (max_seqlen > total) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(total) * H >= (1LL << 31) - 256) return FA_ERR_UNSUPPORTED;
    const int tiles = (max_seqlen + 127) / 128;
    if (B > 65535 || H > 65535 || (tiles + 1) / 2 > 65535) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

fa_status map_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace

extern "C" {

size_t fa_fwd_workspace_size(int B, int H, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
    // status word + fp32 inputs only: V^T and the tf32 high/low parts of Q, K
    return kStatusBytes + 5 * align256(static_cast<size_t>(B) * H * N * d * sizeof(float));
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
    const size_t rows = static_cast<size_t>(B) * H * N;
    return kStatusBytes + 2 * align256(rows * sizeof(float)) + align256(rows * d * sizeof(float));
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, const uint8_t* blockmask, const int32_t* kv_len, fa_dtype dtype,
                 void* workspace, size_t ws_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    fa_status st = check_shape(B, H, N, d, scale);
    if (st != FA_OK) return st;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        !aligned(workspace, 256) || (kv_len && !aligned(kv_len, 4)))
        return FA_ERR_INVALID_ARG;
    if (dtype == FA_FP32 && d != 64) return FA_ERR_UNSUPPORTED;
    const size_t need = dtype == FA_FP32 ? fa_fwd_workspace_size(B, H, N, d) : kStatusBytes;
    if (ws_bytes < need) return FA_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    fa::FwdArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.blockmask = blockmask;
    a.kv_len = kv_len;
    a.fp32 = dtype == FA_FP32;
    a.status = static_cast<int*>(workspace);
    a.fp32_scratch = static_cast<char*>(workspace) + kStatusBytes;
    a.ev_begin = g_ev_begin;
    a.ev_end = g_ev_end;
    if (cudaMemsetAsync(a.status, 0, sizeof(int) * 4, s) != cudaSuccess) return FA_ERR_CUDA;
    int n = 0;
    st = map_cuda(fa::launch_fwd(a, s, &n));
    if (st == FA_OK) g_last_launches = n;
    return st;
}

size_t fa_fwd_varlen_workspace_size(int H, int total, int d) {
    if (H <= 0 || total <= 0 || d <= 0) return 0;
    return kStatusBytes;
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens,
                        int B, int H, int total, int max_seqlen, int d, float scale, int causal, fa_dtype dtype,
                        void* workspace, size_t ws_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !cu_seqlens || !workspace) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    fa_status st = check_varlen_shape(B, H, total, max_seqlen, d, scale);
    if (st != FA_OK) return st;
    if (dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        !aligned(cu_seqlens, 4) || !aligned(workspace, 256))
        return FA_ERR_INVALID_ARG;
    if (ws_bytes < fa_fwd_varlen_workspace_size(H, total, d)) return FA_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    fa::FwdArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.N = max_seqlen;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.cu_seqlens = cu_seqlens;
    a.total = total;
    a.status = static_cast<int*>(workspace);
    a.ev_begin = g_ev_begin;
    a.ev_end = g_ev_end;
    if (cudaMemsetAsync(a.status, 0, sizeof(int) * 4, s) != cudaSuccess) return FA_ERR_CUDA;
    int n = 0;
    st = map_cuda(fa::launch_fwd(a, s, &n));
    if (st == FA_OK) g_last_launches = n;
    return st;
}

// Rows per head of the -L / -D blocks of a packed backward pass: every
// sequence starts on a 128-row boundary, which costs at most 128 rows each.
static long long varlen_lpad(int B, int total) {
    return (static_cast<long long>(total) + 127) / 128 * 128 + 128LL * B;
}

size_t fa_bwd_varlen_workspace_size(int B, int H, int total, int d) {
    if (B <= 0 || H <= 0 || total <= 0 || d <= 0) return 0;
    const size_t lrows = static_cast<size_t>(H) * varlen_lpad(B, total);
    return kStatusBytes + align256((static_cast<size_t>(B) + 1) * sizeof(int32_t)) +
           2 * align256(lrows * sizeof(float)) + align256(static_cast<size_t>(total) * H * d * sizeof(float));
}

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, const int32_t* cu_seqlens, int B, int H,
                        int total, int max_seqlen, int d, float scale, int causal, fa_dtype dtype, void* workspace,
                        size_t ws_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !cu_seqlens || !workspace)
        return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    fa_status st = check_varlen_shape(B, H, total, max_seqlen, d, scale);
    if (st != FA_OK) return st;
    if (dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
        !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(cu_seqlens, 4) ||
        !aligned(workspace, 256))
        return FA_ERR_INVALID_ARG;
    if (ws_bytes < fa_bwd_varlen_workspace_size(B, H, total, d)) return FA_ERR_INVALID_ARG;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    fa::BwdArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.H = H;
    a.N = max_seqlen;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.cu_seqlens = cu_seqlens;
    a.total = total;
    a.lpad = varlen_lpad(B, total);
    const size_t lrows = static_cast<size_t>(H) * a.lpad;
    char* ws = static_cast<char*>(workspace);
    size_t off = kStatusBytes;
    a.status = reinterpret_cast<int*>(ws);
    a.cu_tiles = reinterpret_cast<int32_t*>(ws + off);
    off += align256((static_cast<size_t>(B) + 1) * sizeof(int32_t));
    a.delta = reinterpret_cast<float*>(ws + off);
    off += align256(lrows * sizeof(float));
    a.lse2 = reinterpret_cast<float*>(ws + off);
    off += align256(lrows * sizeof(float));
    a.dq_accum = reinterpret_cast<float*>(ws + off);
    a.ev_begin = g_ev_begin;
    a.ev_end = g_ev_end;
    if (cudaMemsetAsync(a.status, 0, sizeof(int) * 4, s) != cudaSuccess) return FA_ERR_CUDA;
    int n = 0;
    st = map_cuda(fa::launch_bwd(a, s, &n));
    if (st == FA_OK) g_last_launches = n;
    return st;
}

// Splits per head of a decode call: num_splits if given (at most one per 64
// keys), else enough CTAs for a few waves of two per SM while keeping at
// least 512 keys per split; then the keys per split, a multiple of 64.
static void decode_splits(int B, int H, int Nk, int num_splits, int* splits, int* split_keys) {
    const int max_s = (Nk + 63) / 64;
    int s = num_splits;
    if (s <= 0) {
        const long long heads = static_cast<long long>(B) * H;
        const long long want = (152LL * 2 * 3 + heads - 1) / heads;
        s = static_cast<int>(want < 1 ? 1 : want);
        const int by_len = (Nk + 511) / 512;
        if (s > by_len) s = by_len;
    }
    if (s > max_s) s = max_s;
    if (s < 1) s = 1;
    int keys = (Nk + s - 1) / s;
    keys = (keys + 63) / 64 * 64;
    *split_keys = keys;
    *splits = (Nk + keys - 1) / keys;
}

size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0) return 0;
    int S = 1, keys = 64;
    decode_splits(B, H, Nk, num_splits, &S, &keys);
    const size_t parts = static_cast<size_t>(B) * H * Nq * S;
    return kStatusBytes + 2 * align256(parts * sizeof(float)) + align256(parts * d * sizeof(float));
}

fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                    int d, float scale, const int32_t* cache_len, int num_splits, fa_dtype dtype, void* workspace,
                    size_t ws_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0 || d <= 0 || num_splits < 0) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (Nq > 8) return FA_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * H * Nk >= (1LL << 31) || B > 65535 || H > 65535) return FA_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        (cache_len && !aligned(cache_len, 4)) || !aligned(workspace, 256))
        return FA_ERR_INVALID_ARG;
    if (ws_bytes < fa_decode_workspace_size(B, H, Nq, Nk, d, num_splits)) return FA_ERR_INVALID_ARG;

    fa::DecodeArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.cache_len = cache_len;
    a.B = B;
    a.H = H;
    a.Nq = Nq;
    a.Nk = Nk;
    a.d = d;
    a.scale = scale;
    decode_splits(B, H, Nk, num_splits, &a.splits, &a.split_keys);
    const size_t parts = static_cast<size_t>(B) * H * Nq * a.splits;
    char* ws = static_cast<char*>(workspace);
    a.status = reinterpret_cast<int*>(ws);
    a.pm = reinterpret_cast<float*>(ws + kStatusBytes);
    a.pl = reinterpret_cast<float*>(ws + kStatusBytes + align256(parts * sizeof(float)));
    a.po = reinterpret_cast<float*>(ws + kStatusBytes + 2 * align256(parts * sizeof(float)));
    a.ev_begin = g_ev_begin;
    a.ev_end = g_ev_end;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(a.status, 0, sizeof(int) * 4, s) != cudaSuccess) return FA_ERR_CUDA;
    int n = 0;
    fa_status st = map_cuda(fa::launch_decode(a, s, &n));
    if (st == FA_OK) g_last_launches = n;
    return st;
}

size_t fa_fwd_fp8_workspace_size(int B, int H, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return 0;
    const size_t bhn = static_cast<size_t>(B) * H * N, bh = static_cast<size_t>(B) * H;
    const size_t tiles = bh * ((N + 127) / 128);
    return kStatusBytes + 3 * align256(bhn * d) + 3 * align256(tiles * sizeof(int)) + align256(bh * sizeof(int));
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                     float scale, int causal, const int32_t* kv_len, const float* signs, void* workspace,
                     size_t ws_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    fa_status st = check_shape(B, H, N, d, scale);
    if (st != FA_OK) return st;
    if (d != 128) return FA_ERR_UNSUPPORTED;
    if (N / 128 > 65535 || static_cast<long long>(B) * H > 65535) return FA_ERR_UNSUPPORTED;  // quantisation grids
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        (signs && !aligned(signs, 4)) || !aligned(workspace, 256) || (kv_len && !aligned(kv_len, 4)))
        return FA_ERR_INVALID_ARG;
    if (ws_bytes < fa_fwd_fp8_workspace_size(B, H, N, d)) return FA_ERR_INVALID_ARG;
    const size_t bhn = static_cast<size_t>(B) * H * N, bh = static_cast<size_t>(B) * H;
    const size_t tiles = bh * (N / 128);
    char* ws = static_cast<char*>(workspace);
    size_t off = kStatusBytes;
    fa::Fp8Args a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.N = N;
    a.scale = scale;
    a.causal = causal;
    a.kv_len = kv_len;
    a.signs = signs;
    a.status = reinterpret_cast<int*>(ws);
    a.q8 = reinterpret_cast<uint8_t*>(ws + off);
    off += align256(bhn * d);
    a.k8 = reinterpret_cast<uint8_t*>(ws + off);
    off += align256(bhn * d);
    a.vt8 = reinterpret_cast<uint8_t*>(ws + off);
    off += align256(bhn * d);
    a.qexp = reinterpret_cast<int*>(ws + off);
    off += align256(tiles * sizeof(int));
    a.kexp = reinterpret_cast<int*>(ws + off);
    off += align256(tiles * sizeof(int));
    a.vexp = reinterpret_cast<int*>(ws + off);
    off += align256(bh * sizeof(int));
    a.vblk_max = reinterpret_cast<float*>(ws + off);
    a.ev_begin = g_ev_begin;
    a.ev_end = g_ev_end;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(a.status, 0, sizeof(int) * 4, s) != cudaSuccess) return FA_ERR_CUDA;
    int n = 0;
    st = map_cuda(fa::launch_fwd_fp8(a, s, &n));
    if (st == FA_OK) g_last_launches = n;
    return st;
}

// Dropout parameters: byte threshold t = round(256 p) (<= 255), its keep rate.
static bool make_dropout(float p, unsigned long long seed, fa::DropoutArgs* d) {
    if (!(p >= 0.f) || !(p < 1.f)) return false;
    int t = static_cast<int>(lrintf(256.f * p));
    if (t > 255) t = 255;
    d->seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFull);
    d->seed_hi = static_cast<uint32_t>(seed >> 32);
    d->t4 = static_cast<uint32_t>(t) * 0x01010101u;
    d->inv_keep = 256.f / static_cast<float>(256 - t);
    return true;
}

fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                         float scale, int causal, const int32_t* kv_len, float dropout_p, unsigned long long seed,
                         void* workspace, size_t ws_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    fa_status st = check_shape(B, H, N, d, scale);
    if (st != FA_OK) return st;
    fa::FwdArgs a{};
    if (!make_dropout(dropout_p, seed, &a.drop)) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        !aligned(workspace, 256) || (kv_len && !aligned(kv_len, 4)))
        return FA_ERR_INVALID_ARG;
    if (ws_bytes < kStatusBytes) return FA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.kv_len = kv_len;
    a.dropout = 1;
    a.status = static_cast<int*>(workspace);
    a.ev_begin = g_ev_begin;
    a.ev_end = g_ev_end;
    if (cudaMemsetAsync(a.status, 0, sizeof(int) * 4, s) != cudaSuccess) return FA_ERR_CUDA;
    int n = 0;
    st = map_cuda(fa::launch_fwd(a, s, &n));
    if (st == FA_OK) g_last_launches = n;
    return st;
}

fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, const int32_t* kv_len, float dropout_p, unsigned long long seed, void* workspace,
                         size_t ws_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    fa_status st = check_shape(B, H, N, d, scale);
    if (st != FA_OK) return st;
    fa::BwdArgs a{};
    if (!make_dropout(dropout_p, seed, &a.drop)) return FA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
        !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 16) ||
        !aligned(workspace, 256) || (kv_len && !aligned(kv_len, 4)))
        return FA_ERR_INVALID_ARG;
    if (ws_bytes < fa_bwd_workspace_size(B, H, N, d)) return FA_ERR_INVALID_ARG;
    const size_t rows = static_cast<size_t>(B) * H * N;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.kv_len = kv_len;
    a.dropout = 1;
    char* ws = static_cast<char*>(workspace);
    a.status = reinterpret_cast<int*>(ws);
    a.delta = reinterpret_cast<float*>(ws + kStatusBytes);
    a.lse2 = reinterpret_cast<float*>(ws + kStatusBytes + align256(rows * sizeof(float)));
    a.dq_accum = reinterpret_cast<float*>(ws + kStatusBytes + 2 * align256(rows * sizeof(float)));
    a.ev_begin = g_ev_begin;
    a.ev_end = g_ev_end;
    if (cudaMemsetAsync(a.status, 0, sizeof(int) * 4, s) != cudaSuccess) return FA_ERR_CUDA;
    int n = 0;
    st = map_cuda(fa::launch_bwd(a, s, &n));
    if (st == FA_OK) g_last_launches = n;
    return st;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                 const uint8_t* blockmask, const int32_t* kv_len, fa_dtype dtype, void* workspace, size_t ws_bytes,
                 void* stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16 && dtype != FA_FP32) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    fa_status st = check_shape(B, H, N, d, scale);
    if (st != FA_OK) return st;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
        !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 16) ||
        !aligned(workspace, 256) || (kv_len && !aligned(kv_len, 4)))
        return FA_ERR_INVALID_ARG;
    if (dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    if (ws_bytes < fa_bwd_workspace_size(B, H, N, d)) return FA_ERR_INVALID_ARG;

    const size_t rows = static_cast<size_t>(B) * H * N;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    fa::BwdArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal;
    a.blockmask = blockmask;
    a.kv_len = kv_len;
    char* ws = static_cast<char*>(workspace);
    a.status = reinterpret_cast<int*>(ws);
    a.delta = reinterpret_cast<float*>(ws + kStatusBytes);
    a.lse2 = reinterpret_cast<float*>(ws + kStatusBytes + align256(rows * sizeof(float)));
    a.dq_accum = reinterpret_cast<float*>(ws + kStatusBytes + 2 * align256(rows * sizeof(float)));
    a.ev_begin = g_ev_begin;
    a.ev_end = g_ev_end;
    if (cudaMemsetAsync(a.status, 0, sizeof(int) * 4, s) != cudaSuccess) return FA_ERR_CUDA;
    int n = 0;
    st = map_cuda(fa::launch_bwd(a, s, &n));
    if (st == FA_OK) g_last_launches = n;
    return st;
}

fa_status fa_get_status(void* workspace, void* stream) {
    if (!workspace) return FA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
    if (word == 0) return FA_OK;
    if (cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    if ((word & 0xFF) == FA_ERR_TIMEOUT) return FA_ERR_TIMEOUT;
    if ((word & 0xFF) == FA_ERR_INVALID_ARG) return FA_ERR_INVALID_ARG;
    return FA_ERR_CUDA;
}

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: unsupported size or type";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA runtime or launch error";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a device-side wait gave up";
    }
    return "unknown fa_status";
}

int fa_last_launch_count(void) { return g_last_launches; }

fa_status fa_set_timing_events(void* begin, void* end) {
    if ((begin == nullptr) != (end == nullptr)) return FA_ERR_INVALID_ARG;
    g_ev_begin = static_cast<cudaEvent_t>(begin);
    g_ev_end = static_cast<cudaEvent_t>(end);
    return FA_OK;
}

}  // extern "C"

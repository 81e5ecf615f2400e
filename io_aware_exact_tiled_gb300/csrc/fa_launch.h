// Internal interface between the C-ABI layer (fa_api.cu) and the kernel
// launchers (fa_fwd.cu, fa_bwd.cu). Arguments are already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_philox.cuh"

namespace fa {

struct FwdArgs {
    const void *q, *k, *v;
    void* o;
    float* lse;
    int B, H, N, d;
    float scale;
    int causal;
    const uint8_t* blockmask;
    const int32_t* kv_len;
    int fp32;
    void* fp32_scratch;  // fp32 only: V^T [B,H,d,N], then Qh, Ql, Kh, Kl [B,H,N,d]
    int* status;
    cudaEvent_t ev_begin, ev_end;  // optional, recorded around the main kernel
    // Packed variable-length batch (bf16 only): q, k, v, o are [total, H, d],
    // lse is [H, total], sequence b is tokens cu_seqlens[b] .. cu_seqlens[b+1]-1
    // and N is the longest sequence. Null for the [B, H, N, d] layout.
    const int32_t* cu_seqlens;
    int total;
    // dropout on the probabilities (bf16, no tile mask, no packed batch)
    int dropout;
    DropoutArgs drop;
};

struct BwdArgs {
    const void *q, *k, *v, *o, *dout;
    const float* lse;
    void *dq, *dk, *dv;
    int B, H, N, d;
    float scale;
    int causal;
    const uint8_t* blockmask;
    const int32_t* kv_len;
    float* delta;     // [B,H,N] scratch: -D = -rowsum(dO * O)
    float* lse2;      // [B,H,N] scratch: -L in log2 units
    float* dq_accum;  // [B,H,N,d] fp32 scratch
    int* status;
    cudaEvent_t ev_begin, ev_end;  // optional, recorded around the main kernel
    // Packed variable-length batch (see FwdArgs): q, k, v, o, dout, dq, dk,
    // dv and dq_accum are [total, H, d], lse is [H, total]; delta and lse2
    // are [H][lpad] with each sequence starting at a multiple of 128 rows
    // (cu_tiles[b] * 128, cu_tiles being the running count of 128-row tiles,
    // computed on the device into the workspace). Null for [B, H, N, d].
    const int32_t* cu_seqlens;
    int32_t* cu_tiles;  // [B + 1] scratch
    int total;
    long long lpad;     // rows per head of delta / lse2: align128(total) + 128 * B
    int dropout;
    DropoutArgs drop;
};

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream, int* nlaunch);
cudaError_t launch_fwd_bf16_t1(const FwdArgs& a, cudaStream_t stream, int* nlaunch);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t stream, int* nlaunch);

}  // namespace fa

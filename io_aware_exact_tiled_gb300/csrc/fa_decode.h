// Internal interface of the split-key decoding kernels (fa_decode.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Kernel parameters. Partial results of split c of query row
// (b, h, qi) = row: pm[row * S + c] (maximum, log2 units, scale applied),
// pl[row * S + c] (sum of exp2(s - m)), po[(row * S + c) * d + :]
// (unnormalised output).
struct DecodeParams {
    const void* q;           // [B,H,Nq,d] bf16
    void* o;                 // [B,H,Nq,d] bf16
    float* lse;              // [B,H,Nq] fp32
    const int32_t* cache_len;  // [B] or null (= Nk)
    int B, H, Nq, Nk;
    int S;      // splits per head
    int split;  // keys per split (multiple of 64)
    float scale_log2;
    float *pm, *pl, *po;
    int* status;
};

struct DecodeArgs {
    const void *q, *k, *v;
    void* o;
    float* lse;
    const int32_t* cache_len;
    int B, H, Nq, Nk, d;
    float scale;
    int splits, split_keys;
    float *pm, *pl, *po;
    int* status;
    cudaEvent_t ev_begin, ev_end;  // optional, recorded around the split kernel
};

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream, int* nlaunch);

}  // namespace fa

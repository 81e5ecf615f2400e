// Internal interface of the FP8 forward path (fa_fwd_fp8.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

struct Fp8Args {
    const void *q, *k, *v;  // [B,H,N,128] bf16
    void* o;                // [B,H,N,128] bf16
    float* lse;             // [B,H,N]
    int B, H, N;
    float scale;
    int causal;
    const int32_t* kv_len;  // [B] or null
    const float* signs;     // [128] +-1: the random signs of the rotation; null: no rotation
    // workspace
    uint8_t *q8, *k8;       // [B,H,N,128] E4M3 (rotated Q, K)
    uint8_t* vt8;           // [B,H,128,N] E4M3 (V transposed)
    int *qexp, *kexp;       // [B,H,N/128] block scale exponents
    int* vexp;              // [B,H]
    float* vblk_max;        // [B,H,N/128] max |v| per 128-row block (scratch)
    int* status;
    cudaEvent_t ev_begin, ev_end;  // optional, recorded around the attention kernel
};

cudaError_t launch_fwd_fp8(const Fp8Args& a, cudaStream_t stream, int* nlaunch);

}  // namespace fa

// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory themselves.
//
// fa_bwd needs a caller-supplied workspace (the fp32 dQ accumulator, the row
// sums D = rowsum(dO * O), L in log2 units and a status word). Some callers
// have no way to provide one at the moment they run the backward pass: a
// plug-in hosted by a runtime that hands it tensors but no allocator, or a
// latency-critical loop that must not call cudaMalloc / cudaFree because
// those calls can synchronise the whole device and stall other streams. This
// entry point serves them with a scratch buffer that lives in the library
// itself: a file-scope device array of fixed size, created when the library's
// device code is loaded and kept by every GPU that loads it until the process
// exits. Nothing is allocated per call.
//
// Limits and sharing:
//  * The scratch holds kNoAllocScratchBytes (32 MiB). A call whose workspace
//    (fa_bwd_workspace_size(B, H, N, d)) does not fit is rejected with
//    FA_ERR_UNSUPPORTED before anything is launched.
//  * Every call on a device uses the same array, which keeps whatever the
//    previous call left in it. The backward pass re-initialises what must
//    start at zero (the dQ accumulator and the status word) on every call.
//    Two calls that can run at the same time on the GPU (on different streams,
//    or from different host threads without ordering) race on the array and
//    give wrong results; order them on one stream.
//  * The device address of the array is looked up once per device, on the
//    first call made while that device is current (cudaGetSymbolAddress). Make
//    that first call on each device before any stream capture begins. The
//    address is cached for the life of the process: cudaDeviceReset unloads
//    the library's device code, so after a reset this entry point must not be
//    called again on that device.
//  * A device-side wait that gives up records FA_ERR_TIMEOUT in the array's
//    status word; fa_bwd_noalloc_get_status reads and clears it.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fa.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself. Host code must not use this name as a pointer: on the
// host it only identifies the symbol; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_bwd_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_bwd_scratch on the current device (looked up once per
// device), or null if the lookup failed.
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || !ptr) return nullptr;
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                    const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                    float scale, int causal, const uint8_t* blockmask, const int32_t* kv_len,
                                    fa_dtype dtype, void* stream) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0) return FA_ERR_INVALID_ARG;
    if (fa_bwd_workspace_size(B, H, N, d) > kNoAllocScratchBytes) return FA_ERR_UNSUPPORTED;
    void* scratch = scratch_on_current_device();
    if (!scratch) return FA_ERR_CUDA;
    return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, blockmask, kv_len, dtype, scratch,
                  kNoAllocScratchBytes, stream);
}

extern "C" fa_status fa_bwd_noalloc_get_status(void* stream) {
    void* scratch = scratch_on_current_device();
    if (!scratch) return FA_ERR_CUDA;
    // the status word sits at the start of the scratch, as in any fa_bwd workspace
    return fa_get_status(scratch, stream);
}

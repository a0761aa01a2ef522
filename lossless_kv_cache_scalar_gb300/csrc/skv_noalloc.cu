// skv_noalloc.cu -- skv_decode_noalloc: whole-stream decode whose scratch
// lives in a fixed array inside this library instead of a caller workspace.
//
// For callers that cannot call cudaMalloc or hand over a workspace: a host
// application whose device memory is owned by its own pool and which gives a
// plugin no allocator, or a latency-critical path where an allocation (and the
// device synchronisation cudaFree implies) is not allowed. This variant needs
// no workspace argument; its scratch (the P_hat table and the per-channel
// 1/sigma table that skv_decode keeps in the caller's workspace) is a
// file-scope device array of SKV_NOALLOC_SCRATCH_BYTES, which every GPU that
// loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "skv.h"

namespace {

constexpr unsigned long long kScratchBytes = SKV_NOALLOC_SCRATCH_BYTES;

// The scratch itself. In host code this name is only a host-side stand-in;
// kernels get the device address looked up below.
static __device__ __align__(256) unsigned char skv_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];   // device address per device ordinal, once looked up
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device; looked up once
// per device, with that device current, on the first call made on it.
int32_t scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, skv_noalloc_scratch) != cudaSuccess || !p) return SKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SKV_OK;
}

}  // namespace

extern "C" int32_t skv_decode_noalloc(const skv_layout *lay, const void *bitstream,
                                      uint64_t bitstream_bytes, const uint64_t *offsets,
                                      const void *mu, const float *sigma, const uint64_t *counts,
                                      void *kv_out, int32_t *status, void *stream) {
    uint64_t need = 0;
    const int32_t r = skv_workspace_bytes(lay, 0, &need);
    if (r != SKV_OK) return r;
    if (need > kScratchBytes) return SKV_ERR_INVALID_ARG;   // layout too large for the fixed scratch
    void *ws = nullptr;
    const int32_t a = scratch_address(&ws);
    if (a != SKV_OK) return a;
    return skv_decode(lay, bitstream, bitstream_bytes, offsets, mu, sigma, counts, kv_out, status,
                      ws, kScratchBytes, stream);
}

// skv_peak.cu -- issue-rate probes for the arithmetic roofline of the coder.
//
// The coder's kernels are bound by 32-bit integer and binary32 arithmetic,
// not by memory or tensor cores, so their roofline needs the rate at which an
// SM issues those operations. Each probe keeps every SM full (8 CTAs of 256
// threads) and every thread busy with 8 independent dependency chains of one
// operation written as inline PTX (so the optimiser neither folds nor drops
// it), and reports operations per second. The mixed probe interleaves the four
// kinds 1:1:1:1, close to the coder's own mix.
#include <cuda_runtime.h>

#include <cstdint>

namespace skv {

constexpr int kPeakChains = 8;
constexpr int kPeakUnroll = 16;

template <int KIND>
__device__ __forceinline__ void step(uint32_t (&u)[kPeakChains], float (&f)[kPeakChains], uint32_t k) {
#pragma unroll
    for (int c = 0; c < kPeakChains; ++c) {
        if (KIND == 0) {          // three-input integer add
            asm volatile("add.u32 %0, %0, %1;\n\tadd.u32 %0, %0, %2;" : "+r"(u[c]) : "r"(k), "r"(u[(c + 1) % kPeakChains]));
        } else if (KIND == 1) {   // three-input logic
            asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(u[c]) : "r"(k), "r"(u[(c + 3) % kPeakChains]));
        } else if (KIND == 2) {   // integer multiply-add
            asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(u[c]) : "r"(k | 1u), "r"(u[(c + 5) % kPeakChains]));
        } else if (KIND == 3) {   // binary32 multiply
            asm volatile("mul.rn.f32 %0, %0, %1;" : "+f"(f[c]) : "f"(1.0000001f));
        } else {                  // the four kinds in turn
            const int kk = c & 3;
            if (kk == 0) asm volatile("add.u32 %0, %0, %1;\n\tadd.u32 %0, %0, %2;" : "+r"(u[c]) : "r"(k), "r"(u[(c + 1) % kPeakChains]));
            else if (kk == 1) asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(u[c]) : "r"(k), "r"(u[(c + 3) % kPeakChains]));
            else if (kk == 2) asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(u[c]) : "r"(k | 1u), "r"(u[(c + 5) % kPeakChains]));
            else asm volatile("mul.rn.f32 %0, %0, %1;" : "+f"(f[c]) : "f"(1.0000001f));
        }
    }
}

// Operations issued per chain per step: the add probe's two PTX adds may fuse
// into one three-input add, so it counts as two 32-bit operations either way
// (the algorithmic counts also count a + b + c as two).
template <int KIND>
__global__ void __launch_bounds__(256) peak_kernel(uint32_t iters, uint32_t seed, uint32_t *sink) {
    uint32_t u[kPeakChains];
    float f[kPeakChains];
#pragma unroll
    for (int c = 0; c < kPeakChains; ++c) {
        u[c] = seed ^ (threadIdx.x * 0x9E3779B9u + c);
        f[c] = 1.0f + (float)c * 1e-3f;
    }
    const uint32_t k = seed | 1u;
    for (uint32_t i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < kPeakUnroll; ++j) step<KIND>(u, f, k + i);
    }
    uint32_t acc = 0;
#pragma unroll
    for (int c = 0; c < kPeakChains; ++c) acc ^= u[c] ^ __float_as_uint(f[c]);
    if (acc == 0x12345678u) sink[0] = acc;            // keeps the chains live
}

int launch_peak(int kind, uint32_t iters, uint32_t *sink, uint32_t blocks, cudaStream_t st) {
    switch (kind) {
        case 0: peak_kernel<0><<<blocks, 256, 0, st>>>(iters, 7u, sink); break;
        case 1: peak_kernel<1><<<blocks, 256, 0, st>>>(iters, 7u, sink); break;
        case 2: peak_kernel<2><<<blocks, 256, 0, st>>>(iters, 7u, sink); break;
        case 3: peak_kernel<3><<<blocks, 256, 0, st>>>(iters, 7u, sink); break;
        default: peak_kernel<4><<<blocks, 256, 0, st>>>(iters, 7u, sink); break;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

// 32-bit operations one launch issues: threads x iters x unroll x chains x
// (2 for the add probe, 1 for the others; the mix averages 5/4).
uint64_t peak_ops(int kind, uint32_t iters, uint32_t blocks) {
    const uint64_t per = (uint64_t)blocks * 256u * iters * kPeakUnroll;
    if (kind == 0) return per * kPeakChains * 2u;
    if (kind == 4) return per * (kPeakChains / 4u) * 5u;
    return per * kPeakChains;
}

}  // namespace skv

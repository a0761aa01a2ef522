// skv_calib.cu -- the two steps just before the coder: the code histogram
// behind p_hat, and the per-channel calibration of sigma.
//
// The Speculative KV Coding wiki's mixture section takes p_hat as the
// empirical marginal of the codes; its predictor-choice section, and the
// predictor-engineering section of the blog "推测性KV编码", take sigma as a
// per-(kv, head, channel) residual scale, measured once on calibration tokens
// and then frozen. The blog's information-theory section gives the scale that
// minimises the Gaussian code length: the mean squared residual about mu.
#include <cuda_runtime.h>

#include "skv_model.cuh"

namespace skv {

// ---------------------------------------------------------------- histogram

// bf16: all 65,536 u32 bins (256 KB) do not fit one CTA's shared memory, but
// the codes whose biased exponent is below 192 (|value| < 2^65, both signs:
// 2 x 24,576 codes, 192 KB) do, and a KV cache holds almost nothing else. So
// each CTA (one per SM) counts those in shared memory and adds the rest (if
// any) straight to the u64 counts in global memory; at the end it adds its
// nonzero shared bins to the counts. The result is exact for any input; only
// the speed depends on the values.
constexpr int kHistThreads = 1024;
constexpr int kHistUnroll = 4;             // 16-byte loads in flight per thread
constexpr uint32_t kHistHalf = 192u << 7;  // codes per sign kept in shared memory
constexpr int kHistSmem = 2 * kHistHalf * sizeof(uint32_t);

__global__ void __launch_bounds__(kHistThreads, 1)
    hist_bf16_kernel(const uint16_t *__restrict__ codes, uint64_t n, uint32_t head,
                     unsigned long long *__restrict__ counts) {
    extern __shared__ uint32_t bins[];     // [sign][code & 0x7FFF < kHistHalf]
    for (uint32_t i = threadIdx.x; i < 2 * kHistHalf; i += blockDim.x) bins[i] = 0u;
    __syncthreads();
    auto add = [&](uint32_t code) {
        const uint32_t mag = code & 0x7FFFu;
        if (mag < kHistHalf) atomicAdd(&bins[(code >> 15) * kHistHalf + mag], 1u);
        else atomicAdd(counts + code, 1ull);
    };
    auto add2 = [&](uint32_t w) { add(w & 0xFFFFu); add(w >> 16); };
    // codes[head .. head + 8 nvec) are 16-byte aligned; the rest go one by one
    const uint64_t nvec = (n - head) / 8;
    const uint4 *vec = reinterpret_cast<const uint4 *>(codes + head);
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint64_t v = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; v + (kHistUnroll - 1) * stride < nvec; v += kHistUnroll * stride) {
        uint4 q[kHistUnroll];
#pragma unroll
        for (int u = 0; u < kHistUnroll; ++u) q[u] = __ldg(vec + v + u * stride);
#pragma unroll
        for (int u = 0; u < kHistUnroll; ++u) { add2(q[u].x); add2(q[u].y); add2(q[u].z); add2(q[u].w); }
    }
    for (; v < nvec; v += stride) {
        const uint4 q = __ldg(vec + v);
        add2(q.x); add2(q.y); add2(q.z); add2(q.w);
    }
    if (blockIdx.x == 0) {
        const uint64_t tail0 = head + 8 * nvec;
        if (threadIdx.x < head) add(codes[threadIdx.x]);
        if (threadIdx.x < n - tail0) add(codes[tail0 + threadIdx.x]);
    }
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < 2 * kHistHalf; i += blockDim.x) {
        const uint32_t c = bins[i];
        const uint32_t code = (i >= kHistHalf ? 0x8000u : 0u) | (i % kHistHalf);
        if (c) atomicAdd(counts + code, (unsigned long long)c);
    }
}

// e4m3: 256 bins fit easily, so each warp keeps its own copy (fewer
// collisions between warps on the popular codes), summed at the end.
constexpr int kHist8Warps = 8;

__global__ void __launch_bounds__(kHist8Warps * 32) hist_e4m3_kernel(const uint8_t *__restrict__ codes,
                                                                     uint64_t n, uint32_t head,
                                                                     unsigned long long *__restrict__ counts) {
    __shared__ uint32_t bins[kHist8Warps][256];
    const uint32_t warp = threadIdx.x >> 5;
    for (uint32_t i = threadIdx.x; i < kHist8Warps * 256u; i += blockDim.x) (&bins[0][0])[i] = 0u;
    __syncthreads();
    uint32_t *mine = bins[warp];
    auto add4 = [&](uint32_t w) {
        atomicAdd(mine + (w & 0xFFu), 1u);
        atomicAdd(mine + ((w >> 8) & 0xFFu), 1u);
        atomicAdd(mine + ((w >> 16) & 0xFFu), 1u);
        atomicAdd(mine + (w >> 24), 1u);
    };
    const uint64_t nvec = (n - head) / 16;
    const uint4 *vec = reinterpret_cast<const uint4 *>(codes + head);
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint64_t v = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; v + (kHistUnroll - 1) * stride < nvec; v += kHistUnroll * stride) {
        uint4 q[kHistUnroll];
#pragma unroll
        for (int u = 0; u < kHistUnroll; ++u) q[u] = __ldg(vec + v + u * stride);
#pragma unroll
        for (int u = 0; u < kHistUnroll; ++u) { add4(q[u].x); add4(q[u].y); add4(q[u].z); add4(q[u].w); }
    }
    for (; v < nvec; v += stride) {
        const uint4 q = __ldg(vec + v);
        add4(q.x); add4(q.y); add4(q.z); add4(q.w);
    }
    if (blockIdx.x == 0) {
        const uint64_t tail0 = head + 16 * nvec;
        if (threadIdx.x < head) atomicAdd(mine + codes[threadIdx.x], 1u);
        if (threadIdx.x < n - tail0) atomicAdd(mine + codes[tail0 + threadIdx.x], 1u);
    }
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < 256u; i += blockDim.x) {
        uint32_t c = 0;
#pragma unroll
        for (int w = 0; w < kHist8Warps; ++w) c += bins[w][i];
        if (c) atomicAdd(counts + i, (unsigned long long)c);
    }
}

// -------------------------------------------------------- sigma calibration

// One thread per (plane, sigma block, channel); consecutive threads take
// consecutive channels, so each token row is read coalesced. Over the first
// t_cal tokens of the block (the plane's first t_cal tokens without sigma
// blocks), in ascending order, an element counts when its KV and mu codes are both finite
// and its mask byte (if a mask is given) is nonzero:
//     r = fl64(value(kv) - value(mu)),  S = S + fl64(r * r)  (binary64 throughout)
//     sigma = fl32(sqrt(fl64(S / n_counted)))
// then clamped into the valid range [2^-126, FLT_MAX] (no counted element gives
// 2^-126). Every step is an IEEE round-to-nearest operation named by its
// intrinsic, in a fixed order, so the result is exact and reproducible.
constexpr int kCalibThreads = 256;
constexpr int kCalibBatch = 8;        // token rows loaded ahead of the serial sum

struct CalibArgs {
    Geom g;
    const uint8_t *kv, *mu, *mask;
    uint64_t t_cal;
    float *sigma;
};

// Exact binary64 value of a finite code, assembled with integer operations
// (GB300 issues few binary64 operations per clock; this leaves them for the
// subtract, multiply and add that the definition needs). A code's value has
// at most 8 significant bits, so it always fits: normal codes rebias the
// exponent, subnormal codes normalise their mantissa m as 2^k (1 + f).
template <uint32_t DT>
__device__ __forceinline__ double code_f64(uint32_t b) {
    constexpr uint32_t mbits = DT == SKV_BF16 ? 7u : 3u;       // mantissa bits
    constexpr int ebias = DT == SKV_BF16 ? 127 : 7;
    constexpr int sub_exp = 1 - ebias - (int)mbits;           // value of a subnormal's unit: 2^sub_exp
    const uint32_t sign = (b >> (mbits + (DT == SKV_BF16 ? 8u : 4u))) & 1u;
    const uint32_t e = (b >> mbits) & (DT == SKV_BF16 ? 0xFFu : 0xFu);
    const uint32_t m = b & ((1u << mbits) - 1u);
    uint32_t hi;
    if (e != 0u) {
        hi = ((uint32_t)(e - ebias + 1023) << 20) | (m << (20u - mbits));
    } else if (m != 0u) {
        const uint32_t k = 31u - __clz(m);                    // m = 2^k + rest
        hi = ((uint32_t)((int)k + sub_exp + 1023) << 20) | ((m - (1u << k)) << (20u - k));
    } else {
        hi = 0u;
    }
    return __hiloint2double((int)(hi | (sign << 31)), 0);
}

template <uint32_t DT>
__global__ void __launch_bounds__(kCalibThreads) calib_kernel(const CalibArgs a) {
    using K = Codes<DT>;
    const Geom &g = a.g;
    const uint64_t id = (uint64_t)blockIdx.x * kCalibThreads + threadIdx.x;
    if (id >= g.n_planes * g.n_sblk * g.HD) return;
    const uint64_t row = id / g.HD, c = id % g.HD;        // row = plane * n_sblk + block
    const uint64_t plane = row / g.n_sblk, blk = row % g.n_sblk;
    const uint64_t t_first = blk * g.SB;                  // 0 without sigma blocks
    const uint64_t t_cal = a.t_cal < g.T - t_first ? a.t_cal : g.T - t_first;
    const uint64_t e0 = (plane * g.T + t_first) * g.HD + c;   // element of the first token
    auto load = [&](const uint8_t *p, uint64_t el) -> uint32_t {
        return K::bytes == 2 ? __ldg(reinterpret_cast<const uint16_t *>(p) + el) : __ldg(p + el);
    };
    double S = 0.0;
    uint64_t cnt = 0;
    for (uint64_t t0 = 0; t0 < t_cal; t0 += kCalibBatch) {
        uint32_t kb[kCalibBatch], mb[kCalibBatch], keep[kCalibBatch];
#pragma unroll
        for (int i = 0; i < kCalibBatch; ++i) {
            const uint64_t t = t0 + i;
            const bool in = t < t_cal;
            const uint64_t el = e0 + (in ? t : 0) * g.HD;
            kb[i] = load(a.kv, el);
            mb[i] = load(a.mu, el);
            keep[i] = in && (a.mask == nullptr || __ldg(a.mask + el) != 0);
        }
#pragma unroll
        for (int i = 0; i < kCalibBatch; ++i) {
            if (keep[i] && K::finite(kb[i]) && K::finite(mb[i])) {
                const double r = __dsub_rn(code_f64<DT>(kb[i]), code_f64<DT>(mb[i]));
                S = __dadd_rn(S, __dmul_rn(r, r));
                ++cnt;
            }
        }
    }
    float s = 1.17549435e-38f;                            // 2^-126
    if (cnt) {
        const double rms = __dsqrt_rn(__ddiv_rn(S, (double)cnt));
        s = __double2float_rn(rms);
        if (!(s >= 1.17549435e-38f)) s = 1.17549435e-38f;
        if (s > 3.40282347e38f) s = 3.40282347e38f;
    }
    a.sigma[id] = s;
}

int launch_histogram(uint32_t dtype, const void *codes, uint64_t n, unsigned long long *counts,
                     cudaStream_t st) {
    if (n == 0) return 0;
    const uint32_t bytes = dtype == SKV_BF16 ? 2u : 1u;
    const uint32_t mis = (uint32_t)((uintptr_t)codes & 15u);
    uint64_t head = mis ? (16u - mis) / bytes : 0;
    if (head > n) head = n;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    if (dtype == SKV_BF16) {
        if (cudaFuncSetAttribute(hist_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kHistSmem) !=
            cudaSuccess)
            return 1;
        hist_bf16_kernel<<<(unsigned)sms, kHistThreads, kHistSmem, st>>>(static_cast<const uint16_t *>(codes),
                                                                          n, (uint32_t)head, counts);
    } else {
        hist_e4m3_kernel<<<(unsigned)(sms * 4), kHist8Warps * 32, 0, st>>>(
            static_cast<const uint8_t *>(codes), n, (uint32_t)head, counts);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_calibrate(const Geom &g, const void *kv, const void *mu, const uint8_t *mask,
                     uint64_t t_cal, float *sigma, cudaStream_t st) {
    const uint64_t threads = g.n_planes * g.n_sblk * g.HD;
    const uint64_t blocks = (threads + kCalibThreads - 1) / kCalibThreads;
    if (blocks == 0) return 0;
    const CalibArgs ca{g, static_cast<const uint8_t *>(kv), static_cast<const uint8_t *>(mu), mask,
                       t_cal, sigma};
    if (g.dtype == SKV_BF16)
        calib_kernel<SKV_BF16><<<(unsigned)blocks, kCalibThreads, 0, st>>>(ca);
    else
        calib_kernel<SKV_E4M3><<<(unsigned)blocks, kCalibThreads, 0, st>>>(ca);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace skv

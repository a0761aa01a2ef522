// skv_rq.cu -- lowering 2b-bit quantised KV codes to b bits, the progressive
// quantisation step of PM-KVQ that the third page (its PM-KVQ section) puts
// beside the coder.
//
// Equivalent Right Shift keeps the zero point and grows the scale to
// S_b = (2^b + 1) S_2b, so the new code is round(q / (2^b + 1)); the page
// notes this equals dequantising and requantising and needs only integer adds
// and shifts. Here: with t = q + 2^(b-1), a = t >> b and c = t mod 2^b,
// floor(t / (2^b + 1)) = a - [a > c] (t / (2^b + 1) = a - (a - c) / (2^b + 1)
// and |a - c| < 2^b + 1), and [a > c] = 1 - ((c - a + 2^b) >> b). The two
// shift baselines of the page's ablation are also provided: Direct Right Shift
// q >> b and Modified Right Shift min((q + 2^(b-1)) >> b, 2^b - 1).
//
// HBM-bound: each thread turns 32 bytes of 2b-bit codes into 16 bytes of
// b-bit codes with two 16-byte loads and one 16-byte store.
#include <cuda_runtime.h>

#include <cstdint>

namespace skv {

template <uint32_t B, uint32_t MODE>
__device__ __forceinline__ uint32_t lower(uint32_t q) {
    if (MODE == 1) return q >> B;                                   // direct right shift
    if (MODE == 2) return min((q + (1u << (B - 1))) >> B, (1u << B) - 1u);   // modified
    const uint32_t t = q + (1u << (B - 1));                         // equivalent right shift
    const uint32_t a = t >> B;
    return a - 1u + ((t - (a << B) - a + (1u << B)) >> B);
}

// 256 input bits (128 / B codes of 2B bits) -> 128 output bits.
template <uint32_t B, uint32_t MODE>
__device__ __forceinline__ uint4 lower_unit(const uint32_t (&w)[8]) {
    constexpr uint32_t W = 2u * B, N = 128u / B;
    uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (uint32_t i = 0; i < N; ++i) {
        const uint32_t q = (w[(W * i) / 32u] >> ((W * i) % 32u)) & ((W == 32u) ? 0xFFFFFFFFu : ((1u << W) - 1u));
        o[(B * i) / 32u] |= lower<B, MODE>(q) << ((B * i) % 32u);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// B = 4 (8 -> 4 bits), the same arithmetic four codes at a time, one per
// byte of a word. With q = 16 hi + lo: t = q + 8 gives a = t >> 4 = hi +
// [lo >= 8] <= 16 and c = t mod 16 = (lo + 8) mod 16, and every intermediate
// (lo + 8 <= 23, c + 16 - a in [0, 31], a + x >= 1) stays inside its byte.
template <uint32_t MODE>
__device__ __forceinline__ uint32_t lower4_word(uint32_t w) {
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu, lo = w & 0x0F0F0F0Fu;
    uint32_t r;
    if (MODE == 1) {
        r = hi;                                                      // q >> 4
    } else {
        const uint32_t lo8 = lo + 0x08080808u;
        const uint32_t a = hi + ((lo8 >> 4) & 0x01010101u);           // (q + 8) >> 4
        if (MODE == 2) {
            r = a - ((a >> 4) & 0x01010101u);                         // min(a, 15)
        } else {
            const uint32_t c = lo8 & 0x0F0F0F0Fu;
            const uint32_t x = ((c + 0x10101010u - a) >> 4) & 0x01010101u;   // [c >= a]
            r = a + x - 0x01010101u;                                  // a - [a > c]
        }
    }
    const uint32_t t = r | (r >> 4);                                  // codes 0|1 in byte 0, 2|3 in byte 2
    return (t & 0xFFu) | ((t >> 8) & 0xFF00u);
}

template <uint32_t B, uint32_t MODE>
__global__ void __launch_bounds__(256) rq_kernel(const uint8_t *__restrict__ in, uint64_t n,
                                                 uint8_t *__restrict__ out, const float *__restrict__ s_in,
                                                 float *__restrict__ s_out, uint64_t n_groups) {
    constexpr uint64_t N = 128u / B;                                // codes per unit
    const uint64_t units = n / N;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (uint64_t u = tid; u < units; u += stride) {
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(in) + 2 * u);
        const uint4 b = __ldg(reinterpret_cast<const uint4 *>(in) + 2 * u + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        if (B == 4) {
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = lower4_word<MODE>(w[2 * i]) | (lower4_word<MODE>(w[2 * i + 1]) << 16);
            reinterpret_cast<uint4 *>(out)[u] = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            reinterpret_cast<uint4 *>(out)[u] = lower_unit<B, MODE>(w);
        }
    }
    // the last, partial unit: whole bytes (n B is a multiple of 8)
    const uint64_t rest = n - units * N;
    if (rest && tid == 0) {
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        const uint64_t in_bytes = rest * 2u * B / 8u, out_bytes = rest * B / 8u;
        for (uint64_t i = 0; i < in_bytes; ++i) w[i / 4] |= (uint32_t)in[units * 32u + i] << (8u * (i % 4));
        const uint4 o = lower_unit<B, MODE>(w);
        const uint32_t ov[4] = {o.x, o.y, o.z, o.w};
        for (uint64_t i = 0; i < out_bytes; ++i) out[units * 16u + i] = (uint8_t)(ov[i / 4] >> (8u * (i % 4)));
    }
    // scales: (2^B + 1) S for ERS, 2^B S for the shifts (one rounding of the exact product)
    const float k = MODE == 0 ? (float)((1u << B) + 1u) : (float)(1u << B);
    for (uint64_t g = tid; g < n_groups; g += stride) s_out[g] = __fmul_rn(k, s_in[g]);
}

template <uint32_t B>
static void launch_b(uint32_t mode, const uint8_t *in, uint64_t n, uint8_t *out, const float *s_in,
                     float *s_out, uint64_t n_groups, unsigned grid, cudaStream_t st) {
    if (mode == 0) rq_kernel<B, 0><<<grid, 256, 0, st>>>(in, n, out, s_in, s_out, n_groups);
    else if (mode == 1) rq_kernel<B, 1><<<grid, 256, 0, st>>>(in, n, out, s_in, s_out, n_groups);
    else rq_kernel<B, 2><<<grid, 256, 0, st>>>(in, n, out, s_in, s_out, n_groups);
}

int launch_requantize(uint32_t mode, uint32_t b, const void *in, uint64_t n, void *out, const float *s_in,
                      float *s_out, uint64_t n_groups, cudaStream_t st) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    const uint64_t units = n / (128u / b) + 1u;
    uint64_t work = units > n_groups ? units : n_groups;
    uint64_t grid = (work + 255u) / 256u;
    const uint64_t cap = (uint64_t)sms * 8u;          // 8 CTAs of 256 threads per SM, grid-stride beyond
    if (grid > cap) grid = cap;
    const uint8_t *i8 = static_cast<const uint8_t *>(in);
    uint8_t *o8 = static_cast<uint8_t *>(out);
    switch (b) {
        case 1: launch_b<1>(mode, i8, n, o8, s_in, s_out, n_groups, (unsigned)grid, st); break;
        case 2: launch_b<2>(mode, i8, n, o8, s_in, s_out, n_groups, (unsigned)grid, st); break;
        case 4: launch_b<4>(mode, i8, n, o8, s_in, s_out, n_groups, (unsigned)grid, st); break;
        default: launch_b<8>(mode, i8, n, o8, s_in, s_out, n_groups, (unsigned)grid, st); break;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace skv

// skv_model.cuh -- the per-scalar mixture model and the rANS step, on the device.
//
// The model is the three-component mixture of the Speculative KV Coding wiki
// (mixture section): 0.95 N(mu, sigma^2) + 0.03 N(mu, (3 sigma)^2) +
// 0.02 p_hat, integrated over each code's rounding interval. Its integer form
// (SKV v1 format §5) must be bit-identical at encoder and decoder, which
// the 推测性KV编码 blog's deployment section demands of any arithmetic coder:
// every float step below is one IEEE binary32 operation with round-to-nearest,
// written with explicit _rn intrinsics so nothing is contracted into an FMA,
// and the build keeps subnormals (no -ftz).
#pragma once

#include <cstdint>

#include "phi_q24.h"
#include "skv_internal.h"

namespace skv {

// T[j + 2048] = round_half_even(2^24 Phi(j / 256)), SKV v1 format §3.
static __device__ const uint32_t kPhiQ24[4097] = {SKV_PHI_Q24_VALUES};

// Tables staged in shared memory by every CTA that evaluates the model: the
// Phi pairs (T[j], T[j+1] - T[j]) over [-8, 8] (entry 4096 = (2^24, 0)), or,
// WIDE, the same pairs extended over [-24, 24] with the saturated values
// ((0, 0) below -8, (2^24, 0) from 8 on), which give the same Phi_q without
// clamping z to [-8, 8] first (96 KB instead of 32 KB of shared memory).
template <bool WIDE> struct PhiTables {
    static constexpr int kCenter = WIDE ? 6144 : 2048;
    static constexpr uint32_t kEntries = 2u * kCenter + 1u;
    uint2 phi[kEntries];
};
using Tables = PhiTables<false>;
using TablesWide = PhiTables<true>;
struct Tables8 {         // e4m3 only: the whole alphabet fits on chip
    float edge[257];
    uint32_t phat[257];
    float value[256];    // value of each code (by bit pattern; NaN codes unused)
};

struct Weights {
    uint32_t n, w, h;    // narrow, wide, marginal; sum 100
};

// ---------------------------------------------------------------- code order

template <uint32_t DT> struct Codes;

template <> struct Codes<SKV_BF16> {
    static constexpr uint32_t N = 65536u, m = 24u, V = 8u, bytes = 2u;
    static constexpr uint64_t L = 1ull << 31;
    __device__ __forceinline__ static uint32_t ord(uint32_t b) {
        return b ^ ((b & 0x8000u) ? 0xFFFFu : 0x8000u);
    }
    __device__ __forceinline__ static uint32_t code(uint32_t o) {
        return o ^ ((o < 0x8000u) ? 0xFFFFu : 0x8000u);
    }
    __device__ __forceinline__ static bool finite(uint32_t b) { return (b & 0x7F80u) != 0x7F80u; }
    __device__ __forceinline__ static float value(uint32_t b) { return __uint_as_float(b << 16); }
    // Edge E(o) (SKV v1 format §2) straight from the bits: for a positive code
    // k >= 1 the binary32 pattern (k << 16) - 0x8000 lies half a bf16 step below
    // code k, which is the exact midpoint of codes k-1 and k (binary32 spacing is
    // uniform within a binade and the bf16 grid is a subset of it); negative
    // edges mirror positive ones, E(o) = -E(N - o).
    __device__ __forceinline__ static float edge(const Tables8 *, uint32_t o) {
        const int k = (int)o - 32768;
        const uint32_t a = (uint32_t)abs(k);
        uint32_t bits = (a << 16) - 0x8000u;
        bits = (a == 0u) ? 0u : bits;
        bits = (a > 0x7F7Fu) ? 0x7F800000u : bits;
        bits |= (k < 0) ? 0x80000000u : 0u;
        return __uint_as_float(bits);
    }
    __device__ __forceinline__ static uint32_t phat(const Tables8 *, const uint32_t *__restrict__ g,
                                                    uint32_t o) {
        return __ldg(g + o);
    }
    // element e of a 16-byte vector
    __device__ __forceinline__ static uint32_t get(const uint4 &v, int e) {
        const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
        return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
    }
    __device__ __forceinline__ static void put(uint4 &v, int e, uint32_t c) {
        uint32_t &w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
        w = (e & 1) ? ((w & 0xFFFFu) | (c << 16)) : ((w & 0xFFFF0000u) | c);
    }
};

template <> struct Codes<SKV_E4M3> {
    static constexpr uint32_t N = 256u, m = 16u, V = 16u, bytes = 1u;
    static constexpr uint64_t L = 1ull << 23;
    __device__ __forceinline__ static uint32_t ord(uint32_t b) {
        return b ^ ((b & 0x80u) ? 0xFFu : 0x80u);
    }
    __device__ __forceinline__ static uint32_t code(uint32_t o) {
        return o ^ ((o < 0x80u) ? 0xFFu : 0x80u);
    }
    __device__ __forceinline__ static bool finite(uint32_t b) { return (b & 0x7Fu) != 0x7Fu; }
    // OCP e4m3: bias 7, 3 mantissa bits, subnormals m * 2^-9, no infinity.
    __device__ __forceinline__ static float value(uint32_t b) {
        const uint32_t e = (b >> 3) & 15u, mt = b & 7u;
        float v = (e == 0u) ? __fmul_rn(__uint2float_rn(mt), 0.001953125f)
                            : __uint_as_float(((e + 120u) << 23) | (mt << 20));
        return (b & 0x80u) ? -v : v;
    }
    __device__ __forceinline__ static float edge(const Tables8 *t8, uint32_t o) { return t8->edge[o]; }
    __device__ __forceinline__ static uint32_t phat(const Tables8 *t8, const uint32_t *, uint32_t o) {
        return t8->phat[o];
    }
    __device__ __forceinline__ static uint32_t get(const uint4 &v, int e) {
        const uint32_t w = (e >> 2) == 0 ? v.x : (e >> 2) == 1 ? v.y : (e >> 2) == 2 ? v.z : v.w;
        return (w >> (8 * (e & 3))) & 0xFFu;
    }
    __device__ __forceinline__ static void put(uint4 &v, int e, uint32_t c) {
        uint32_t &w = (e >> 2) == 0 ? v.x : (e >> 2) == 1 ? v.y : (e >> 2) == 2 ? v.z : v.w;
        const int sh = 8 * (e & 3);
        w = (w & ~(0xFFu << sh)) | (c << sh);
    }
};

// Edge of ordinal o computed from the code values (SKV v1 format §2), used to
// fill the e4m3 edge table; the bf16 path uses the equivalent bit form above.
template <uint32_t DT>
__device__ float edge_from_values(uint32_t o) {
    using K = Codes<DT>;
    const uint32_t maxc = (DT == SKV_BF16) ? 0x7F7Fu : 0x7Eu;
    const uint32_t o_lo = K::ord(maxc | (K::N / 2)), o_hi = K::ord(maxc);
    if (o <= o_lo) return __int_as_float(0xFF800000);
    if (o > o_hi) return __int_as_float(0x7F800000);
    const float a = K::value(K::code(o - 1)), b = K::value(K::code(o));
    return __fadd_rn(__fmul_rn(0.5f, a), __fmul_rn(0.5f, b));
}

// Stage the Phi pairs into shared memory (no barrier).
template <bool WIDE>
__device__ void stage_phi(PhiTables<WIDE> &t) {
    constexpr int off = PhiTables<WIDE>::kCenter - 2048;     // entry of T[0]
    for (uint32_t i = threadIdx.x; i < PhiTables<WIDE>::kEntries; i += blockDim.x) {
        const int j = (int)i - off;
        uint2 e;
        if (j < 0) e = make_uint2(0u, 0u);
        else if (j >= 4096) e = make_uint2(1u << 24, 0u);
        else e = make_uint2(kPhiQ24[j], kPhiQ24[j + 1] - kPhiQ24[j]);
        t.phi[i] = e;
    }
}

// The e4m3 code tables (edge E(o) and P_hat(o) for o = 0..256, value of each
// code) lane-sliced in shared memory: entry i of lane l at word 32 i + l, so
// that the 32 lanes of a warp, each looking up its own code, hit 32 distinct
// banks (one shared copy makes those lookups collide on banks).
struct Sliced8 {
    static constexpr uint32_t kEdge = 0, kPhat = 257u * 32u, kValue = 2u * 257u * 32u;
    static constexpr uint32_t kWords = kValue + 256u * 32u;
    const uint32_t *p;   // the tables' base, offset to this lane's slice
    __device__ __forceinline__ explicit Sliced8(const void *base)
        : p(reinterpret_cast<const uint32_t *>(base) + (threadIdx.x & 31u)) {}
    __device__ __forceinline__ float edge(uint32_t o) const { return __uint_as_float(p[kEdge + (o << 5)]); }
    __device__ __forceinline__ uint32_t phat(uint32_t o) const { return p[kPhat + (o << 5)]; }
    __device__ __forceinline__ float value(uint32_t c) const { return __uint_as_float(p[kValue + (c << 5)]); }
};

// Stage the Phi pairs (and, for e4m3, the edges and P_hat) into shared memory.
template <uint32_t DT, bool WIDE>
__device__ void stage_tables(PhiTables<WIDE> &t, Tables8 &t8, const uint32_t *__restrict__ phat) {
    stage_phi(t);
    if (DT == SKV_E4M3) {
        for (uint32_t o = threadIdx.x; o <= 256u; o += blockDim.x) {
            t8.edge[o] = edge_from_values<SKV_E4M3>(o);
            t8.phat[o] = phat[o];
        }
        for (uint32_t b = threadIdx.x; b < 256u; b += blockDim.x) t8.value[b] = Codes<SKV_E4M3>::value(b);
    }
    __syncthreads();
}

// Fill the lane-sliced e4m3 tables at base (Sliced8::kWords words; no barrier).
__device__ inline void stage_sliced8(void *base, const uint32_t *__restrict__ phat) {
    uint32_t *sl = reinterpret_cast<uint32_t *>(base);
    for (uint32_t i = threadIdx.x; i < 257u * 32u; i += blockDim.x) {
        sl[Sliced8::kEdge + i] = __float_as_uint(edge_from_values<SKV_E4M3>(i >> 5));
        sl[Sliced8::kPhat + i] = phat[i >> 5];
        if (i < 256u * 32u) sl[Sliced8::kValue + i] = __float_as_uint(Codes<SKV_E4M3>::value(i >> 5));
    }
}

// -------------------------------------------------------------- model: C(o)
//
// C(o) of SKV v1 format §5 in a form that keeps most steps on the binary32
// pipe, each step exact:
//  - zq = floor(z 2^16): one multiply-add rounded down, z 2^16 + 1.5 2^23,
//    whose exact value lies in [2^23, 2^24) where binary32 spacing is 1, so the
//    rounding is the floor and the result's bit pattern is kMagicBits + zq;
//  - zw = floor(zq / 3): (zq + 3 2^19) is exact in binary32 (an integer below
//    2^22), and its product with the binary32 value just above 1/3 exceeds the
//    true quotient by less than 0.032, which never crosses the next integer
//    (the quotient's fraction is 0, 1/3 or 2/3), so a second multiply-add
//    rounded down gives floor((zq + 3 2^19) / 3) = zw + 2^19 in its bits;
//  - Phi_q's table position j and remainder r come from the biased bits
//    directly (the bias is a multiple of 256);
//  - floor(S (M - N) / 2^24) = hi32(2S (M - N) 2^7), then / 100 by the
//    multiply-high with ceil(2^37 / 100), exact for every 32-bit dividend.
// Every identity is exact over the whole range the format allows, so C(o) is
// bit-identical to the section 5 formula.

constexpr uint32_t kMagicBits = 0x4B400000u;     // bits of 1.5 2^23: bits = kMagicBits + integer part

// Phi_q at the grid position k held as b = bias + k (bias a multiple of 2^8).
template <bool WIDE>
__device__ __forceinline__ uint32_t phi_b(const PhiTables<WIDE> &t, uint32_t b, uint32_t bias) {
    const uint2 e = t.phi[(int)(b >> 8) - (int)(bias >> 8) + PhiTables<WIDE>::kCenter];
    return e.x + ((e.y * (b & 255u)) >> 8);
}

// C(o) for an element with predictor value mu and rs = fl32(1/sigma), from
// the edge E = E(o) and P_hat(o).
template <uint32_t DT, bool WIDE>
__device__ __forceinline__ uint32_t cdf_from(const PhiTables<WIDE> &t, const Weights w, float E, uint32_t ph,
                                             uint32_t o, float mu, float rs) {
    constexpr uint32_t MN = (1u << Codes<DT>::m) - Codes<DT>::N;
    float z = __fmul_rn(__fsub_rn(E, mu), rs);
    z = fminf(fmaxf(z, -24.0f), 24.0f);
    const float tq = __fmaf_rd(z, 65536.0f, 12582912.0f);          // bits: kMagicBits + zq
    const uint32_t bq = __float_as_uint(tq);
    const uint32_t bn = WIDE ? bq : min(max(bq, kMagicBits - 524288u), kMagicBits + 524288u);
    // bits: kMagicBits + 2^19 + zw
    const uint32_t bw = __float_as_uint(__fmaf_rd(__fadd_rn(tq, -11010048.0f), 0.333333343f, 12582912.0f));
    // 2S (< 2^32): the weights doubled
    const uint32_t S2 = (2u * w.n) * phi_b(t, bn, kMagicBits) + (2u * w.w) * phi_b(t, bw, kMagicBits + 524288u) +
                        (2u * w.h) * ph;
    return o + (__umulhi(__umulhi(S2, MN << 7), 0x51EB851Fu) >> 5);
}

// C(o) with the edge and P_hat from the code's own tables.
template <uint32_t DT, bool WIDE>
__device__ __forceinline__ uint32_t cdf(const PhiTables<WIDE> &t, const Tables8 *t8, const Weights w,
                                        const uint32_t *__restrict__ phat, uint32_t o, float mu,
                                        float rs) {
    using K = Codes<DT>;
    return cdf_from<DT>(t, w, K::edge(t8, o), K::phat(t8, phat, o), o, mu, rs);
}

// C(o) as cdf<SKV_BF16>, with the edge E(o) and P_hat(o) read as one pair
// from the per-call table ep (ep[o] = (bits of E(o), P_hat(o))) instead of
// being rebuilt from the code bits: one 8-byte load replaces the edge's
// integer work and the P_hat load.
template <bool WIDE>
__device__ __forceinline__ uint32_t cdf_ep(const PhiTables<WIDE> &t, const Weights w,
                                           const uint2 *__restrict__ ep, uint32_t o, float mu,
                                           float rs) {
    const uint2 e = __ldg(ep + o);
    return cdf_from<SKV_BF16>(t, w, __uint_as_float(e.x), e.y, o, mu, rs);
}

// ------------------------------------------------------------------- rANS

// Approximate reciprocal of f (one MUFU op), computed off the state chain.
__device__ __forceinline__ float recip(uint32_t f) {
    float rf;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rf) : "f"(__uint2float_rn(f)));
    return rf;
}

// q = floor(x / f), r = x mod f for f in [1, 2^24] and x < 2^39 f, given
// rf = recip(f) (relative error below 2^-22). The binary32 estimate gives q to
// within 2^17 + 1; one more estimate on the signed remainder lands within one
// step, fixed by a final compare.
__device__ __forceinline__ uint64_t divmod(uint64_t x, uint32_t f, float rf, uint32_t &r_out) {
    const uint64_t q1 = __float2ull_rz(__fmul_rn(__ull2float_rn(x), rf));
    long long r = (long long)(x - q1 * (uint64_t)f);
    const int q2 = __float2int_rn(__fmul_rn(__ll2float_rn(r), rf));
    r -= (long long)q2 * (long long)f;
    long long q = (long long)q1 + q2;
    if (r < 0) { r += f; q -= 1; }
    r_out = (uint32_t)r;
    return (uint64_t)q;
}

// Encode one symbol after renormalisation: x = (x / f) M + (x mod f) + c.
template <uint32_t DT>
__device__ __forceinline__ uint64_t rans_put(uint64_t x, uint32_t c, uint32_t f, float rf) {
    uint32_t r;
    const uint64_t q = divmod(x, f, rf, r);
    return (q << Codes<DT>::m) + r + c;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ void set_status(int32_t *status, int32_t code) {
    atomicCAS(status, 0, code);
}

}  // namespace skv

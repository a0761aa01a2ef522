// skv_peak.cu -- issue-rate probes for the arithmetic roofline of the coder.
//
// The coder's kernels are bound by 32-bit integer and binary32 arithmetic,
// not by memory or tensor cores, so their roofline needs the rate at which an
// SM executes that arithmetic. Two kinds of probe, both keeping every SM full
// (8 CTAs of 256 threads) and every thread busy with 8 independent dependency
// chains of operations written as inline PTX (so the optimiser neither folds
// nor drops them):
//
//  - one per instruction class of skv_ops.h (kind = the class), for the rate
//    of each class alone;
//  - one per operation table of skv_ops.h (kind = kNumOpClasses + table):
//    each loop iteration issues exactly the table's per-scalar counts, the
//    classes interleaved evenly, so the probe's scalars per second is the
//    fastest this GPU runs the format's own arithmetic: the arithmetic
//    roofline of the encode and decode kernels.
//
// Table lookups are pointer chases through a 32 KB shared-memory table (lds)
// and a 16 KB global table that stays in L1 (ldt), so each load's address is
// the previous load's data, as in the coder where a table index comes from
// arithmetic on loaded values. The 32 lanes of a warp read 32 consecutive
// 8-byte entries (no bank conflict, two cache lines): the best case of a
// table lookup, as a roofline wants.
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "skv_ops.h"

namespace skv {

constexpr int kChains = 8;
constexpr int kClassSteps = 16;          // single-class probe: steps per iteration
constexpr uint32_t kStabPairs = 4096;    // 32 KB shared table of (next, next) addresses
constexpr uint32_t kGtabPairs = 2048;    // 16 KB global table of (next, next) indices

static __device__ uint2 g_probe_table[kGtabPairs];

struct Chains {
    uint32_t u[kChains];
    float f[kChains];
    uint32_t s[kChains];     // shared-table addresses
    uint32_t g[kChains];     // global-table indices
    uint32_t d[kChains];     // this thread's store slots (shared addresses)
};

// One operation of class C on chain c.
template <int C>
__device__ __forceinline__ void op(Chains &x, int c, uint32_t k, const uint2 *gt) {
    const int c1 = (c + 1) & (kChains - 1), c3 = (c + 3) & (kChains - 1), c4 = c ^ 4;
    if (C == kOpFp32) {
        asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(x.f[c]) : "f"(0.99999f), "f"(x.f[c1]));
    } else if (C == kOpFminmax) {
        if (c & 1) asm volatile("min.f32 %0, %0, %1;" : "+f"(x.f[c]) : "f"(x.f[c3]));
        else asm volatile("max.f32 %0, %0, %1;" : "+f"(x.f[c]) : "f"(x.f[c3]));
    } else if (C == kOpIadd) {
        asm volatile("add.u32 %0, %0, %1;" : "+r"(x.u[c]) : "r"(x.u[c1]));
    } else if (C == kOpLogic) {
        asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(x.u[c]) : "r"(k), "r"(x.u[c3]));
    } else if (C == kOpShift) {
        asm volatile("shf.r.wrap.b32 %0, %0, %1, %2;" : "+r"(x.u[c]) : "r"(x.u[c3]), "r"(k));
    } else if (C == kOpIminmax) {
        if (c & 1) asm volatile("min.s32 %0, %0, %1;" : "+r"(x.u[c]) : "r"(x.u[c3]));
        else asm volatile("max.s32 %0, %0, %1;" : "+r"(x.u[c]) : "r"(x.u[c3]));
    } else if (C == kOpImad) {
        asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(x.u[c]) : "r"(k | 1u), "r"(x.u[c1]));
    } else if (C == kOpImadHi) {
        // hi(u * (2^32 - 1)) = u - 1 for u >= 1: a long-lived chain
        asm volatile("mul.hi.u32 %0, %0, %1;" : "+r"(x.u[c]) : "r"(k | 0xFFFFFFFFu));
    } else if (C == kOpImadWide) {
        // both halves of the product stay live (chains c and c ^ 4)
        asm volatile("{\n\t.reg .u64 t;\n\tmul.wide.u32 t, %0, %2;\n\tmov.b64 {%0, %1}, t;\n\t}"
                     : "+r"(x.u[c]), "+r"(x.u[c4]) : "r"(k | 1u));
    } else if (C == kOpCvt) {
        // chains c and c ^ 1 pass one value back and forth: float -> int -> float
        if (c & 1) asm volatile("cvt.rmi.s32.f32 %0, %1;" : "=r"(x.u[c]) : "f"(x.f[c ^ 1]));
        else asm volatile("cvt.rn.f32.s32 %0, %1;" : "=f"(x.f[c]) : "r"(x.u[c ^ 1]));
    } else if (C == kOpMufu) {
        // lg2 and ex2 in turn along the pair (c, c ^ 1)
        if (c & 1) asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(x.f[c]) : "f"(x.f[c ^ 1]));
        else asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(x.f[c]) : "f"(x.f[c ^ 1]));
    } else if (C == kOpPopc) {
        asm volatile("popc.b32 %0, %0;" : "+r"(x.u[c]));
    } else if (C == kOpVote) {
        asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\tvote.sync.ballot.b32 %0, p, 0xffffffff;\n\t}"
                     : "+r"(x.u[c]));
    } else if (C == kOpLds) {
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%0];" : "+r"(x.s[c]), "+r"(x.s[c4]));
    } else if (C == kOpLdt) {
        uint32_t a, b;
        asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "l"(gt + x.g[c]));
        x.g[c] = a;
        x.g[c4] = b;
    } else if (C == kOpSts) {
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(x.d[c]), "r"(x.u[c]) : "memory");
    }
}

// The classes of table T in an evenly interleaved order: position p takes the
// class furthest behind its share. A vote brings its own setp, which the table
// counts under logic, so logic gives up one place per vote.
template <int T> constexpr uint32_t mix_count(int c) {
    return c == kOpLogic ? kOpCount[T][kOpLogic] - kOpCount[T][kOpVote] : kOpCount[T][c];
}
template <int T> constexpr uint32_t mix_len() {
    uint32_t n = 0;
    for (int c = 0; c < kNumOpClasses; ++c) n += mix_count<T>(c);
    return n;
}
// Class at position p of table T's sequence.
template <int T> constexpr int seq_class(uint32_t p) {
    uint32_t done[kNumOpClasses] = {};
    int best = 0;
    for (uint32_t q = 0; q <= p; ++q) {
        best = 0;
        long long best_lag = -(1ll << 62);
        for (int c = 0; c < kNumOpClasses; ++c) {
            if (done[c] >= mix_count<T>(c)) continue;
            const long long lag = (long long)mix_count<T>(c) * (q + 1) - (long long)done[c] * mix_len<T>();
            if (lag > best_lag) { best_lag = lag; best = c; }
        }
        ++done[best];
    }
    return best;
}

// Compile-time constants for device code (evaluated by the host compiler).
template <int T> struct MixLen { static constexpr int value = (int)mix_len<T>(); };
template <int T, int P> struct SeqAt { static constexpr int value = seq_class<T>((uint32_t)P); };

// One scalar's worth of table T: its sequence, position p on chain p mod 8.
template <int T, int... P>
__device__ __forceinline__ void run_mix(Chains &x, uint32_t k, const uint2 *gt, std::integer_sequence<int, P...>) {
    (op<SeqAt<T, P>::value>(x, P & (kChains - 1), k, gt), ...);
}

template <int KIND>
__global__ void __launch_bounds__(256) probe_kernel(uint32_t iters, uint32_t k, uint32_t *sink) {
    __shared__ uint2 stab[kStabPairs];
    __shared__ uint32_t dump[256 * kChains];
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(stab);
    // each entry holds the addresses of two other entries in the same lane
    // column (index mod 32), so a warp's lanes keep reading consecutive entries
    for (uint32_t i = threadIdx.x; i < kStabPairs; i += blockDim.x) {
        const uint32_t a = (i + 32u * 7u) & (kStabPairs - 1u);
        const uint32_t b = (i + 32u * 29u) & (kStabPairs - 1u);
        stab[i] = make_uint2(sbase + 8u * a, sbase + 8u * b);
    }
    __syncthreads();
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    Chains x;
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
        x.u[c] = (k ^ (threadIdx.x * 0x9E3779B9u + c)) | 1u;
        x.f[c] = 1.0f + (float)c * 1e-3f;
        x.s[c] = sbase + 8u * ((lane + 32u * (c * 13u + warp * 5u)) & (kStabPairs - 1u));
        x.g[c] = (lane + 32u * (c * 11u + warp * 3u)) & (kGtabPairs - 1u);
        x.d[c] = (uint32_t)__cvta_generic_to_shared(&dump[threadIdx.x * kChains + c]);
    }
    const uint2 *gt = g_probe_table;
    if constexpr (KIND < kNumOpClasses) {
        for (uint32_t i = 0; i < iters; ++i) {
#pragma unroll
            for (int j = 0; j < kClassSteps; ++j) {
#pragma unroll
                for (int c = 0; c < kChains; ++c) op<KIND < kNumOpClasses ? KIND : 0>(x, c, k + i, gt);
            }
        }
    } else {
        constexpr int T = (KIND >= kNumOpClasses && KIND - kNumOpClasses < kNumOpTables) ? KIND - kNumOpClasses : 0;
        for (uint32_t i = 0; i < iters; ++i)
            run_mix<T>(x, k + i, gt, std::make_integer_sequence<int, MixLen<T>::value>{});
    }
    uint32_t acc = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c) acc ^= x.u[c] ^ __float_as_uint(x.f[c]) ^ x.s[c] ^ x.g[c];
    if (acc == 0x12345678u) sink[0] = acc;            // keeps the chains live
}

__global__ void probe_table_kernel() {
    for (uint32_t i = threadIdx.x; i < kGtabPairs; i += blockDim.x)
        g_probe_table[i] = make_uint2((i + 32u * 5u) & (kGtabPairs - 1u), (i + 32u * 23u) & (kGtabPairs - 1u));
}

template <int KIND>
static void launch_kind(uint32_t iters, uint32_t *sink, uint32_t blocks, cudaStream_t st) {
    probe_kernel<KIND><<<blocks, 256, 0, st>>>(iters, 7u, sink);
}

template <int... K>
static bool launch_any(int kind, uint32_t iters, uint32_t *sink, uint32_t blocks, cudaStream_t st,
                       std::integer_sequence<int, K...>) {
    bool done = false;
    ((kind == K ? (launch_kind<K>(iters, sink, blocks, st), done = true) : false), ...);
    return done;
}

int num_probe_kinds() { return kNumOpClasses + kNumOpTables; }

int launch_peak(int kind, uint32_t iters, uint32_t *sink, uint32_t blocks, cudaStream_t st) {
    if (kind < 0 || kind >= num_probe_kinds()) return 1;
    probe_table_kernel<<<1, 256, 0, st>>>();
    if (!launch_any(kind, iters, sink, blocks, st,
                    std::make_integer_sequence<int, kNumOpClasses + kNumOpTables>{}))
        return 1;
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

// What one launch issues: for a class probe, its instructions times the
// class's 32-bit weight (a vote probe's setp not counted); for a table probe,
// the scalars it models (one per thread and iteration).
uint64_t peak_ops(int kind, uint32_t iters, uint32_t blocks) {
    const uint64_t per = (uint64_t)blocks * 256u * iters;
    if (kind < kNumOpClasses) return per * kClassSteps * kChains * kOpWeight[kind];
    return per;
}

}  // namespace skv

// skv_decode.cu -- decoder kernel: CDF inversion fused with the rANS state
// update and word refill (FORMAT.md sections 5-7).
//
// The decoder of the Speculative KV Coding wiki's pipeline section: from the
// bits and the same (mu, sigma) it restores every code exactly. One warp
// decodes one group of 32 streams; lane l is stream 32 g + l and walks its
// vectors in increasing order. Per scalar: slot = x mod M, find the code o
// with C(o) <= slot < C(o+1) by a search over the monotone code order that
// starts at mu's own code, update x, and refill one 32-bit word when x falls
// below L. Words are consumed in ascending lane order per step (a ballot gives
// each lane its index); they are staged in a per-warp shared-memory ring by
// cp.async so the refill never waits on global memory.
#include <cuda_runtime.h>

#include "skv_model.cuh"

namespace skv {

constexpr int kDecWarps = 8;
constexpr uint32_t kRing = 1024;       // words per warp ring
constexpr uint32_t kBlock = 256;       // words per cp.async batch (2 x 16 B per lane)

// The code o with C(o) <= s < C(o+1), and its (c, f). C(0) = 0 <= s and
// C(N) = M > s hold by construction, so the ends are never evaluated. The
// search gallops away from o0 (mu's own code) and then bisects.
template <uint32_t DT>
__device__ __forceinline__ uint32_t find_symbol(const Tables &t, const Tables8 *t8, const Weights w,
                                                const uint32_t *__restrict__ phat, uint32_t s,
                                                float mu, float rs, uint32_t o0, uint32_t &c_out,
                                                uint32_t &f_out) {
    using K = Codes<DT>;
    constexpr uint32_t M = 1u << K::m;
    uint32_t lo, hi, clo, chi;
    const uint32_t c0 = cdf<DT>(t, t8, w, phat, o0, mu, rs);
    uint32_t step = 1;
    if (s >= c0) {
        lo = o0; clo = c0;
        for (;;) {
            hi = min(lo + step, K::N);
            chi = (hi == K::N) ? M : cdf<DT>(t, t8, w, phat, hi, mu, rs);
            if (chi > s) break;
            lo = hi; clo = chi; step <<= 1;
        }
    } else {
        hi = o0; chi = c0;
        for (;;) {
            lo = hi > step ? hi - step : 0u;
            clo = (lo == 0u) ? 0u : cdf<DT>(t, t8, w, phat, lo, mu, rs);
            if (clo <= s) break;
            hi = lo; chi = clo; step <<= 1;
        }
    }
    while (hi - lo > 1u) {
        const uint32_t mid = (lo + hi) >> 1;
        const uint32_t cm = cdf<DT>(t, t8, w, phat, mid, mu, rs);
        if (cm <= s) { lo = mid; clo = cm; } else { hi = mid; chi = cm; }
    }
    c_out = clo;
    f_out = chi - clo;
    return lo;
}

__device__ __forceinline__ void cp_async16(uint32_t *smem, const uint32_t *gmem) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <uint32_t DT>
__global__ void __launch_bounds__(kDecWarps * 32, 2) decode_kernel(const DecArgs a) {
    using K = Codes<DT>;
    constexpr uint32_t V = K::V, m = K::m;
    constexpr uint32_t M = 1u << m;
    constexpr uint64_t L = K::L;
    __shared__ Tables tab;
    __shared__ Tables8 tab8;
    extern __shared__ __align__(16) uint32_t ring_all[];
    stage_tables<DT>(tab, tab8, a.phat);

    const Geom &g = a.g;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint64_t gid = (uint64_t)blockIdx.x * kDecWarps + warp;
    if (gid >= a.n_units * g.G) return;
    uint32_t *ring = ring_all + warp * kRing;
    const uint64_t unit = gid / g.G;
    const uint32_t grp = (uint32_t)(gid % g.G);
    const uint64_t k = a.ids ? (uint64_t)a.ids[unit] : unit;
    if (k >= g.n_chunks) {
        if (lane == 0) set_status(a.status, SKV_ERR_INVALID_ARG);
        return;
    }
    const ChunkSpan cs = chunk_span(g, k);
    const uint64_t off0 = a.offsets[k], off1 = a.offsets[k + 1];
    if (off0 > off1 || off1 > a.stream_bytes || (off0 & 15u) || off1 - off0 < g.hdr_bytes) {
        if (lane == 0) set_status(a.status, SKV_ERR_CORRUPT);
        return;
    }
    const uint8_t *cp = a.stream + off0;

    // Word counts of all groups; this group's words start after the padded
    // word arrays of the groups before it.
    const uint32_t nw_l = lane < g.G ? reinterpret_cast<const uint32_t *>(cp + 8ull * g.W)[lane] : 0u;
    const uint64_t pw_l = ((uint64_t)nw_l + 3u) & ~uint64_t(3);
    uint64_t incl = pw_l;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= (uint32_t)d) incl += v;
    }
    const uint64_t total_w = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint64_t before_w = __shfl_sync(0xFFFFFFFFu, incl - pw_l, grp);
    const uint32_t nw = __shfl_sync(0xFFFFFFFFu, nw_l, grp);
    if ((uint64_t)g.hdr_bytes + 4ull * total_w != off1 - off0) {
        if (lane == 0) set_status(a.status, SKV_ERR_CORRUPT);
        return;
    }
    const uint32_t *words = reinterpret_cast<const uint32_t *>(cp + g.hdr_bytes) + before_w;
    const uint32_t nwp4 = (nw + 3u) & ~3u;

    const uint32_t s = grp * 32u + lane;
    uint64_t x = reinterpret_cast<const uint64_t *>(cp)[s];
    bool corrupt = (x < L) || (x >= (1ull << (m + 39)));
    if (__any_sync(0xFFFFFFFFu, corrupt)) {
        if (lane == 0) set_status(a.status, SKV_ERR_CORRUPT);
        return;
    }

    const int64_t nq = (int64_t)stream_vectors(g, cs.n_vec, s);
    const int64_t nq0 = (int64_t)stream_vectors(g, cs.n_vec, grp * 32u);
    const uint8_t *mup = a.mu + cs.elem0 * K::bytes;
    const float *rsp = a.rsig + cs.plane * g.HD;
    uint8_t *outp = a.ids ? a.out + unit * a.page_elems * K::bytes : a.out + cs.elem0 * K::bytes;
    const Weights w{g.w_n, g.w_w, g.w_h};
    const uint32_t lt = lanemask_lt();
    bool bad_mu = false;

    uint32_t rp = 0;        // next word to consume (warp-uniform)
    uint32_t filled = 0;    // words requested into the ring so far (warp-uniform)

    uint4 mu_n = make_uint4(0, 0, 0, 0);
    float4 rs_n[V / 4];
    auto fetch = [&](int64_t j) {
        if (j < nq) {
            const uint64_t q = s + (uint64_t)j * g.W;
            mu_n = __ldg(reinterpret_cast<const uint4 *>(mup) + q);
            const uint32_t c0 = (uint32_t)((q * V) % g.HD);
#pragma unroll
            for (int i = 0; i < (int)(V / 4); ++i)
                rs_n[i] = __ldg(reinterpret_cast<const float4 *>(rsp + c0) + i);
        }
    };
    fetch(0);

    for (int64_t j = 0; j < nq0; ++j) {
        // Keep the ring ahead of the reader: one step uses at most 32 V words.
        const uint32_t need = min(nw, rp + 32u * V);
        const uint32_t target = min(nwp4, rp + 32u * V + kBlock);
        bool issued_extra = false;
        while (filled < target) {
            for (uint32_t u = lane; u < kBlock / 4; u += 32) {
                const uint32_t w0 = filled + 4u * u;
                if (w0 < nwp4) cp_async16(ring + (w0 & (kRing - 1)), words + w0);
            }
            cp_async_commit();
            issued_extra = filled >= need;
            filled += kBlock;
        }
        if (issued_extra) cp_async_wait1(); else cp_async_wait0();
        __syncwarp();

        const bool active = j < nq;
        const uint4 muv = mu_n;
        float rsv[V];
#pragma unroll
        for (int i = 0; i < (int)(V / 4); ++i) {
            rsv[4 * i + 0] = rs_n[i].x; rsv[4 * i + 1] = rs_n[i].y;
            rsv[4 * i + 2] = rs_n[i].z; rsv[4 * i + 3] = rs_n[i].w;
        }
        fetch(j + 1);
        uint4 outv = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < (int)V; ++e) {
            if (active) {
                const uint32_t mc = K::get(muv, e);
                const bool fin = K::finite(mc);
                bad_mu |= !fin;
                const float mu = fin ? K::value(mc) : 0.0f;
                const uint32_t slot = (uint32_t)x & (M - 1u);
                uint32_t c, f;
                const uint32_t o = find_symbol<DT>(tab, &tab8, w, a.phat, slot, mu, rsv[e],
                                                   K::ord(mc), c, f);
                x = (uint64_t)f * (x >> m) + slot - c;
                K::put(outv, e, K::code(o));
            }
            const bool refill = active && x < L;
            const uint32_t ball = __ballot_sync(0xFFFFFFFFu, refill);
            if (ball) {
                if (refill) {
                    const uint32_t idx = rp + __popc(ball & lt);
                    uint32_t wd = 0;
                    if (idx < nw) wd = ring[idx & (kRing - 1)];
                    else corrupt = true;
                    x = (x << 32) | wd;
                }
                rp += __popc(ball);
            }
        }
        if (active) reinterpret_cast<uint4 *>(outp)[s + (uint64_t)j * g.W] = outv;
    }
    cp_async_wait0();
    corrupt |= (x != L);
    if (lane == 0 && rp != nw) corrupt = true;
    if (__any_sync(0xFFFFFFFFu, corrupt) && lane == 0) set_status(a.status, SKV_ERR_CORRUPT);
    if (__any_sync(0xFFFFFFFFu, bad_mu) && lane == 0) set_status(a.status, SKV_ERR_NONFINITE_MU);
}

int launch_decode(const DecArgs &a, cudaStream_t st) {
    const uint64_t blocks = (a.n_units * a.g.G + kDecWarps - 1) / kDecWarps;
    if (blocks == 0) return 0;
    const size_t dyn = kDecWarps * kRing * sizeof(uint32_t);
    cudaError_t e;
    if (a.g.dtype == SKV_BF16) {
        e = cudaFuncSetAttribute(decode_kernel<SKV_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess) return 1;
        decode_kernel<SKV_BF16><<<(unsigned)blocks, kDecWarps * 32, dyn, st>>>(a);
    } else {
        e = cudaFuncSetAttribute(decode_kernel<SKV_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
        if (e != cudaSuccess) return 1;
        decode_kernel<SKV_E4M3><<<(unsigned)blocks, kDecWarps * 32, dyn, st>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace skv

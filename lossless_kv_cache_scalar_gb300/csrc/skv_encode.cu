// skv_encode.cu -- encoder kernels: per-scalar model + warp-interleaved rANS,
// chunk-size scan, and compaction into the final bitstream (SKV v1 format §6-7).
//
// The encoder is the "arithmetic coder emits bits" box of the Speculative KV
// Coding wiki's pipeline section, in its rANS form. One warp owns one group of
// 32 streams of one chunk; lane l is stream 32 g + l. A stream is encoded
// backwards (rANS is last-in first-out), so the warp walks its vectors from
// the last to the first and each vector's scalars from the last to the first.
// The words a step emits are ordered with a ballot: the decoder will read them
// at that step in ascending lane order, so the encoder writes them, downwards
// from the top of the group's scratch slot, in the same ascending order.
#include <cuda_runtime.h>

#include "skv_model.cuh"

namespace skv {

// Warps of the one persistent CTA per SM: bf16 runs 32 (64 registers each;
// more warps in flight hide the serial rANS chain better than more registers
// per warp), e4m3, with twice the scalars per vector, 16.
template <uint32_t DT> struct EncShape;
template <> struct EncShape<SKV_BF16> { static constexpr int warps = 32; };
template <> struct EncShape<SKV_E4M3> { static constexpr int warps = 16; };

// Model phase for scalars [e0, e0 + 8) of a vector: (c, f) and 1/f of each.
// No branches and no dependence on the rANS state, so the eight evaluations
// interleave freely.
template <uint32_t DT>
__device__ __forceinline__ void model8(const TablesWide &tab, const void *codes, const Weights w,
                                       const uint2 *__restrict__ ep,
                                       const uint4 &kvv,
                                       const uint4 &muv, const float *rsv, int e0, uint32_t *cc,
                                       uint32_t *ff, float *rf, bool &bad_mu) {
    using K = Codes<DT>;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = e0 + i;
        const uint32_t mc = K::get(muv, e);
        const bool fin = K::finite(mc);
        bad_mu |= !fin;
        const Sliced8 t8(codes);          // e4m3: the lane-sliced code tables
        const float mu = fin ? (DT == SKV_E4M3 ? t8.value(mc) : K::value(mc)) : 0.0f;
        const uint32_t o = K::ord(K::get(kvv, e));
        uint32_t c, f;
        if (DT == SKV_BF16) {
            c = cdf_ep(tab, w, ep, o, mu, rsv[e]);
            f = cdf_ep(tab, w, ep, o + 1u, mu, rsv[e]) - c;
        } else {
            c = cdf_from<DT>(tab, w, t8.edge(o), t8.phat(o), o, mu, rsv[e]);
            f = cdf_from<DT>(tab, w, t8.edge(o + 1u), t8.phat(o + 1u), o + 1u, mu, rsv[e]) - c;
        }
        cc[i] = c;
        ff[i] = f;
        rf[i] = recip(f);
    }
}

// Encode one group of 32 streams (gid = chunk * G + group) with this warp.
template <uint32_t DT>
__device__ __forceinline__ void encode_group(const EncArgs &a, const TablesWide &tab, const void *codes,
                                             uint64_t gid) {
    using K = Codes<DT>;
    constexpr uint32_t V = K::V;
    const Geom &g = a.g;
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t k = gid / g.G;
    const uint32_t grp = (uint32_t)(gid % g.G);
    const ChunkSpan cs = chunk_span(g, k);
    const uint32_t s = grp * 32u + lane;
    const int64_t nq = (int64_t)stream_vectors(g, cs.n_vec, s);
    const int64_t nq0 = (int64_t)stream_vectors(g, cs.n_vec, grp * 32u);
    const uint8_t *kvp = a.kv + cs.elem0 * K::bytes;
    const uint8_t *mup = a.mu + cs.elem0 * K::bytes;
    const float *rsp = a.rsig + sigma_row(g, k) * g.HD;
    uint32_t *slot = a.scratch + gid * g.cap_words;
    const Weights w{g.w_n, g.w_w, g.w_h};
    const uint32_t lt = lanemask_lt();

    uint32_t pos = (uint32_t)g.cap_words;   // words live in [pos, cap_words)
    uint64_t x = K::L;
    bool bad_mu = false, overflow = false;

    // Register double buffer: the next vector is in flight while one is coded.
    uint4 kv_n = make_uint4(0, 0, 0, 0), mu_n = kv_n;
    float4 rs_n[V / 4];
    auto fetch = [&](int64_t j) {
        if (j >= 0 && j < nq) {
            const uint64_t q = s + (uint64_t)j * g.W;
            kv_n = __ldg(reinterpret_cast<const uint4 *>(kvp) + q);
            mu_n = __ldg(reinterpret_cast<const uint4 *>(mup) + q);
            const uint32_t c0 = (uint32_t)((q * V) % g.HD);
#pragma unroll
            for (int i = 0; i < (int)(V / 4); ++i)
                rs_n[i] = __ldg(reinterpret_cast<const float4 *>(rsp + c0) + i);
        }
    };
    fetch(nq0 - 1);

    for (int64_t j = nq0 - 1; j >= 0; --j) {
        const bool active = j < nq;
        const uint4 kvv = kv_n, muv = mu_n;
        float rsv[V];
#pragma unroll
        for (int i = 0; i < (int)(V / 4); ++i) {
            rsv[4 * i + 0] = rs_n[i].x; rsv[4 * i + 1] = rs_n[i].y;
            rsv[4 * i + 2] = rs_n[i].z; rsv[4 * i + 3] = rs_n[i].w;
        }
        fetch(j - 1);
        // Eight scalars at a time, last eight first: model phase, then the
        // rANS phase backwards through them.
#pragma unroll
        for (int h = (int)V / 8 - 1; h >= 0; --h) {
            uint32_t cc[8], ff[8];
            float rf[8];
            model8<DT>(tab, codes, w, a.ep, kvv, muv, rsv, 8 * h, cc, ff, rf, bad_mu);
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                const uint32_t f = active ? ff[i] : 1u;
                const bool emit = active && (x >= ((uint64_t)f << 39));
                const uint32_t ball = __ballot_sync(0xFFFFFFFFu, emit);
                if (ball) {
                    const uint32_t cnt = __popc(ball);
                    // 32-bit word position; cap_words bounds every stream, so running
                    // out of the slot (flagged) is not expected to happen
                    if (cnt <= pos) {                  // warp-uniform
                        if (emit) slot[pos - cnt + __popc(ball & lt)] = (uint32_t)x;
                        pos -= cnt;
                    } else {
                        overflow = true;
                    }
                    if (emit) x >>= 32;
                }
                if (active) x = rans_put<DT>(x, cc[i], f, rf[i]);
            }
        }
    }
    a.states[gid * 32u + lane] = x;
    if (lane == 0) a.nwords[gid] = overflow ? 0u : (uint32_t)(g.cap_words - pos);
    if (__any_sync(0xFFFFFFFFu, bad_mu && nq > 0) && lane == 0) set_status(a.status, SKV_ERR_NONFINITE_MU);
    if (__any_sync(0xFFFFFFFFu, overflow) && lane == 0) set_status(a.status, SKV_ERR_CAPACITY);
}

// One persistent CTA per SM: the tables are staged once (the wide Phi table:
// it saves the narrow component's clamp in every C(o); for e4m3 also the
// lane-sliced code tables, 2% faster than one shared copy); each warp's first
// group is warp * gridDim.x + blockIdx.x (so a small input spreads over all
// SMs instead of filling the first CTAs), and after that each warp takes the
// next group from a global counter until none are left, so warps stay busy
// until the end and no CTA waits on its slowest warp.
template <uint32_t DT>
__global__ void __launch_bounds__(EncShape<DT>::warps * 32, 1) encode_kernel(const EncArgs a) {
    extern __shared__ __align__(16) uint8_t enc_smem[];
    TablesWide &tab = *reinterpret_cast<TablesWide *>(enc_smem);
    uint8_t *codes = enc_smem + sizeof(TablesWide);     // e4m3: Sliced8 tables
    if (DT == SKV_E4M3) stage_sliced8(codes, a.phat);
    stage_phi(tab);
    __syncthreads();
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint64_t first_dynamic = (uint64_t)gridDim.x * EncShape<DT>::warps;
    uint64_t gid = (uint64_t)warp * gridDim.x + blockIdx.x;
    while (gid < a.g.n_groups) {
        encode_group<DT>(a, tab, codes, gid);
        __syncwarp();
        unsigned long long t = 0;
        if (lane == 0) t = atomicAdd(a.next_group, 1ull);
        gid = first_dynamic + __shfl_sync(0xFFFFFFFFu, t, 0);
    }
}

// Per-chunk sizes (SKV v1 format §7) and their exclusive scan into offsets.
__global__ void __launch_bounds__(1024) scan_kernel(const ScanArgs a) {
    const Geom &g = a.g;
    __shared__ uint64_t warp_tot[32];
    __shared__ uint64_t carry;
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (uint64_t base = 0; base < g.n_chunks; base += 1024) {
        const uint64_t k = base + tid;
        uint64_t size = 0;
        if (k < g.n_chunks) {
            size = g.hdr_bytes;
            for (uint32_t j = 0; j < g.G; ++j) size += pad16(4ull * a.nwords[k * g.G + j]);
        }
        uint64_t incl = size;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= (uint32_t)d) incl += v;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            uint64_t t = warp_tot[lane];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint64_t v = __shfl_up_sync(0xFFFFFFFFu, t, d);
                if (lane >= (uint32_t)d) t += v;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const uint64_t before = carry + (warp ? warp_tot[warp - 1] : 0ull) + incl - size;
        if (k < g.n_chunks) a.offsets[k] = before;
        __syncthreads();
        if (tid == 1023) carry = before + size;
        __syncthreads();
    }
    if (tid == 0) {
        a.offsets[g.n_chunks] = carry;
        if (carry > a.out_capacity) set_status(a.status, SKV_ERR_CAPACITY);
    }
}

// Copy each chunk's states, word counts and words to its place in the stream.
// The words of all the chunk's groups form one run of 16-byte units (each
// group's words padded to 4), so the whole CTA copies them at once: a thread
// gathers four words per unit from the group's scratch slot (which starts at
// any word) and writes the unit with one 16-byte store, four units in flight.
constexpr int kCompactThreads = 512;
constexpr int kCompactUnroll = 4;

__global__ void __launch_bounds__(kCompactThreads) compact_kernel(const CompactArgs a) {
    const Geom &g = a.g;
    __shared__ uint32_t s_nw[8];        // words of each group (G <= 8)
    __shared__ uint64_t s_unit[9];      // first unit of each group, then the total
    for (uint64_t k = blockIdx.x; k < g.n_chunks; k += gridDim.x) {
        const uint64_t off = a.offsets[k], end = a.offsets[k + 1];
        if (end > a.out_capacity) continue;            // same for the whole CTA
        uint8_t *dst = a.out + off;
        uint64_t *st = reinterpret_cast<uint64_t *>(dst);
        for (uint32_t i = threadIdx.x; i < g.W; i += blockDim.x) st[i] = a.states[k * g.W + i];
        uint32_t *hw = reinterpret_cast<uint32_t *>(dst + 8ull * g.W);
        const uint32_t hwords = (uint32_t)(pad16(4ull * g.G) / 4);
        for (uint32_t i = threadIdx.x; i < hwords; i += blockDim.x)
            hw[i] = i < g.G ? a.nwords[k * g.G + i] : 0u;
        if (threadIdx.x == 0) {
            uint64_t u = 0;
            for (uint32_t j = 0; j < g.G; ++j) {
                const uint32_t nw = a.nwords[k * g.G + j];
                s_nw[j] = nw;
                s_unit[j] = u;
                u += (nw + 3u) / 4u;
            }
            s_unit[g.G] = u;
        }
        __syncthreads();
        const uint64_t units = s_unit[g.G];
        uint4 *dst4 = reinterpret_cast<uint4 *>(dst + g.hdr_bytes);
        for (uint64_t u0 = threadIdx.x; u0 < units; u0 += (uint64_t)kCompactUnroll * blockDim.x) {
            uint4 v[kCompactUnroll];
#pragma unroll
            for (int r = 0; r < kCompactUnroll; ++r) {
                const uint64_t u = u0 + (uint64_t)r * blockDim.x;
                v[r] = make_uint4(0u, 0u, 0u, 0u);
                if (u < units) {
                    uint32_t j = 0;
                    while (j + 1 < g.G && s_unit[j + 1] <= u) ++j;
                    const uint32_t nw = s_nw[j];
                    const uint32_t i = 4u * (uint32_t)(u - s_unit[j]);
                    const uint32_t *src = a.scratch + (k * g.G + j) * g.cap_words + (g.cap_words - nw);
                    v[r].x = src[i];                           // i < nw: a unit holds at least one word
                    v[r].y = i + 1u < nw ? src[i + 1u] : 0u;
                    v[r].z = i + 2u < nw ? src[i + 2u] : 0u;
                    v[r].w = i + 3u < nw ? src[i + 3u] : 0u;
                }
            }
#pragma unroll
            for (int r = 0; r < kCompactUnroll; ++r) {
                const uint64_t u = u0 + (uint64_t)r * blockDim.x;
                if (u < units) dst4[u] = v[r];
            }
        }
        __syncthreads();                               // s_nw / s_unit are rewritten for the next chunk
    }
}

template <uint32_t DT>
static int launch_encode_t(const EncArgs &a, cudaStream_t st) {
    constexpr int W = EncShape<DT>::warps;
    uint64_t blocks = a.g.n_groups;            // at most one CTA per SM, at least one group each
    if (blocks == 0) return 0;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    if (blocks > (uint64_t)sms) blocks = (uint64_t)sms;
    const int smem = (int)(sizeof(TablesWide) + (DT == SKV_E4M3 ? 4u * Sliced8::kWords : 0u));
    if (cudaFuncSetAttribute(encode_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 1;
    encode_kernel<DT><<<(unsigned)blocks, W * 32, smem, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_encode(const EncArgs &a, cudaStream_t st) {
    return a.g.dtype == SKV_BF16 ? launch_encode_t<SKV_BF16>(a, st) : launch_encode_t<SKV_E4M3>(a, st);
}

int launch_scan(const ScanArgs &a, cudaStream_t st) {
    scan_kernel<<<1, 1024, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_compact(const CompactArgs &a, cudaStream_t st) {
    if (a.g.n_chunks == 0) return 0;
    const uint64_t blocks = a.g.n_chunks < 65535u ? a.g.n_chunks : 65535u;
    compact_kernel<<<(unsigned)blocks, kCompactThreads, 0, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

}  // namespace skv

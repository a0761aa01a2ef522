// skv_api.cu -- the C ABI (include/skv.h): argument checks, workspace layout,
// the per-call set-up kernel (sigma -> 1/sigma, marginal counts -> P_hat
// table) and the launches of the encoder and decoder kernels.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "skv_model.cuh"
#include "skv_ops.h"

namespace skv {

int launch_encode(const EncArgs &a, cudaStream_t st);
int launch_scan(const ScanArgs &a, cudaStream_t st);
int launch_compact(const CompactArgs &a, cudaStream_t st);
int launch_decode(const DecArgs &a, cudaStream_t st);
int launch_histogram(uint32_t dtype, const void *codes, uint64_t n, unsigned long long *counts,
                     cudaStream_t st);
int launch_calibrate(const Geom &g, const void *kv, const void *mu, const uint8_t *mask,
                     uint64_t t_cal, float *sigma, cudaStream_t st);
int launch_requantize(uint32_t mode, uint32_t b, const void *in, uint64_t n, void *out, const float *s_in,
                      float *s_out, uint64_t n_groups, cudaStream_t st);
int launch_peak(int kind, uint32_t iters, uint32_t *sink, uint32_t blocks, cudaStream_t st);
uint64_t peak_ops(int kind, uint32_t iters, uint32_t blocks);
int num_probe_kinds();
int launch_search_eval(const SearchArgs &sa, cudaStream_t st);
int launch_search_aids(const Geom &g, const uint32_t *phat, float *qt, uint16_t *inv_lo,
                       uint16_t *inv_hi, cudaStream_t st);

// ------------------------------------------------------------- set-up kernel

// P_hat(o) = floor(2^24 cum(o) / total) exactly (SKV v1 format §5): a
// binary32 estimate cum * (2^24 / total), within a few units of the result,
// then integer correction with 128-bit products. `scale` = 2^24 / total is
// computed once per thread (binary64 division is slow, and the set-up builds
// all entries on one SM).
__device__ uint32_t phat_entry(uint64_t cum, uint64_t total, float scale) {
    const unsigned __int128 lhs = (unsigned __int128)cum << 24;
    const float est = __fmul_rn(__ull2float_rn(cum), scale);
    uint32_t p = est >= 16777216.0f ? 16777216u : (uint32_t)est;
    while (p < 16777216u && (unsigned __int128)(p + 1u) * total <= lhs) ++p;
    while (p > 0u && (unsigned __int128)p * total > lhs) --p;
    return p;
}

// Orders of P_hat built by one set-up CTA (one per thread).
constexpr uint32_t kSetupThreads = 1024;

// Block-wide sum of one uint64 per thread (blockDim kSetupThreads); `red` is
// 32 words of shared memory. Every thread gets the sum.
__device__ uint64_t block_sum(uint64_t v, uint64_t *red) {
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
    __syncthreads();                                  // red may still be read from a previous use
    if (lane == 0) red[warp] = v;
    __syncthreads();
    uint64_t t = red[lane];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, d);
    return t;
}

// All CTAs validate sigma and write rsig = fl32(1/sigma) (grid-stride). CTA b
// < ceil(N / 1024) also builds P_hat for the code orders [1024 b, 1024 b +
// 1024): it sums the whole histogram (the total) and the part below its range
// (its starting count), both from L2, then scans its 1,024 counts, one per
// thread, coalesced. Spread over CTAs this way the exact entries (128-bit
// products) are not all computed on one SM.
template <uint32_t DT>
__global__ void __launch_bounds__(kSetupThreads) setup_kernel(const SetupArgs a) {
    using K = Codes<DT>;
    const Geom &g = a.g;
    const uint32_t tid = threadIdx.x;
    __shared__ uint64_t red[32];
    __shared__ int bad_sigma;
    if (tid == 0) bad_sigma = 0;
    __syncthreads();

    const uint64_t nsig = g.n_planes * g.n_sblk * g.HD;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + tid; i < nsig; i += (uint64_t)gridDim.x * blockDim.x) {
        const float sg = a.sigma[i];
        const bool ok = isfinite(sg) && sg >= 1.17549435e-38f;   // 2^-126
        a.rsig[i] = ok ? __frcp_rn(sg) : 1.0f;
        if (!ok) bad_sigma = 1;
    }

    const uint32_t o0 = blockIdx.x * kSetupThreads;
    if (o0 < K::N) {
        const uint32_t o = o0 + tid;                  // this thread's order
        const bool mine = o < K::N;
        uint64_t total = 0, base = 0;
        if (g.w_h) {
            uint64_t t = 0, b = 0;
            for (uint32_t q = tid; q < K::N; q += kSetupThreads) {
                const uint64_t c = a.counts[K::code(q)];
                t += c;
                if (q < o0) b += c;
            }
            total = block_sum(t, red);
            base = block_sum(b, red);
        }
        if (total == 0) {                             // no marginal term, or an empty histogram
            if (mine) {
                a.phat[o] = 0u;
                if (DT == SKV_BF16 && a.ep) a.ep[o] = make_uint2(__float_as_uint(K::edge(nullptr, o)), 0u);
            }
            if (blockIdx.x == 0 && tid == 0) {
                a.phat[K::N] = 0u;
                if (DT == SKV_BF16 && a.ep) a.ep[K::N] = make_uint2(__float_as_uint(K::edge(nullptr, K::N)), 0u);
                if (g.w_h) set_status(a.status, SKV_ERR_EMPTY_MARGINAL);
            }
        } else {
            // exclusive scan of this CTA's counts, one per thread
            const uint32_t lane = tid & 31u, warp = tid >> 5;
            const uint64_t c = mine ? a.counts[K::code(o)] : 0ull;
            uint64_t incl = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= (uint32_t)d) incl += v;
            }
            __syncthreads();
            if (lane == 31) red[warp] = incl;
            __syncthreads();
            if (warp == 0) {
                uint64_t t = red[lane];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const uint64_t v = __shfl_up_sync(0xFFFFFFFFu, t, d);
                    if (lane >= (uint32_t)d) t += v;
                }
                red[lane] = t;
            }
            __syncthreads();
            const uint64_t cum = base + (warp ? red[warp - 1] : 0ull) + incl - c;
            if (mine) {
                const float scale = (float)(16777216.0 / (double)total);
                const uint32_t p = phat_entry(cum, total, scale);
                a.phat[o] = p;
                if (DT == SKV_BF16 && a.ep) a.ep[o] = make_uint2(__float_as_uint(K::edge(nullptr, o)), p);
            }
            if (blockIdx.x == 0 && tid == 0) {
                a.phat[K::N] = 1u << 24;
                if (DT == SKV_BF16 && a.ep) a.ep[K::N] = make_uint2(__float_as_uint(K::edge(nullptr, K::N)), 1u << 24);
            }
        }
    }
    __syncthreads();
    if (tid == 0 && bad_sigma) set_status(a.status, SKV_ERR_BAD_SIGMA);
}

// The set-up grid: enough CTAs for P_hat and for the sigmas, at most 1,024.
template <uint32_t DT>
static int launch_setup_t(const SetupArgs &s, cudaStream_t st) {
    const uint64_t nsig = s.g.n_planes * s.g.n_sblk * s.g.HD;
    uint64_t grid = (Codes<DT>::N + kSetupThreads - 1) / kSetupThreads;
    const uint64_t gs = (nsig + 65535u) / 65536u;       // 64 sigmas per thread at most
    if (gs > grid) grid = gs;
    if (grid > 1024u) grid = 1024u;
    setup_kernel<DT><<<(unsigned)grid, kSetupThreads, 0, st>>>(s);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

static int launch_setup(const SetupArgs &s, cudaStream_t st) {
    return s.g.dtype == SKV_BF16 ? launch_setup_t<SKV_BF16>(s, st) : launch_setup_t<SKV_E4M3>(s, st);
}

// C(o) for independent (mu, sigma, o) queries (model-kernel checks).
template <uint32_t DT>
__global__ void __launch_bounds__(256) cdf_eval_kernel(const CdfArgs a) {
    using K = Codes<DT>;
    __shared__ Tables tab;
    __shared__ Tables8 tab8;
    stage_tables<DT>(tab, tab8, a.phat);
    const Weights w{a.g.w_n, a.g.w_w, a.g.w_h};
    bool bad_mu = false, bad_sig = false;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.n;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t mc = a.mu_codes[i] & (K::N - 1u);
        const float sg = a.sigmas[i];
        const bool ok = isfinite(sg) && sg >= 1.17549435e-38f;
        bad_sig |= !ok;
        const float rs = ok ? __frcp_rn(sg) : 1.0f;
        const bool fin = K::finite(mc);
        bad_mu |= !fin;
        const float mu = fin ? K::value(mc) : 0.0f;
        const uint32_t o = min(a.ords[i], K::N);
        a.C[i] = (o == K::N) ? (1u << K::m) : cdf<DT>(tab, &tab8, w, a.phat, o, mu, rs);
    }
    if (bad_sig) set_status(a.status, SKV_ERR_BAD_SIGMA);
    if (bad_mu) set_status(a.status, SKV_ERR_NONFINITE_MU);
}

// --------------------------------------------------------------- host side

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static int32_t make_geom(const skv_layout *lay, Geom &g) {
    if (!lay || lay->version != SKV_FORMAT_VERSION) return SKV_ERR_INVALID_ARG;
    if (lay->dtype != SKV_BF16 && lay->dtype != SKV_E4M3) return SKV_ERR_INVALID_ARG;
    if (!lay->n_layers || !lay->n_kv || !lay->n_heads || !lay->head_dim) return SKV_ERR_INVALID_ARG;
    if (!lay->tokens_per_chunk) return SKV_ERR_INVALID_ARG;
    if (lay->sigma_block_tokens % lay->tokens_per_chunk != 0) return SKV_ERR_INVALID_ARG;
    const uint32_t W = lay->streams_per_chunk;
    if (W == 0 || W % 32 != 0 || W > 256) return SKV_ERR_INVALID_ARG;
    if (lay->w_narrow + lay->w_wide + lay->w_marginal != 100u) return SKV_ERR_INVALID_ARG;
    const DtypeInfo d = dtype_info(lay->dtype);
    const uint64_t HD = (uint64_t)lay->n_heads * lay->head_dim;
    if ((HD * d.bytes) % 16 != 0 || HD > (1ull << 24)) return SKV_ERR_INVALID_ARG;
    if (lay->n_tokens > (1ull << 40)) return SKV_ERR_INVALID_ARG;
    {
        // every size below is a product of these: bound them so none overflows
        const unsigned __int128 planes = (unsigned __int128)lay->n_layers * lay->n_kv;
        const uint64_t nsb = lay->sigma_block_tokens
                                 ? (lay->n_tokens + lay->sigma_block_tokens - 1) / lay->sigma_block_tokens
                                 : 1u;
        if (planes * lay->n_tokens * HD > ((unsigned __int128)1 << 48)) return SKV_ERR_INVALID_ARG;
        if (planes * nsb * HD > ((unsigned __int128)1 << 40)) return SKV_ERR_INVALID_ARG;
    }
    std::memset(&g, 0, sizeof g);
    g.dtype = lay->dtype;
    g.n_kv = lay->n_kv;
    g.HD = (uint32_t)HD;
    g.W = W;
    g.G = W / 32;
    g.Tc = lay->tokens_per_chunk;
    g.T = lay->n_tokens;
    g.P = (lay->n_tokens + lay->tokens_per_chunk - 1) / lay->tokens_per_chunk;
    g.n_planes = (uint64_t)lay->n_layers * lay->n_kv;
    g.n_chunks = g.n_planes * g.P;
    g.SB = lay->sigma_block_tokens;
    g.n_sblk = g.SB ? (g.T + g.SB - 1) / g.SB : 1;
    g.n_groups = g.n_chunks * g.G;
    g.w_n = lay->w_narrow;
    g.w_w = lay->w_wide;
    g.w_h = lay->w_marginal;
    g.hdr_bytes = (uint32_t)(8ull * W + pad16(4ull * g.G));
    // scratch words per group: the longest stream of a full chunk bounds all
    const uint64_t ntok_full = g.T < g.Tc ? g.T : g.Tc;
    const uint64_t nvec_full = ntok_full * HD / d.V;
    const uint64_t nmax = stream_vectors(g, nvec_full, 0) * d.V;
    g.cap_words = 32ull * ((nmax * (d.m + 1) + 31) / 32);
    if (g.cap_words > 0xFFFFFFF0ull) return SKV_ERR_INVALID_ARG;
    return SKV_OK;
}

// Worst-case bytes of one chunk with n_vec vectors (SKV v1 format §8).
static uint64_t chunk_max_bytes(const Geom &g, uint64_t n_vec) {
    const DtypeInfo d = dtype_info(g.dtype);
    uint64_t b = g.hdr_bytes;
    for (uint32_t j = 0; j < g.G; ++j) {
        const uint64_t nmax = stream_vectors(g, n_vec, 32 * j) * d.V;
        b += pad16(4ull * 32ull * ((nmax * (d.m + 1) + 31) / 32));
    }
    return b;
}

struct Workspace {
    uint2 *ep;
    uint32_t *phat;
    float *rsig;
    float *qt;
    uint16_t *inv_lo, *inv_hi;
    uint64_t *states;
    unsigned long long *ctr;
    uint32_t *nwords;
    uint32_t *scratch;
    uint64_t bytes;
};

static uint64_t round256(uint64_t b) { return (b + 255u) & ~uint64_t(255); }

// Workspace kinds: the encoder's, the decoder's minimum, and the decoder's
// with the outlier inverse tables (faster on data with far outliers).
enum WsKind { WS_ENCODE = 1, WS_DECODE_MIN = 0, WS_DECODE_FULL = 2 };

static Workspace carve(const Geom &g, int kind, uint8_t *base) {
    // offsets are computed as integers and only then turned into pointers
    const DtypeInfo d = dtype_info(g.dtype);
    uint64_t off = 0, o_phat, o_rsig, o_qt = 0, o_lo = 0, o_hi = 0, o_states = 0, o_nwords = 0,
             o_scratch = 0;
    o_phat = off;
    off += round256(4ull * (d.N + 1));
    o_rsig = off;
    off += round256(4ull * g.n_planes * g.n_sblk * g.HD);
    uint64_t o_ep = 0;
    if ((kind == WS_ENCODE || kind == WS_DECODE_FULL) && g.dtype == SKV_BF16) {
        o_ep = off;
        off += round256(8ull * (d.N + 1));
    }
    uint64_t o_ctr = 0;
    if (kind == WS_ENCODE) {
        o_ctr = off;
        off += 256;
        o_states = off;
        off += round256(8ull * 32ull * g.n_groups);
        o_nwords = off;
        off += round256(4ull * g.n_groups);
        o_scratch = off;
        off += round256(4ull * g.cap_words * g.n_groups);
    } else {
        o_qt = off;
        off += round256(4ull * kQuantFloats);
        if (kind == WS_DECODE_FULL) {
            o_lo = off;
            off += round256(2ull << d.m);
            o_hi = off;
            off += round256(2ull << d.m);
        }
    }
    Workspace w{};
    w.bytes = off;
    if (base) {
        w.phat = reinterpret_cast<uint32_t *>(base + o_phat);
        w.rsig = reinterpret_cast<float *>(base + o_rsig);
        if (kind == WS_ENCODE) {
            if (g.dtype == SKV_BF16) w.ep = reinterpret_cast<uint2 *>(base + o_ep);
            w.states = reinterpret_cast<uint64_t *>(base + o_states);
            w.ctr = reinterpret_cast<unsigned long long *>(base + o_ctr);
            w.nwords = reinterpret_cast<uint32_t *>(base + o_nwords);
            w.scratch = reinterpret_cast<uint32_t *>(base + o_scratch);
        } else {
            w.qt = reinterpret_cast<float *>(base + o_qt);
            if (kind == WS_DECODE_FULL && g.dtype == SKV_BF16) w.ep = reinterpret_cast<uint2 *>(base + o_ep);
            if (kind == WS_DECODE_FULL) {
                w.inv_lo = reinterpret_cast<uint16_t *>(base + o_lo);
                w.inv_hi = reinterpret_cast<uint16_t *>(base + o_hi);
            }
        }
    }
    return w;
}

static int32_t run_setup(const Geom &g, const float *sigma, const uint64_t *counts,
                         const Workspace &ws, int32_t *status, cudaStream_t st) {
    SetupArgs s{g, sigma, counts, ws.phat, ws.rsig, ws.ep, status};
    return launch_setup(s, st) ? SKV_ERR_CUDA : SKV_OK;
}

static int32_t common_checks(const Geom &g, const float *sigma, const uint64_t *counts,
                             int32_t *status, void *workspace, uint64_t ws_bytes, int kind) {
    if (!sigma || !status || !workspace) return SKV_ERR_INVALID_ARG;
    if (g.w_h && !counts) return SKV_ERR_INVALID_ARG;
    if (((uintptr_t)workspace & 255u) != 0) return SKV_ERR_INVALID_ARG;
    if (ws_bytes < carve(g, kind, nullptr).bytes) return SKV_ERR_INVALID_ARG;
    return SKV_OK;
}

// ------------------------------------------------ host-buffer pipelines

// A sub-layout of layers [l0, l0 + nl) of lay: its chunks are chunks
// [2 l0 P, 2 (l0 + nl) P) of the whole cache (planes are layer-major), and its
// bitstream is the same bytes as theirs (chunks code independently).
static skv_layout sub_layout(const skv_layout *lay, uint32_t nl) {
    skv_layout s = *lay;
    s.n_layers = nl;
    return s;
}

// Device staging of the host pipelines for batches of `lpb` layers: the
// decoder's or encoder's tables for the whole layout, then two halves.
struct HostStaging {
    uint32_t *phat;
    float *rsig;
    uint2 *ep;             // bf16 (edge, P_hat) pairs (encode; decode with inverse tables)
    float *qt;             // decode
    uint16_t *inv_lo, *inv_hi;
    uint64_t *states;      // encode: one batch
    unsigned long long *ctr;
    uint32_t *nwords;
    uint32_t *scratch;
    uint8_t *kv[2], *mu[2], *bits[2];
    uint64_t *offs[2];
    uint64_t out_cap;      // bytes of bits[h]
    uint64_t bytes;
};

static HostStaging carve_host(const Geom &g, const Geom &gb, bool encode, bool inv, uint8_t *base) {
    const DtypeInfo d = dtype_info(g.dtype);
    uint64_t off = 0;
    auto take = [&](uint64_t n) { const uint64_t o = off; off += round256(n); return o; };
    const uint64_t o_phat = take(4ull * (d.N + 1));
    const uint64_t o_rsig = take(4ull * g.n_planes * g.n_sblk * g.HD);
    const bool ep = g.dtype == SKV_BF16 && (encode || inv);
    const uint64_t o_ep = ep ? take(8ull * (d.N + 1)) : 0;
    uint64_t o_qt = 0, o_lo = 0, o_hi = 0, o_states = 0, o_ctr = 0, o_nw = 0, o_scr = 0;
    if (encode) {
        o_states = take(8ull * 32ull * gb.n_groups);
        o_ctr = take(8);
        o_nw = take(4ull * gb.n_groups);
        o_scr = take(4ull * gb.cap_words * gb.n_groups);
    } else {
        o_qt = take(4ull * kQuantFloats);
        if (inv) { o_lo = take(2ull << d.m); o_hi = take(2ull << d.m); }
    }
    const uint64_t raw = gb.n_planes * gb.T * gb.HD * d.bytes;
    uint64_t cap = 0;
    {
        const uint64_t full = chunk_max_bytes(gb, (uint64_t)gb.Tc * gb.HD / d.V);
        const uint64_t last = chunk_max_bytes(gb, (gb.T - (gb.P - 1) * gb.Tc) * gb.HD / d.V);
        cap = gb.n_chunks ? gb.n_planes * ((gb.P - 1) * full + last) : 0;
    }
    uint64_t o_kv[2], o_mu[2], o_bits[2], o_offs[2];
    for (int h = 0; h < 2; ++h) {
        o_kv[h] = take(raw);
        o_mu[h] = take(raw);
        o_bits[h] = take(cap);
        o_offs[h] = take(8ull * (gb.n_chunks + 1));
    }
    HostStaging st{};
    st.bytes = off;
    st.out_cap = cap;
    if (base) {
        st.phat = reinterpret_cast<uint32_t *>(base + o_phat);
        st.rsig = reinterpret_cast<float *>(base + o_rsig);
        if (ep) st.ep = reinterpret_cast<uint2 *>(base + o_ep);
        if (encode) {
            st.states = reinterpret_cast<uint64_t *>(base + o_states);
            st.ctr = reinterpret_cast<unsigned long long *>(base + o_ctr);
            st.nwords = reinterpret_cast<uint32_t *>(base + o_nw);
            st.scratch = reinterpret_cast<uint32_t *>(base + o_scr);
        } else {
            st.qt = reinterpret_cast<float *>(base + o_qt);
            if (inv) {
                st.inv_lo = reinterpret_cast<uint16_t *>(base + o_lo);
                st.inv_hi = reinterpret_cast<uint16_t *>(base + o_hi);
            }
        }
        for (int h = 0; h < 2; ++h) {
            st.kv[h] = base + o_kv[h];
            st.mu[h] = base + o_mu[h];
            st.bits[h] = base + o_bits[h];
            st.offs[h] = reinterpret_cast<uint64_t *>(base + o_offs[h]);
        }
    }
    return st;
}

// Geometry of the batch layout (lpb layers), checked.
static int32_t batch_geom(const skv_layout *lay, uint32_t lpb, Geom &g, Geom &gb) {
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    if (lpb == 0) return SKV_ERR_INVALID_ARG;
    if (lpb > lay->n_layers) lpb = lay->n_layers;
    const skv_layout sb = sub_layout(lay, lpb);
    return make_geom(&sb, gb);
}

struct EventPair {
    cudaEvent_t e[2] = {nullptr, nullptr};
    bool make() {
        for (int h = 0; h < 2; ++h)
            if (cudaEventCreateWithFlags(&e[h], cudaEventDisableTiming) != cudaSuccess) return false;
        return true;
    }
    ~EventPair() {
        for (int h = 0; h < 2; ++h)
            if (e[h]) cudaEventDestroy(e[h]);
    }
};

}  // namespace skv

using namespace skv;

extern "C" {

uint32_t skv_version(void) { return SKV_FORMAT_VERSION; }

const char *skv_status_string(int32_t s) {
    switch (s) {
        case SKV_OK: return "OK";
        case SKV_ERR_INVALID_ARG: return "INVALID_ARG";
        case SKV_ERR_CUDA: return "CUDA";
        case SKV_ERR_NONFINITE_MU: return "NONFINITE_MU";
        case SKV_ERR_BAD_SIGMA: return "BAD_SIGMA";
        case SKV_ERR_EMPTY_MARGINAL: return "EMPTY_MARGINAL";
        case SKV_ERR_CAPACITY: return "CAPACITY";
        case SKV_ERR_CORRUPT: return "CORRUPT";
        case SKV_ERR_TIMEOUT: return "TIMEOUT";
        default: return "UNKNOWN";
    }
}

int32_t skv_layout_init(skv_layout *lay, uint32_t dtype, uint32_t n_layers, uint32_t n_kv,
                        uint32_t n_heads, uint32_t head_dim, uint64_t n_tokens) {
    if (!lay) return SKV_ERR_INVALID_ARG;
    std::memset(lay, 0, sizeof *lay);
    lay->version = SKV_FORMAT_VERSION;
    lay->dtype = dtype;
    lay->n_layers = n_layers;
    lay->n_kv = n_kv;
    lay->n_heads = n_heads;
    lay->head_dim = head_dim;
    lay->n_tokens = n_tokens;
    lay->tokens_per_chunk = 256;
    lay->streams_per_chunk = 64;
    lay->w_narrow = 95;
    lay->w_wide = 3;
    lay->w_marginal = 2;
    return skv_layout_check(lay);
}

int32_t skv_layout_check(const skv_layout *lay) {
    Geom g;
    return make_geom(lay, g);
}

int32_t skv_num_chunks(const skv_layout *lay, uint64_t *n_chunks) {
    Geom g;
    const int32_t r = make_geom(lay, g);
    if (r != SKV_OK || !n_chunks) return SKV_ERR_INVALID_ARG;
    *n_chunks = g.n_chunks;
    return SKV_OK;
}

int32_t skv_max_encoded_bytes(const skv_layout *lay, uint64_t *bytes) {
    Geom g;
    if (make_geom(lay, g) != SKV_OK || !bytes) return SKV_ERR_INVALID_ARG;
    if (g.n_chunks == 0) { *bytes = 0; return SKV_OK; }
    const DtypeInfo d = dtype_info(g.dtype);
    const uint64_t full = chunk_max_bytes(g, (uint64_t)g.Tc * g.HD / d.V);
    const uint64_t last_tok = g.T - (g.P - 1) * g.Tc;
    const uint64_t last = chunk_max_bytes(g, last_tok * g.HD / d.V);
    *bytes = g.n_planes * ((g.P - 1) * full + last);
    return SKV_OK;
}

int32_t skv_workspace_bytes(const skv_layout *lay, int32_t op, uint64_t *bytes) {
    Geom g;
    if (make_geom(lay, g) != SKV_OK || !bytes) return SKV_ERR_INVALID_ARG;
    if (op != WS_ENCODE && op != WS_DECODE_MIN && op != WS_DECODE_FULL) return SKV_ERR_INVALID_ARG;
    *bytes = carve(g, op, nullptr).bytes;
    return SKV_OK;
}

int32_t skv_encode(const skv_layout *lay, const void *kv, const void *mu, const float *sigma,
                   const uint64_t *counts, void *out, uint64_t out_capacity, uint64_t *offsets,
                   int32_t *status, void *workspace, uint64_t ws_bytes, void *stream) {
    Geom g;
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    r = common_checks(g, sigma, counts, status, workspace, ws_bytes, WS_ENCODE);
    if (r != SKV_OK) return r;
    if (!offsets || (g.n_chunks && (!kv || !mu || !out))) return SKV_ERR_INVALID_ARG;
    if (g.n_chunks && (!aligned16(kv) || !aligned16(mu) || !aligned16(out))) return SKV_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return SKV_ERR_CUDA;
    const Workspace ws = carve(g, WS_ENCODE, static_cast<uint8_t *>(workspace));
    if ((r = run_setup(g, sigma, counts, ws, status, st)) != SKV_OK) return r;
    EncArgs ea{g, static_cast<const uint8_t *>(kv), static_cast<const uint8_t *>(mu), ws.phat,
               ws.ep, ws.rsig, ws.states, ws.nwords, ws.scratch, status, ws.ctr};
    if (cudaMemsetAsync(ws.ctr, 0, sizeof(unsigned long long), st) != cudaSuccess) return SKV_ERR_CUDA;
    if (launch_encode(ea, st)) return SKV_ERR_CUDA;
    ScanArgs sa{g, ws.nwords, offsets, out_capacity, status};
    if (launch_scan(sa, st)) return SKV_ERR_CUDA;
    CompactArgs ca{g, ws.states, ws.nwords, ws.scratch, offsets, static_cast<uint8_t *>(out),
                   out_capacity};
    if (launch_compact(ca, st)) return SKV_ERR_CUDA;
    return SKV_OK;
}

// Decoder tables (P_hat, 1/sigma, quantiles, and with a full workspace the
// outlier inverse tables) built on the stream into the workspace.
static int32_t decode_tables(const Geom &g, const float *sigma, const uint64_t *counts,
                             int32_t *status, void *workspace, uint64_t ws_bytes, cudaStream_t st,
                             Workspace &ws) {
    const int kind = ws_bytes >= carve(g, WS_DECODE_FULL, nullptr).bytes ? WS_DECODE_FULL : WS_DECODE_MIN;
    ws = carve(g, kind, static_cast<uint8_t *>(workspace));
    const int32_t r = run_setup(g, sigma, counts, ws, status, st);
    if (r != SKV_OK) return r;
    if (launch_search_aids(g, ws.phat, ws.qt, ws.inv_lo, ws.inv_hi, st)) return SKV_ERR_CUDA;
    return SKV_OK;
}

static int32_t decode_launch(const Geom &g, const void *bitstream, uint64_t bitstream_bytes,
                             const uint64_t *offsets, const void *mu, const uint32_t *ids,
                             uint64_t n_units, bool pages, void *out, int32_t *status,
                             const Workspace &ws, cudaStream_t st) {
    if (n_units == 0) return SKV_OK;
    DecArgs da{g, static_cast<const uint8_t *>(bitstream), bitstream_bytes, offsets,
               static_cast<const uint8_t *>(mu), ws.phat, ws.rsig, ws.qt, ws.inv_lo, ws.inv_hi,
               pages ? ids : nullptr,
               n_units, static_cast<uint8_t *>(out), (uint64_t)g.Tc * g.HD, status, 0, 0, ws.ep, nullptr};
    return launch_decode(da, st) ? SKV_ERR_CUDA : SKV_OK;
}

static int32_t decode_args_check(const void *bitstream, const uint64_t *offsets,
                                 const void *mu, const uint32_t *ids, uint64_t n_units, bool pages,
                                 void *out) {
    if (n_units && (!bitstream || !offsets || !mu || !out)) return SKV_ERR_INVALID_ARG;
    if (pages && n_units && !ids) return SKV_ERR_INVALID_ARG;
    if (n_units && (!aligned16(bitstream) || !aligned16(mu) || !aligned16(out))) return SKV_ERR_INVALID_ARG;
    return SKV_OK;
}

static int32_t decode_impl(const skv_layout *lay, const void *bitstream, uint64_t bitstream_bytes,
                           const uint64_t *offsets, const void *mu, const float *sigma,
                           const uint64_t *counts, const uint32_t *ids, uint64_t n_units,
                           bool pages, void *out, int32_t *status, void *workspace,
                           uint64_t ws_bytes, void *stream) {
    Geom g;
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    r = common_checks(g, sigma, counts, status, workspace, ws_bytes, WS_DECODE_MIN);
    if (r != SKV_OK) return r;
    if (!pages) n_units = g.n_chunks;
    if ((r = decode_args_check(bitstream, offsets, mu, ids, n_units, pages, out)) != SKV_OK) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return SKV_ERR_CUDA;
    Workspace ws;
    if ((r = decode_tables(g, sigma, counts, status, workspace, ws_bytes, st, ws)) != SKV_OK) return r;
    return decode_launch(g, bitstream, bitstream_bytes, offsets, mu, ids, n_units, pages, out, status,
                         ws, st);
}

int32_t skv_decode(const skv_layout *lay, const void *bitstream, uint64_t bitstream_bytes,
                   const uint64_t *offsets, const void *mu, const float *sigma,
                   const uint64_t *counts, void *kv_out, int32_t *status, void *workspace,
                   uint64_t ws_bytes, void *stream) {
    return decode_impl(lay, bitstream, bitstream_bytes, offsets, mu, sigma, counts, nullptr, 0,
                       false, kv_out, status, workspace, ws_bytes, stream);
}

int32_t skv_decode_chunks(const skv_layout *lay, const void *bitstream, uint64_t bitstream_bytes,
                          const uint64_t *offsets, const void *mu, const float *sigma,
                          const uint64_t *counts, const uint32_t *chunk_ids, uint32_t n_ids,
                          void *pages_out, int32_t *status, void *workspace, uint64_t ws_bytes,
                          void *stream) {
    return decode_impl(lay, bitstream, bitstream_bytes, offsets, mu, sigma, counts, chunk_ids,
                       n_ids, true, pages_out, status, workspace, ws_bytes, stream);
}

int32_t skv_decode_prepare(const skv_layout *lay, const float *sigma, const uint64_t *counts,
                           int32_t *status, void *workspace, uint64_t ws_bytes, void *stream) {
    Geom g;
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    if ((r = common_checks(g, sigma, counts, status, workspace, ws_bytes, WS_DECODE_MIN)) != SKV_OK)
        return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return SKV_ERR_CUDA;
    Workspace ws;
    return decode_tables(g, sigma, counts, status, workspace, ws_bytes, st, ws);
}

int32_t skv_decode_chunks_prepared(const skv_layout *lay, const void *bitstream,
                                   uint64_t bitstream_bytes, const uint64_t *offsets, const void *mu,
                                   const uint32_t *chunk_ids, uint32_t n_ids, void *pages_out,
                                   int32_t *status, const void *workspace, uint64_t ws_bytes,
                                   void *stream) {
    Geom g;
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    if (!status || !workspace || ((uintptr_t)workspace & 255u) != 0) return SKV_ERR_INVALID_ARG;
    if (ws_bytes < carve(g, WS_DECODE_MIN, nullptr).bytes) return SKV_ERR_INVALID_ARG;
    if ((r = decode_args_check(bitstream, offsets, mu, chunk_ids, n_ids, true, pages_out)) != SKV_OK)
        return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return SKV_ERR_CUDA;
    const int kind = ws_bytes >= carve(g, WS_DECODE_FULL, nullptr).bytes ? WS_DECODE_FULL : WS_DECODE_MIN;
    const Workspace ws = carve(g, kind, static_cast<uint8_t *>(const_cast<void *>(workspace)));
    return decode_launch(g, bitstream, bitstream_bytes, offsets, mu, chunk_ids, n_ids, true, pages_out,
                         status, ws, st);
}

int32_t skv_cdf_eval(const skv_layout *lay, const uint64_t *counts, uint64_t n,
                     const uint32_t *mu_codes, const float *sigmas, const uint32_t *ords,
                     uint32_t *C_out, int32_t *status, void *workspace, uint64_t ws_bytes,
                     void *stream) {
    Geom g;
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    if (!status || !workspace || (g.w_h && !counts)) return SKV_ERR_INVALID_ARG;
    if (n && (!mu_codes || !sigmas || !ords || !C_out)) return SKV_ERR_INVALID_ARG;
    if (((uintptr_t)workspace & 255u) != 0 || ws_bytes < carve(g, WS_DECODE_MIN, nullptr).bytes)
        return SKV_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return SKV_ERR_CUDA;
    const Workspace ws = carve(g, WS_DECODE_MIN, static_cast<uint8_t *>(workspace));
    // P_hat only; sigma is per query here, so rsig is not built
    Geom g1 = g;
    g1.n_planes = 0;
    SetupArgs s{g1, nullptr, counts, ws.phat, ws.rsig, nullptr, status};
    if (launch_setup(s, st)) return SKV_ERR_CUDA;
    if (n == 0) return SKV_OK;
    CdfArgs ca{g, ws.phat, n, mu_codes, sigmas, ords, C_out, status};
    const uint64_t blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    if (g.dtype == SKV_BF16) cdf_eval_kernel<SKV_BF16><<<(unsigned)blocks, 256, 0, st>>>(ca);
    else cdf_eval_kernel<SKV_E4M3><<<(unsigned)blocks, 256, 0, st>>>(ca);
    return cudaGetLastError() == cudaSuccess ? SKV_OK : SKV_ERR_CUDA;
}

int32_t skv_histogram(uint32_t dtype, const void *codes, uint64_t n, uint64_t *counts,
                      int32_t accumulate, void *stream) {
    if (dtype != SKV_BF16 && dtype != SKV_E4M3) return SKV_ERR_INVALID_ARG;
    const DtypeInfo d = dtype_info(dtype);
    if (!counts || ((uintptr_t)counts & 7u) != 0) return SKV_ERR_INVALID_ARG;
    if (n && (!codes || ((uintptr_t)codes % d.bytes) != 0)) return SKV_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!accumulate && cudaMemsetAsync(counts, 0, sizeof(uint64_t) * d.N, st) != cudaSuccess)
        return SKV_ERR_CUDA;
    return launch_histogram(dtype, codes, n, reinterpret_cast<unsigned long long *>(counts), st)
               ? SKV_ERR_CUDA : SKV_OK;
}

int32_t skv_calibrate_sigma(const skv_layout *lay, const void *kv, const void *mu, const uint8_t *mask,
                            uint64_t t_cal, float *sigma, void *stream) {
    Geom g;
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    if (t_cal == 0 || t_cal > g.T || (g.SB && t_cal > g.SB) || !kv || !mu || !sigma)
        return SKV_ERR_INVALID_ARG;
    const uint32_t b = dtype_info(g.dtype).bytes;
    if (((uintptr_t)kv % b) != 0 || ((uintptr_t)mu % b) != 0 || ((uintptr_t)sigma & 3u) != 0)
        return SKV_ERR_INVALID_ARG;
    return launch_calibrate(g, kv, mu, mask, t_cal, sigma, static_cast<cudaStream_t>(stream))
               ? SKV_ERR_CUDA : SKV_OK;
}

int32_t skv_offload_plan(const uint64_t *host_offsets, uint64_t n_chunks, uint64_t batch_bytes,
                         uint64_t max_chunks, uint64_t *batch_first, uint64_t max_batches,
                         uint64_t *n_batches) {
    if (!host_offsets || !n_batches || (max_batches && !batch_first)) return SKV_ERR_INVALID_ARG;
    uint64_t nb = 0, first = 0;
    while (first < n_chunks) {
        // the longest run of whole chunks from `first` whose bytes fit one batch
        uint64_t last = first;
        while (last < n_chunks) {
            const uint64_t a = host_offsets[last], b = host_offsets[last + 1];
            if (b < a) return SKV_ERR_CORRUPT;
            if (b - host_offsets[first] > batch_bytes) break;
            if (max_chunks && last - first == max_chunks) break;
            ++last;
        }
        if (last == first) return SKV_ERR_INVALID_ARG;   // one chunk is larger than a batch
        if (nb < max_batches) batch_first[nb] = first;
        ++nb;
        first = last;
    }
    if (nb < max_batches) batch_first[nb] = n_chunks;
    *n_batches = nb;
    // with a plan requested, it needs nb + 1 entries (the last is n_chunks)
    if (max_batches != 0 && max_batches < nb + 1) return SKV_ERR_INVALID_ARG;
    return SKV_OK;
}

int32_t skv_decode_offload(const skv_layout *lay, const void *host_bitstream, uint64_t bitstream_bytes,
                           const uint64_t *host_offsets, const uint64_t *offsets, const void *mu,
                           const float *sigma, const uint64_t *counts, void *kv_out, int32_t *status,
                           void *workspace, uint64_t ws_bytes, void *staging, uint64_t staging_bytes,
                           void *stream, void *copy_stream) {
    Geom g;
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    if ((r = common_checks(g, sigma, counts, status, workspace, ws_bytes, WS_DECODE_MIN)) != SKV_OK) return r;
    if (g.n_chunks && (!host_bitstream || !host_offsets || !staging || !aligned16(staging)))
        return SKV_ERR_INVALID_ARG;
    if ((r = decode_args_check(staging, offsets, mu, nullptr, g.n_chunks, false, kv_out)) != SKV_OK)
        return r;
    if (g.n_chunks && (host_offsets[0] != 0 || host_offsets[g.n_chunks] > bitstream_bytes))
        return SKV_ERR_CORRUPT;
    // plan on the host: two staging halves, each batch a run of whole chunks.
    // A batch is also cut at a whole number of decoder waves (the chunks whose
    // warps are resident at once), so that no batch ends on a mostly empty wave.
    const uint64_t half = (staging_bytes / 2) & ~uint64_t(15);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SKV_ERR_CUDA;
    const uint64_t wave = std::max<uint64_t>(1, (uint64_t)sms * kDecResidentWarps / g.G);
    const uint64_t mean = g.n_chunks ? std::max<uint64_t>(1, host_offsets[g.n_chunks] / g.n_chunks) : 1;
    const uint64_t per_batch = std::max<uint64_t>(1, half / mean / wave) * wave;
    uint64_t nb = 0;
    if ((r = skv_offload_plan(host_offsets, g.n_chunks, half, per_batch, nullptr, 0, &nb)) != SKV_OK)
        return r;
    uint64_t *first = static_cast<uint64_t *>(std::malloc(sizeof(uint64_t) * (nb + 1)));
    if (!first) return SKV_ERR_INVALID_ARG;
    if ((r = skv_offload_plan(host_offsets, g.n_chunks, half, per_batch, first, nb + 1, &nb)) != SKV_OK) {
        std::free(first);
        return r;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
    cudaEvent_t copied[2] = {nullptr, nullptr}, freed[2] = {nullptr, nullptr};
    bool ok = true;
    for (int h = 0; h < 2 && ok; ++h)
        ok = cudaEventCreateWithFlags(&copied[h], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&freed[h], cudaEventDisableTiming) == cudaSuccess;
    Workspace ws;
    if (ok) ok = cudaMemsetAsync(status, 0, sizeof(int32_t), st) == cudaSuccess;
    if (ok) ok = decode_tables(g, sigma, counts, status, workspace, ws_bytes, st, ws) == SKV_OK;
    // batch b: copy into half b % 2 once the decode of batch b - 2 is done with it,
    // then decode it on the compute stream once the copy has landed
    for (uint64_t b = 0; b < nb && ok; ++b) {
        const int h = (int)(b & 1u);
        uint8_t *dst = static_cast<uint8_t *>(staging) + h * half;
        const uint64_t k0 = first[b], k1 = first[b + 1];
        const uint64_t o0 = host_offsets[k0], bytes = host_offsets[k1] - o0;
        if (b >= 2) ok = cudaStreamWaitEvent(cs, freed[h], 0) == cudaSuccess;
        if (ok) ok = cudaMemcpyAsync(dst, static_cast<const uint8_t *>(host_bitstream) + o0, bytes,
                                     cudaMemcpyHostToDevice, cs) == cudaSuccess;
        if (ok) ok = cudaEventRecord(copied[h], cs) == cudaSuccess;
        if (ok) ok = cudaStreamWaitEvent(st, copied[h], 0) == cudaSuccess;
        if (ok) {
            DecArgs da{g, dst, bytes, offsets, static_cast<const uint8_t *>(mu), ws.phat, ws.rsig, ws.qt,
                       ws.inv_lo, ws.inv_hi, nullptr, k1 - k0, static_cast<uint8_t *>(kv_out),
                       (uint64_t)g.Tc * g.HD, status, o0, k0, ws.ep, nullptr};
            ok = launch_decode(da, st) == 0;
        }
        if (ok) ok = cudaEventRecord(freed[h], st) == cudaSuccess;
    }
    for (int h = 0; h < 2; ++h) {
        if (copied[h]) cudaEventDestroy(copied[h]);
        if (freed[h]) cudaEventDestroy(freed[h]);
    }
    std::free(first);
    return ok ? SKV_OK : SKV_ERR_CUDA;
}

int32_t skv_requantize(uint32_t mode, uint32_t b, const void *in, uint64_t n, void *out,
                       const float *scale_in, float *scale_out, uint64_t group, void *stream) {
    if (mode > SKV_RQ_MRS || !(b == 1 || b == 2 || b == 4 || b == 8) || group == 0) return SKV_ERR_INVALID_ARG;
    if ((n * b) % 8 != 0) return SKV_ERR_INVALID_ARG;
    if (n == 0) return SKV_OK;
    if (!in || !out || !aligned16(in) || !aligned16(out) || !scale_in || !scale_out ||
        ((uintptr_t)scale_in & 3u) || ((uintptr_t)scale_out & 3u))
        return SKV_ERR_INVALID_ARG;
    const uint64_t n_groups = (n + group - 1) / group;
    return launch_requantize(mode, b, in, n, out, scale_in, scale_out, n_groups,
                             static_cast<cudaStream_t>(stream)) ? SKV_ERR_CUDA : SKV_OK;
}

int32_t skv_peak_probe(int32_t kind, uint32_t iters, uint32_t *sink, uint64_t *ops, void *stream) {
    if (kind < 0 || kind >= num_probe_kinds() || iters == 0 || !sink || !ops) return SKV_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SKV_ERR_CUDA;
    const uint32_t blocks = (uint32_t)sms * 8u;
    *ops = peak_ops(kind, iters, blocks);
    return launch_peak(kind, iters, sink, blocks, static_cast<cudaStream_t>(stream)) ? SKV_ERR_CUDA : SKV_OK;
}

int32_t skv_op_table(int32_t table, uint32_t *counts, uint32_t *weights, uint32_t n) {
    if (table < 0 || table >= kNumOpTables || n != (uint32_t)kNumOpClasses || !counts || !weights)
        return SKV_ERR_INVALID_ARG;
    for (int c = 0; c < kNumOpClasses; ++c) {
        counts[c] = kOpCount[table][c];
        weights[c] = kOpWeight[c];
    }
    return SKV_OK;
}

int32_t skv_host_staging_bytes(const skv_layout *lay, uint32_t layers_per_batch, int32_t op,
                               uint64_t *bytes) {
    Geom g, gb;
    if (!bytes || (op != 0 && op != 1 && op != 2)) return SKV_ERR_INVALID_ARG;
    const int32_t r = batch_geom(lay, layers_per_batch, g, gb);
    if (r != SKV_OK) return r;
    *bytes = carve_host(g, gb, op == 1, op == 2, nullptr).bytes;
    return SKV_OK;
}

int32_t skv_encode_host(const skv_layout *lay, const void *host_kv, const void *host_mu, const float *sigma,
                        const uint64_t *counts, void *host_out, uint64_t out_capacity,
                        uint64_t *host_offsets, int32_t *status, void *staging, uint64_t staging_bytes,
                        uint32_t layers_per_batch, void *stream, void *copy_stream, void *copy_out_stream) {
    Geom g, gb;
    int32_t r = batch_geom(lay, layers_per_batch, g, gb);
    if (r != SKV_OK) return r;
    const uint32_t lpb = layers_per_batch < lay->n_layers ? layers_per_batch : lay->n_layers;
    if (!sigma || !status || (g.w_h && !counts) || !host_offsets) return SKV_ERR_INVALID_ARG;
    if (g.n_chunks && (!host_kv || !host_mu || !host_out)) return SKV_ERR_INVALID_ARG;
    if (!staging || ((uintptr_t)staging & 255u) || staging_bytes < carve_host(g, gb, true, false, nullptr).bytes)
        return SKV_ERR_INVALID_ARG;
    const HostStaging hs = carve_host(g, gb, true, false, static_cast<uint8_t *>(staging));
    cudaStream_t st = static_cast<cudaStream_t>(stream), cs = static_cast<cudaStream_t>(copy_stream);
    cudaStream_t os = static_cast<cudaStream_t>(copy_out_stream);
    EventPair copied, encoded, drained;
    if (!copied.make() || !encoded.make() || !drained.make()) return SKV_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return SKV_ERR_CUDA;
    host_offsets[0] = 0;
    if (g.n_chunks == 0) return SKV_OK;
    // tables for the whole cache, once (P_hat, 1/sigma, bf16 pairs)
    SetupArgs sa{g, sigma, counts, hs.phat, hs.rsig, hs.ep, status};
    {
        if (launch_setup(sa, st)) return SKV_ERR_CUDA;
    }
    const DtypeInfo d = dtype_info(g.dtype);
    const uint64_t plane_elems = g.T * g.HD;
    const uint32_t nb = (lay->n_layers + lpb - 1) / lpb;
    uint64_t base = 0;
    int32_t rc = SKV_OK;
    // batch b: copy in (copy stream), encode, scan, compact (stream), copy out
    // (copy-out stream, so copies in and out run at once); its output is
    // collected once the next batch is queued, so the host's wait for the
    // batch's size overlaps the GPU's work on the next one
    auto collect = [&](uint32_t b) -> int32_t {
        const int h = (int)(b & 1u);
        const uint32_t l0 = b * lpb, nl = lay->n_layers - l0 < lpb ? lay->n_layers - l0 : lpb;
        const skv_layout sl = sub_layout(lay, nl);
        Geom gs;
        if (make_geom(&sl, gs) != SKV_OK) return SKV_ERR_INVALID_ARG;   // cannot fail for a valid layout
        const uint64_t kk0 = (uint64_t)l0 * lay->n_kv * g.P;      // the batch's first chunk
        if (cudaStreamWaitEvent(os, encoded.e[h], 0) != cudaSuccess) return SKV_ERR_CUDA;
        if (cudaMemcpyAsync(host_offsets + kk0, hs.offs[h], 8ull * (gs.n_chunks + 1), cudaMemcpyDeviceToHost,
                            os) != cudaSuccess || cudaStreamSynchronize(os) != cudaSuccess)
            return SKV_ERR_CUDA;
        const uint64_t total = host_offsets[kk0 + gs.n_chunks];
        if (total > hs.out_cap || base + total > out_capacity) return SKV_ERR_CAPACITY;
        for (uint64_t j = 0; j <= gs.n_chunks; ++j) host_offsets[kk0 + j] += base;
        if (total && cudaMemcpyAsync(static_cast<uint8_t *>(host_out) + base, hs.bits[h], total,
                                     cudaMemcpyDeviceToHost, os) != cudaSuccess)
            return SKV_ERR_CUDA;
        if (cudaEventRecord(drained.e[h], os) != cudaSuccess) return SKV_ERR_CUDA;
        base += total;
        return SKV_OK;
    };
    for (uint32_t b = 0; b < nb && rc == SKV_OK; ++b) {
        const int h = (int)(b & 1u);
        const uint32_t l0 = b * lpb, nl = lay->n_layers - l0 < lpb ? lay->n_layers - l0 : lpb;
        const skv_layout sl = sub_layout(lay, nl);
        Geom gs;
        if (make_geom(&sl, gs) != SKV_OK) { rc = SKV_ERR_INVALID_ARG; break; }
        const uint64_t e0 = (uint64_t)l0 * lay->n_kv * plane_elems, ne = (uint64_t)nl * lay->n_kv * plane_elems;
        // half h is free once batch b - 2 has been encoded (inputs) and copied out (output)
        if ((b >= 2 && cudaStreamWaitEvent(cs, encoded.e[h], 0) != cudaSuccess) ||
            cudaMemcpyAsync(hs.kv[h], static_cast<const uint8_t *>(host_kv) + e0 * d.bytes, ne * d.bytes,
                            cudaMemcpyHostToDevice, cs) != cudaSuccess ||
            cudaMemcpyAsync(hs.mu[h], static_cast<const uint8_t *>(host_mu) + e0 * d.bytes, ne * d.bytes,
                            cudaMemcpyHostToDevice, cs) != cudaSuccess ||
            cudaEventRecord(copied.e[h], cs) != cudaSuccess || cudaStreamWaitEvent(st, copied.e[h], 0) != cudaSuccess ||
            (b >= 2 && cudaStreamWaitEvent(st, drained.e[h], 0) != cudaSuccess) ||
            cudaMemsetAsync(hs.ctr, 0, sizeof(unsigned long long), st) != cudaSuccess) {
            rc = SKV_ERR_CUDA;
            break;
        }
        EncArgs ea{gs, hs.kv[h], hs.mu[h], hs.phat, hs.ep, hs.rsig + (uint64_t)l0 * lay->n_kv * g.n_sblk * g.HD,
                   hs.states, hs.nwords, hs.scratch, status, hs.ctr};
        ScanArgs sc{gs, hs.nwords, hs.offs[h], hs.out_cap, status};
        CompactArgs ca{gs, hs.states, hs.nwords, hs.scratch, hs.offs[h], hs.bits[h], hs.out_cap};
        if (launch_encode(ea, st) || launch_scan(sc, st) || launch_compact(ca, st) ||
            cudaEventRecord(encoded.e[h], st) != cudaSuccess) {
            rc = SKV_ERR_CUDA;
            break;
        }
        if (b >= 1) rc = collect(b - 1);
    }
    if (rc == SKV_OK) rc = collect(nb - 1);
    // nothing of this call may still be running when it returns (the staging
    // is reused by the next call), whichever way it ends
    const bool done = cudaStreamSynchronize(cs) == cudaSuccess && cudaStreamSynchronize(st) == cudaSuccess &&
                      cudaStreamSynchronize(os) == cudaSuccess;
    return rc != SKV_OK ? rc : (done ? SKV_OK : SKV_ERR_CUDA);
}

int32_t skv_decode_host(const skv_layout *lay, const void *host_bits, uint64_t bitstream_bytes,
                        const uint64_t *host_offsets, const void *host_mu, const float *sigma,
                        const uint64_t *counts, void *host_kv_out, int32_t *status, void *staging,
                        uint64_t staging_bytes, uint32_t layers_per_batch, void *stream, void *copy_stream,
                        void *copy_out_stream) {
    Geom g, gb;
    int32_t r = batch_geom(lay, layers_per_batch, g, gb);
    if (r != SKV_OK) return r;
    const uint32_t lpb = layers_per_batch < lay->n_layers ? layers_per_batch : lay->n_layers;
    if (!sigma || !status || (g.w_h && !counts) || !host_offsets) return SKV_ERR_INVALID_ARG;
    if (g.n_chunks && (!host_bits || !host_mu || !host_kv_out)) return SKV_ERR_INVALID_ARG;
    const bool inv = staging_bytes >= carve_host(g, gb, false, true, nullptr).bytes;
    if (!staging || ((uintptr_t)staging & 255u) || staging_bytes < carve_host(g, gb, false, false, nullptr).bytes)
        return SKV_ERR_INVALID_ARG;
    if (g.n_chunks && host_offsets[0] != 0) return SKV_ERR_CORRUPT;
    for (uint64_t k = 0; k < g.n_chunks; ++k)
        if (host_offsets[k + 1] < host_offsets[k]) return SKV_ERR_CORRUPT;
    if (g.n_chunks && host_offsets[g.n_chunks] > bitstream_bytes) return SKV_ERR_CORRUPT;
    const HostStaging hs = carve_host(g, gb, false, inv, static_cast<uint8_t *>(staging));
    // a batch's bytes must fit its half
    const uint32_t nb = (lay->n_layers + lpb - 1) / lpb;
    for (uint32_t b = 0; b < nb; ++b) {
        const uint64_t k0 = (uint64_t)b * lpb * lay->n_kv * g.P;
        const uint64_t k1 = std::min<uint64_t>(g.n_chunks, k0 + (uint64_t)lpb * lay->n_kv * g.P);
        if (host_offsets[k1] - host_offsets[k0] > hs.out_cap) return SKV_ERR_CORRUPT;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream), cs = static_cast<cudaStream_t>(copy_stream);
    cudaStream_t os = static_cast<cudaStream_t>(copy_out_stream);
    EventPair copied, decoded, drained;
    if (!copied.make() || !decoded.make() || !drained.make()) return SKV_ERR_CUDA;
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return SKV_ERR_CUDA;
    if (g.n_chunks == 0) return SKV_OK;
    Workspace ws{};
    ws.phat = hs.phat; ws.rsig = hs.rsig; ws.qt = hs.qt; ws.inv_lo = hs.inv_lo; ws.inv_hi = hs.inv_hi; ws.ep = hs.ep;
    {
        SetupArgs sa{g, sigma, counts, ws.phat, ws.rsig, ws.ep, status};
        if (launch_setup(sa, st)) return SKV_ERR_CUDA;
        if (launch_search_aids(g, ws.phat, ws.qt, ws.inv_lo, ws.inv_hi, st)) return SKV_ERR_CUDA;
    }
    const DtypeInfo d = dtype_info(g.dtype);
    const uint64_t plane_elems = g.T * g.HD;
    int32_t rc = SKV_OK;
    for (uint32_t b = 0; b < nb; ++b) {
        const int h = (int)(b & 1u);
        const uint32_t l0 = b * lpb, nl = lay->n_layers - l0 < lpb ? lay->n_layers - l0 : lpb;
        const skv_layout sl = sub_layout(lay, nl);
        Geom gs;
        if (make_geom(&sl, gs) != SKV_OK) { rc = SKV_ERR_INVALID_ARG; break; }
        const uint64_t k0 = (uint64_t)l0 * lay->n_kv * g.P;
        const uint64_t o0 = host_offsets[k0], nbytes = host_offsets[k0 + gs.n_chunks] - o0;
        const uint64_t e0 = (uint64_t)l0 * lay->n_kv * plane_elems, ne = (uint64_t)nl * lay->n_kv * plane_elems;
        // half h is free once batch b - 2 has been decoded (inputs) and drained (output)
        bool ok = (b < 2 || cudaStreamWaitEvent(cs, decoded.e[h], 0) == cudaSuccess);
        ok = ok && cudaMemcpyAsync(hs.offs[h], host_offsets + k0, 8ull * (gs.n_chunks + 1), cudaMemcpyHostToDevice,
                                   cs) == cudaSuccess;
        ok = ok && (!nbytes || cudaMemcpyAsync(hs.bits[h], static_cast<const uint8_t *>(host_bits) + o0, nbytes,
                                               cudaMemcpyHostToDevice, cs) == cudaSuccess);
        ok = ok && cudaMemcpyAsync(hs.mu[h], static_cast<const uint8_t *>(host_mu) + e0 * d.bytes, ne * d.bytes,
                                   cudaMemcpyHostToDevice, cs) == cudaSuccess;
        ok = ok && cudaEventRecord(copied.e[h], cs) == cudaSuccess;
        ok = ok && cudaStreamWaitEvent(st, copied.e[h], 0) == cudaSuccess;
        ok = ok && (b < 2 || cudaStreamWaitEvent(st, drained.e[h], 0) == cudaSuccess);
        if (!ok) { rc = SKV_ERR_CUDA; break; }
        DecArgs da{gs, hs.bits[h], nbytes, hs.offs[h], hs.mu[h], ws.phat,
                   ws.rsig + (uint64_t)l0 * lay->n_kv * g.n_sblk * g.HD, ws.qt, ws.inv_lo, ws.inv_hi, nullptr,
                   gs.n_chunks, hs.kv[h], (uint64_t)g.Tc * g.HD, status, o0, 0, ws.ep, nullptr};
        if (launch_decode(da, st) || cudaEventRecord(decoded.e[h], st) != cudaSuccess) { rc = SKV_ERR_CUDA; break; }
        ok = cudaStreamWaitEvent(os, decoded.e[h], 0) == cudaSuccess;
        ok = ok && cudaMemcpyAsync(static_cast<uint8_t *>(host_kv_out) + e0 * d.bytes, hs.kv[h], ne * d.bytes,
                                   cudaMemcpyDeviceToHost, os) == cudaSuccess;
        ok = ok && cudaEventRecord(drained.e[h], os) == cudaSuccess;
        if (!ok) { rc = SKV_ERR_CUDA; break; }
    }
    const bool drained_all = cudaStreamSynchronize(cs) == cudaSuccess && cudaStreamSynchronize(st) == cudaSuccess &&
                             cudaStreamSynchronize(os) == cudaSuccess;
    return rc != SKV_OK ? rc : (drained_all ? SKV_OK : SKV_ERR_CUDA);
}

int32_t skv_search_eval(const skv_layout *lay, const uint64_t *counts, uint64_t n, const uint32_t *mu_codes,
                        const float *sigmas, const uint32_t *slots, uint32_t *o_out, uint32_t *c_out,
                        uint32_t *f_out, int32_t *status, void *workspace, uint64_t ws_bytes, void *stream) {
    Geom g;
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    if (!status || !workspace || (g.w_h && !counts)) return SKV_ERR_INVALID_ARG;
    if (n && (!mu_codes || !sigmas || !slots || !o_out || !c_out || !f_out)) return SKV_ERR_INVALID_ARG;
    if (((uintptr_t)workspace & 255u) != 0 || ws_bytes < carve(g, WS_DECODE_MIN, nullptr).bytes)
        return SKV_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return SKV_ERR_CUDA;
    const int kind = ws_bytes >= carve(g, WS_DECODE_FULL, nullptr).bytes ? WS_DECODE_FULL : WS_DECODE_MIN;
    const Workspace ws = carve(g, kind, static_cast<uint8_t *>(workspace));
    Geom g1 = g;                                       // sigma is per query: no rsig
    g1.n_planes = 0;
    SetupArgs s{g1, nullptr, counts, ws.phat, ws.rsig, ws.ep, status};
    if (launch_setup(s, st)) return SKV_ERR_CUDA;
    if (launch_search_aids(g, ws.phat, ws.qt, ws.inv_lo, ws.inv_hi, st)) return SKV_ERR_CUDA;
    SearchArgs sa{g, ws.phat, ws.ep, ws.qt, ws.inv_lo, ws.inv_hi, n, mu_codes, sigmas, slots, o_out, c_out, f_out,
                  status};
    return launch_search_eval(sa, st) ? SKV_ERR_CUDA : SKV_OK;
}

int32_t skv_decode_pages_host(const skv_layout *lay, const void *host_bitstream, uint64_t bitstream_bytes,
                              const uint64_t *host_offsets, const void *mu, const uint32_t *host_chunk_ids,
                              uint32_t n_ids, void *pages_out, int32_t *status, const void *workspace,
                              uint64_t ws_bytes, void *staging, uint64_t staging_bytes, void *stream,
                              void *copy_stream) {
    Geom g;
    int32_t r = make_geom(lay, g);
    if (r != SKV_OK) return r;
    if (!status || !workspace || ((uintptr_t)workspace & 255u) != 0) return SKV_ERR_INVALID_ARG;
    if (ws_bytes < carve(g, WS_DECODE_MIN, nullptr).bytes) return SKV_ERR_INVALID_ARG;
    if (n_ids == 0) return SKV_OK;
    if (!host_bitstream || !host_offsets || !host_chunk_ids || !mu || !pages_out || !staging ||
        ((uintptr_t)staging & 255u) || !aligned16(mu) || !aligned16(pages_out))
        return SKV_ERR_INVALID_ARG;
    // staging: [chunk ids][per-page byte offsets][the pages' bytes, back to back]
    const uint64_t ids_bytes = round256(4ull * n_ids), offs_bytes = round256(8ull * (n_ids + 1ull));
    if (staging_bytes < ids_bytes + offs_bytes) return SKV_ERR_INVALID_ARG;
    std::vector<uint64_t> uoff(n_ids + 1ull);
    uoff[0] = 0;
    for (uint32_t i = 0; i < n_ids; ++i) {
        const uint64_t k = host_chunk_ids[i];
        if (k >= g.n_chunks) return SKV_ERR_INVALID_ARG;
        const uint64_t a = host_offsets[k], b = host_offsets[k + 1];
        if (b < a || b > bitstream_bytes || ((a | b) & 15u)) return SKV_ERR_CORRUPT;
        uoff[i + 1] = uoff[i] + (b - a);
    }
    if (ids_bytes + offs_bytes + uoff[n_ids] > staging_bytes) return SKV_ERR_INVALID_ARG;
    uint8_t *base = static_cast<uint8_t *>(staging);
    uint32_t *d_ids = reinterpret_cast<uint32_t *>(base);
    uint64_t *d_off = reinterpret_cast<uint64_t *>(base + ids_bytes);
    uint8_t *d_bits = base + ids_bytes + offs_bytes;
    cudaStream_t st = static_cast<cudaStream_t>(stream), cs = static_cast<cudaStream_t>(copy_stream);
    cudaEvent_t copied = nullptr;
    if (cudaEventCreateWithFlags(&copied, cudaEventDisableTiming) != cudaSuccess) return SKV_ERR_CUDA;
    bool ok = cudaMemsetAsync(status, 0, sizeof(int32_t), st) == cudaSuccess;
    // the staging may still be read by this stream's previous decode
    cudaEvent_t prior = nullptr;
    ok = ok && cudaEventCreateWithFlags(&prior, cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventRecord(prior, st) == cudaSuccess && cudaStreamWaitEvent(cs, prior, 0) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(d_ids, host_chunk_ids, 4ull * n_ids, cudaMemcpyHostToDevice, cs) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(d_off, uoff.data(), 8ull * (n_ids + 1ull), cudaMemcpyHostToDevice, cs) == cudaSuccess;
    for (uint32_t i = 0; i < n_ids && ok; ++i) {
        const uint64_t k = host_chunk_ids[i];
        ok = cudaMemcpyAsync(d_bits + uoff[i], static_cast<const uint8_t *>(host_bitstream) + host_offsets[k],
                             uoff[i + 1] - uoff[i], cudaMemcpyHostToDevice, cs) == cudaSuccess;
    }
    ok = ok && cudaEventRecord(copied, cs) == cudaSuccess && cudaStreamWaitEvent(st, copied, 0) == cudaSuccess;
    int32_t rc = ok ? SKV_OK : SKV_ERR_CUDA;
    if (ok) {
        const int kind = ws_bytes >= carve(g, WS_DECODE_FULL, nullptr).bytes ? WS_DECODE_FULL : WS_DECODE_MIN;
        const Workspace ws = carve(g, kind, static_cast<uint8_t *>(const_cast<void *>(workspace)));
        DecArgs da{g, d_bits, uoff[n_ids], nullptr, static_cast<const uint8_t *>(mu), ws.phat, ws.rsig, ws.qt,
                   ws.inv_lo, ws.inv_hi, d_ids, n_ids, static_cast<uint8_t *>(pages_out),
                   (uint64_t)g.Tc * g.HD, status, 0, 0, ws.ep, d_off};
        rc = launch_decode(da, st) ? SKV_ERR_CUDA : SKV_OK;
    }
    if (prior) cudaEventDestroy(prior);
    cudaEventDestroy(copied);
    return rc;
}

}  // extern "C"

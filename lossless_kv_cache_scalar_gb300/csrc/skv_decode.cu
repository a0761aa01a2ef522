// skv_decode.cu -- decoder: CDF inversion fused with the rANS state update and
// word refill (SKV v1 format §§5-7), plus the per-call search aids.
//
// The decoder of the Speculative KV Coding wiki's pipeline section: from the
// bits and the same (mu, sigma) it restores every code exactly. One warp
// decodes one group of 32 streams; lane l is stream 32 g + l and walks its
// vectors in increasing order. Per scalar: slot = x mod M, find the code o
// with C(o) <= slot < C(o+1), update x, and refill one 32-bit word when x
// falls below L. Words are consumed in ascending lane order per step (a
// ballot gives each lane its index) from a per-warp shared-memory ring that
// cp.async keeps ahead of the reader.
//
// Finding o. The exact test is two evaluations of C, the same two the
// encoder makes. Where to test is estimated by inverting the Gaussian part of
// the mixture: with p_hat's share and the floor term taken at a reference
// code, the slot gives a quantile g of G(z) = (w_n Phi(z) + w_w Phi(z/3)) /
// (w_n + w_w); a table in t = -log2(min(g, 1 - g)) gives z = G^-1(g); and
// mu + z sigma rounded to the code grid is the estimate (a code owns the reals
// that round to it, SKV v1 format §2). A first pass takes the reference at
// mu's own code, a second (bf16) at the first estimate; both take P_hat from a
// coarse shared-memory table (every 32nd order, interpolated), which leaves
// their miss rate as it is with the exact P_hat. A far outlier that only
// p_hat explains (both Gaussians saturated, so C is a mu-independent function
// of o) is read from per-call inverse tables instead. When the test fails, the
// lane first takes one secant step from the exact C(o) and f(o) (all missing
// lanes at once); a lane still missing is searched by the whole warp together
// (cooperative_search). Search aids change speed only; the decoded codes are
// fixed by the exact test.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "skv_model.cuh"

namespace skv {

// CTA shape: one persistent CTA of 32 warps per SM for both code types. The
// Phi pairs, quantile table, (bf16) coarse P_hat table and (e4m3) lane-sliced
// code tables are staged once per SM; for bf16 the rest of the SM's L1 caches
// the (edge, P_hat) pair table the exact test reads. (Four 8-warp CTAs per SM measured 4%
// slower for e4m3 and 8% for bf16.)
template <uint32_t DT> struct DecShape { static constexpr int warps = 32, ctas = 1; };
static_assert(DecShape<SKV_BF16>::warps * DecShape<SKV_BF16>::ctas == (int)kDecResidentWarps &&
              DecShape<SKV_E4M3>::warps * DecShape<SKV_E4M3>::ctas == (int)kDecResidentWarps,
              "decoder residency");
constexpr uint32_t kRing = 256;        // words per warp ring: 4 blocks
constexpr uint32_t kBlock = 64;        // words per cp.async block (16 B per lane, 16 lanes)
// per warp: the word ring, then a 512-byte stage holding each lane's 16-byte
// vector of mu codes, transposed ([word][lane]) so lanes hit distinct banks;
// decoded codes overwrite their mu codes in place
constexpr uint32_t kStageWords = 4u * 32u;
constexpr uint32_t kWarpSmem = kRing + kStageWords;   // 32-bit words

// dynamic shared memory layout (bytes): Phi pairs and quantile table, then
// per code type its own tables, then the warps' word rings
constexpr uint32_t kSmPhi = 0;                                        // Tables
constexpr uint32_t kSmQt = (sizeof(Tables) + 15u) & ~15u;              // float2[kQuantN + 1]
constexpr uint32_t kSmCode = (kSmQt + 8u * (kQuantN + 1) + 15u) & ~15u;
// bf16: w_h P_hat at every 32nd code order with its slope, float2[kPcN + 1]:
// the estimates' P_hat (interpolated; the exact test reads the exact table)
constexpr uint32_t kPcShift = 5;
constexpr uint32_t kPcN = 65536u >> kPcShift;
constexpr uint32_t kSmPc = kSmCode;
// e4m3: the lane-sliced code tables (Sliced8; a single shared copy measured
// 6% slower, its bank conflicts keeping the shared-memory pipe busy)
template <uint32_t DT>
__host__ __device__ constexpr uint32_t sm_ring() {           // uint32 [warps][kWarpSmem]
    return DT == SKV_E4M3 ? ((kSmCode + 4u * Sliced8::kWords + 15u) & ~15u)
                          : ((kSmPc + 8u * (kPcN + 1) + 15u) & ~15u);
}
template <uint32_t DT>
constexpr uint32_t dec_smem() { return sm_ring<DT>() + DecShape<DT>::warps * kWarpSmem * 4u; }
static_assert(dec_smem<SKV_BF16>() <= 227u * 1024u && dec_smem<SKV_E4M3>() <= 227u * 1024u,
              "decoder shared memory above the per-CTA limit");

// ------------------------------------------------------------ search aids

// G(z) = (w_n Phi(z) + w_w Phi(z/3)) / (w_n + w_w), the Gaussian part of the mixture.
__device__ float gauss_part(float z, float wn, float ww) {
    return (wn * normcdff(z) + ww * normcdff(z / 3.0f)) / (wn + ww);
}

__device__ float gauss_quantile(float g, float wn, float ww) {
    float lo = -64.0f, hi = 64.0f;
    for (int it = 0; it < 60; ++it) {
        const float mid = 0.5f * (lo + hi);
        if (gauss_part(mid, wn, ww) < g) lo = mid; else hi = mid;
    }
    return 0.5f * (lo + hi);
}

// qt[i] = (z_i, z_{i+1} - z_i), z_i = G^-1(2^-(1 + i/32)), i = 0..kQuantN.
__global__ void __launch_bounds__(256) quant_kernel(const QuantArgs a) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i > kQuantN) return;
    float z0 = 0.0f, z1 = 0.0f;
    if (a.w_n + a.w_w != 0u) {
        const float wn = (float)a.w_n, ww = (float)a.w_w;
        z0 = gauss_quantile(exp2f(-(1.0f + (float)i / kQuantSteps)), wn, ww);
        z1 = (i < kQuantN) ? gauss_quantile(exp2f(-(1.0f + (float)(i + 1) / kQuantSteps)), wn, ww) : z0;
    }
    a.qt[2 * i] = z0;
    a.qt[2 * i + 1] = z1 - z0;
}

// C with both Gaussians saturated: base = 0 below mu (z <= -24), or
// (w_n + w_w) 2^24 above (z >= 24); then C depends on o alone.
template <uint32_t DT>
__device__ __forceinline__ uint32_t c_saturated(uint32_t o, uint32_t base, uint32_t wh,
                                                const uint32_t *__restrict__ phat) {
    constexpr uint32_t MN = (1u << Codes<DT>::m) - Codes<DT>::N;
    const uint32_t S = base + wh * __ldg(phat + o);
    return o + (uint32_t)(((uint64_t)S * MN) >> 24) / 100u;
}

// max{o in [lo, hi) : C_sat(o) <= s}, or lo when there is none; C_sat(o) is
// c_saturated with the given base, non-decreasing in o.
template <uint32_t DT>
__device__ uint32_t sat_search(uint32_t s, uint32_t base, uint32_t wh, const uint32_t *__restrict__ phat,
                               uint32_t lo, uint32_t hi) {
    while (hi - lo > 1u) {
        const uint32_t mid = (lo + hi) >> 1;
        if (c_saturated<DT>(mid, base, wh, phat) <= s) lo = mid; else hi = mid;
    }
    return lo;
}

// inv_lo[s] = max{o < N : C_lo(o) <= s}; inv_hi[s] = max{o < N : C_hi(o) <= s}, 0 if none.
// One block per 256 slots (blockIdx.y picks the table): two searches over all
// codes bound the block's answers, then each slot searches that short range.
template <uint32_t DT>
__global__ void __launch_bounds__(256) inv_kernel(const InvArgs a) {
    using K = Codes<DT>;
    const uint32_t base = blockIdx.y ? (a.g.w_n + a.g.w_w) << 24 : 0u;
    uint16_t *out = blockIdx.y ? a.inv_hi : a.inv_lo;
    __shared__ uint32_t range[2];
    const uint32_t s0 = blockIdx.x * 256u;
    if (threadIdx.x < 2)
        range[threadIdx.x] = sat_search<DT>(s0 + 255u * threadIdx.x, base, a.g.w_h, a.phat, 0u, K::N);
    __syncthreads();
    const uint32_t s = s0 + threadIdx.x;
    out[s] = (uint16_t)sat_search<DT>(s, base, a.g.w_h, a.phat, range[0], range[1] + 1u);
}

int launch_search_aids(const Geom &g, const uint32_t *phat, float *qt, uint16_t *inv_lo,
                       uint16_t *inv_hi, cudaStream_t st) {
    QuantArgs qa{g.w_n, g.w_w, qt};
    quant_kernel<<<(kQuantN + 1 + 255) / 256, 256, 0, st>>>(qa);
    if (cudaGetLastError() != cudaSuccess) return 1;
    if (inv_lo) {
        InvArgs ia{g, phat, inv_lo, inv_hi};
        if (g.dtype == SKV_BF16) inv_kernel<SKV_BF16><<<dim3((1u << 24) / 256, 2), 256, 0, st>>>(ia);
        else inv_kernel<SKV_E4M3><<<dim3((1u << 16) / 256, 2), 256, 0, st>>>(ia);
        if (cudaGetLastError() != cudaSuccess) return 1;
    }
    return 0;
}

// ------------------------------------------------------------- the search

extern __shared__ __align__(16) uint8_t skv_dec_smem[];

__device__ __forceinline__ const Tables &dtab() {
    return *reinterpret_cast<const Tables *>(skv_dec_smem + kSmPhi);
}
// this lane's entries of the lane-sliced e4m3 code tables (Sliced8's layout),
// addressed from the shared array itself so that the loads stay shared-memory
// loads (through a Sliced8 built from a plain pointer the decoder ran 2% slower)
__device__ __forceinline__ const uint32_t *dsl(uint32_t table) {
    return reinterpret_cast<const uint32_t *>(skv_dec_smem + kSmCode) + table + (threadIdx.x & 31u);
}
__device__ __forceinline__ float sl_edge(uint32_t o) { return __uint_as_float(dsl(Sliced8::kEdge)[o << 5]); }
__device__ __forceinline__ uint32_t sl_phat(uint32_t o) { return dsl(Sliced8::kPhat)[o << 5]; }
__device__ __forceinline__ float sl_value(uint32_t c) { return __uint_as_float(dsl(Sliced8::kValue)[c << 5]); }
__device__ __forceinline__ const float2 *dqt() {
    return reinterpret_cast<const float2 *>(skv_dec_smem + kSmQt);
}

// Stage the per-call tables every CTA of the decoder (or of the search check)
// reads: the Phi pairs, the quantile table, (e4m3) the code tables and (bf16)
// the estimates' coarse P_hat table.
template <uint32_t DT>
__device__ void stage_decoder_tables(const float *qt_g, const uint32_t *phat, uint32_t w_h) {
    float *qt = reinterpret_cast<float *>(skv_dec_smem + kSmQt);
    for (uint32_t i = threadIdx.x; i < kQuantFloats; i += blockDim.x) qt[i] = qt_g[i];
    if (DT == SKV_BF16) {
        float2 *pc = reinterpret_cast<float2 *>(skv_dec_smem + kSmPc);
        for (uint32_t i = threadIdx.x; i <= kPcN; i += blockDim.x) {
            const uint32_t p0 = w_h ? phat[i << kPcShift] : 0u;
            const uint32_t p1 = (w_h && i < kPcN) ? phat[(i + 1) << kPcShift] : p0;
            pc[i] = make_float2((float)w_h * (float)p0, (float)w_h * (float)(p1 - p0) * (1.0f / (1u << kPcShift)));
        }
    }
    if (DT == SKV_E4M3) stage_sliced8(skv_dec_smem + kSmCode, phat);
    stage_phi(*reinterpret_cast<Tables *>(skv_dec_smem + kSmPhi));
    __syncthreads();
}

// w_h P_hat(o) for the estimates only: bf16 interpolated in the coarse table
// (the estimate is as good as with the exact value), e4m3 exact from its table.
template <uint32_t DT>
__device__ __forceinline__ float phat_est(const DecArgs &a, uint32_t o) {
    if (DT == SKV_BF16) {
        const float2 e = reinterpret_cast<const float2 *>(skv_dec_smem + kSmPc)[o >> kPcShift];
        return fmaf((float)(o & ((1u << kPcShift) - 1u)), e.y, e.x);
    }
    return (float)(a.g.w_h * sl_phat(o));
}

// C(o) and P_hat(o) for the decoder: with EP (bf16 and a full workspace) from
// the per-call (edge bits, P_hat) pair table, else (bf16) from the code bits
// and the P_hat table, or (e4m3) from the lane-sliced code tables. All give
// the same values.
template <uint32_t DT, bool EP>
__device__ __forceinline__ uint32_t cdf_dec(const DecArgs &a, uint32_t o, float mu, float rs) {
    const Weights w{a.g.w_n, a.g.w_w, a.g.w_h};
    if (EP) return cdf_ep(dtab(), w, a.ep, o, mu, rs);
    if (DT == SKV_E4M3) return cdf_from<SKV_E4M3>(dtab(), w, sl_edge(o), sl_phat(o), o, mu, rs);
    return cdf<SKV_BF16>(dtab(), nullptr, w, a.phat, o, mu, rs);
}
template <uint32_t DT, bool EP>
__device__ __forceinline__ uint32_t phat_dec(const DecArgs &a, uint32_t o) {
    if (EP) return __ldg(&a.ep[o].y);
    if (DT == SKV_E4M3) return sl_phat(o);
    return Codes<SKV_BF16>::phat(nullptr, a.phat, o);
}

// Round a value to the nearest code (ties to even) and take its order. No
// clamp to the finite codes: every order indexes the tables (o + 1 <= N), and
// an estimate on a non-finite code is only a miss for the exact test (a
// clamp measured 1-1.4% slower).
template <uint32_t DT> __device__ __forceinline__ uint32_t nearest_ord(float x);
template <> __device__ __forceinline__ uint32_t nearest_ord<SKV_BF16>(float x) {
    return Codes<SKV_BF16>::ord((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}
template <> __device__ __forceinline__ uint32_t nearest_ord<SKV_E4M3>(float x) {
    return Codes<SKV_E4M3>::ord((uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3) & 0xFFu);
}

// One estimate of the code of slot s, with p_hat's share and the floor term
// taken at o_ref (ph = w_h P_hat(o_ref)). far: the quantile is within 2^-40 of
// an end, where only p_hat and the floor hold mass; below: nearer the low end.
// Besides the code's order it keeps what a second pass reuses: the quantile gt,
// its log2, the table's z there and the table cell's slope.
struct Estimate {
    uint32_t o;
    float gt, lg, zt, dz;
    bool far, below;
};
template <uint32_t DT>
__device__ __forceinline__ Estimate estimate(const DecArgs &a, float kS, float inv_total, uint32_t s,
                                             uint32_t o_ref, float ph, float mu, float sigma) {
    using K = Codes<DT>;
    constexpr int MN = (int)((1u << K::m) - K::N);
    Estimate r;
    const float ph_top = (float)(a.g.w_h << 24) - ph;
    // the quantile of the Gaussian part, measured from whichever end is nearer
    const int d = (int)s - (int)o_ref;
    r.below = fmaf((float)d, kS, -ph) <= 0.5f / inv_total;     // the divide is loop-invariant
    const int dd = r.below ? d : MN - d;
    // a negative dd (the slot below the reference's p_hat and floor mass) is far
    r.gt = fmaf((float)dd, kS, r.below ? -ph : -ph_top) * inv_total;
    r.far = !(r.gt >= 9.094947e-13f);                   // 2^-40
    // an estimate only: lg2 without subnormal handling (a subnormal gt is far)
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r.lg) : "f"(r.gt));
    const float u = fminf(fmaxf(fmaf(-r.lg, (float)kQuantSteps, -(float)kQuantSteps), 0.0f),
                          (float)kQuantN - 0.001f);
    const int k = (int)u;
    const float2 e = dqt()[k];
    r.zt = fmaf(u - (float)k, e.y, e.x);
    r.dz = e.y * (float)kQuantSteps;
    const float xv = fmaf(r.below ? r.zt : -r.zt, sigma, mu);
    r.o = nearest_ord<DT>(xv);
    return r;
}

// The second pass (bf16): p_hat's share and the floor term retaken at the
// first estimate o1 move the quantile by D; the new quantile's log2 moves z
// along the first pass's table cell (taken at mu's code, the first estimate
// errs outwards on the true code's side, so its side is kept).
__device__ __forceinline__ uint32_t estimate2(float kS, float inv_total, const Estimate &e1, uint32_t o_ref,
                                              float ph_ref, uint32_t o1, float ph1, float mu, float sigma,
                                              bool &far) {
    const float D = fmaf((float)(int)(o1 - o_ref), kS, ph1 - ph_ref);
    const float gt = fmaf(e1.below ? -D : D, inv_total, e1.gt);
    far = !(gt >= 9.094947e-13f);
    float lg;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(gt));
    const float zt = fmaf(e1.dz, e1.lg - lg, e1.zt);
    return nearest_ord<SKV_BF16>(fmaf(e1.below ? zt : -zt, sigma, mu));
}

// The slow path, run by the whole warp for one lane whose estimate failed.
// Lane L's slot sL, mu and 1/sigma are broadcast; each round the 32 lanes
// evaluate C at 32 ascending candidates inside the bracket [lo, hi) (C(lo) <=
// sL < C(hi), both known) and a ballot finds the sub-interval holding sL. The
// first round spreads the candidates geometrically away from the failed
// estimate (1, 2, 4, ... codes), so a near miss ends at once and a far one is
// bracketed within a factor of two; later rounds split the bracket 33 ways.
// No 16-bit code space needs more than four rounds after the first.
template <uint32_t DT, bool EP>
__device__ __forceinline__ void cooperative_search(const DecArgs &a, uint32_t L, uint32_t s, float mu,
                                                float rs, uint32_t o, uint32_t clo, uint32_t chi,
                                                uint32_t &o_out, uint32_t &c_out, uint32_t &f_out) {
    using K = Codes<DT>;
    constexpr uint32_t M = 1u << K::m;
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t sL = __shfl_sync(0xFFFFFFFFu, s, L);
    const float muL = __shfl_sync(0xFFFFFFFFu, mu, L);
    const float rsL = __shfl_sync(0xFFFFFFFFu, rs, L);
    const uint32_t oL = __shfl_sync(0xFFFFFFFFu, o, L);
    const uint32_t cloL = __shfl_sync(0xFFFFFFFFu, clo, L);
    const uint32_t chiL = __shfl_sync(0xFFFFFFFFu, chi, L);
    const bool down = sL < cloL;
    uint32_t lo, hi, Clo, Chi;
    if (down) { lo = 0; Clo = 0; hi = oL; Chi = cloL; }
    else { lo = oL + 1u; Clo = chiL; hi = K::N; Chi = M; }
    const Weights w{a.g.w_n, a.g.w_w, a.g.w_h};
    for (int round = 0; hi - lo > 1u; ++round) {
        const uint32_t span = hi - lo;
        uint32_t cand;
        if (round == 0) {
            // 1, 2, 4, ... codes away from the estimate, ascending with the lane
            cand = down ? hi - min(1u << (31u - lane), span - 1u) : lo + min(1u << lane, span - 1u);
        } else {
            cand = lo + 1u + (uint32_t)(((uint64_t)(span - 1u) * lane) / 32u);
        }
        const uint32_t c = cdf_dec<DT, EP>(a, cand, muL, rsL);
        const uint32_t le = __ballot_sync(0xFFFFFFFFu, c <= sL);   // a prefix of the lanes
        const uint32_t k = __popc(le);
        const uint32_t c_lo = __shfl_sync(0xFFFFFFFFu, c, k ? k - 1u : 0u);
        const uint32_t o_lo = __shfl_sync(0xFFFFFFFFu, cand, k ? k - 1u : 0u);
        const uint32_t c_hi = __shfl_sync(0xFFFFFFFFu, c, k < 32u ? k : 31u);
        const uint32_t o_hi = __shfl_sync(0xFFFFFFFFu, cand, k < 32u ? k : 31u);
        if (k > 0u && o_lo > lo) { lo = o_lo; Clo = c_lo; }
        if (k < 32u && o_hi < hi) { hi = o_hi; Chi = c_hi; }
    }
    if (lane == L) { o_out = lo; c_out = Clo; f_out = Chi - Clo; }
}

// max{o < N : C_sat(o) <= s} from the per-call table, or by bisection without it.
template <uint32_t DT>
__device__ __forceinline__ uint32_t saturated_inverse(const DecArgs &a, uint32_t s, uint32_t base) {
    const uint16_t *tab = base ? a.inv_hi : a.inv_lo;
    return tab ? (uint32_t)__ldg(tab + s) : sat_search<DT>(s, base, a.g.w_h, a.phat, 0u, Codes<DT>::N);
}

// The estimated code o for slot s, with c = C(o) and C(o+1) - C(o) in f; the
// caller checks C(o) <= s < C(o+1) and resolves misses cooperatively.
template <uint32_t DT, bool EP>
__device__ __forceinline__ uint32_t find_symbol(const DecArgs &a, float kS, float inv_total,
                                                uint32_t s, float mu, float rs, uint32_t o_mu,
                                                float ph_mu, uint32_t &c_out, uint32_t &f_out) {
    using K = Codes<DT>;
    const Weights w{a.g.w_n, a.g.w_w, a.g.w_h};
    uint32_t o = o_mu;
    bool far = true, below = true;
    if (w.n + w.w) {
        // sigma for the estimate only: an approximate reciprocal is enough
        float sigma;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(sigma) : "f"(rs));
        const Estimate e1 = estimate<DT>(a, kS, inv_total, s, o_mu, ph_mu, mu, sigma);
        o = e1.o;
        far = e1.far;
        below = e1.below;
        uint32_t o_far = 0;
        // a lane already far looks its code up now, so that the table load
        // overlaps the other lanes' second pass
        if (DT == SKV_BF16 && far) o_far = saturated_inverse<DT>(a, s, below ? 0u : (w.n + w.w) << 24);
        if (DT == SKV_BF16 && !far) {
            // second pass (bf16 only: e4m3's eight codes per binade leave the
            // first estimate as good as a second one)
            o = estimate2(kS, inv_total, e1, o_mu, ph_mu, o, phat_est<DT>(a, o), mu, sigma, far);
            // only p_hat holds mass this far out: the saturated inverse gives the code
            if (far) o = saturated_inverse<DT>(a, s, below ? 0u : (w.n + w.w) << 24);
        } else if (far) {
            o = DT == SKV_BF16 ? o_far : saturated_inverse<DT>(a, s, below ? 0u : (w.n + w.w) << 24);
        }
    } else {
        // p_hat alone: the saturated inverse is the answer
        o = saturated_inverse<DT>(a, s, 0u);
    }
    const uint32_t clo = cdf_dec<DT, EP>(a, o, mu, rs);
    const uint32_t chi = cdf_dec<DT, EP>(a, o + 1u, mu, rs);
    c_out = clo;
    f_out = chi - clo;
    return o;
}

// ----------------------------------------------------------------- kernel

__device__ __forceinline__ void cp_async16(uint32_t *smem, const uint32_t *gmem) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// Decode one group of 32 streams (gid = chunk unit * G + group) with this warp.
template <uint32_t DT, bool EP>
__device__ __forceinline__ void decode_group(const DecArgs &a, uint64_t gid, uint32_t *ring) {
    using K = Codes<DT>;
    constexpr uint32_t V = K::V, m = K::m;
    constexpr uint32_t M = 1u << m;
    constexpr uint64_t L = K::L;
    constexpr uint32_t BITS = 8u * K::bytes;
    const Geom &g = a.g;
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t unit = gid / g.G;
    const uint32_t grp = (uint32_t)(gid % g.G);
    const uint64_t k = a.ids ? (uint64_t)a.ids[unit] : a.chunk0 + unit;
    if (k >= g.n_chunks) {
        if (lane == 0) set_status(a.status, SKV_ERR_INVALID_ARG);
        return;
    }
    const ChunkSpan cs = chunk_span(g, k);
    // the chunk's bytes: by chunk id from the offsets table, or (pages gathered
    // into a buffer of their own) by unit from a per-unit table
    const uint64_t o0 = a.unit_offsets ? a.unit_offsets[unit] : a.offsets[k];
    const uint64_t o1 = a.unit_offsets ? a.unit_offsets[unit + 1] : a.offsets[k + 1];
    const uint64_t off0 = o0 - a.origin, off1 = o1 - a.origin;
    if (o0 < a.origin || o0 > o1 || off1 > a.stream_bytes || (off0 & 15u) || off1 - off0 < g.hdr_bytes) {
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

    const uint64_t nq = stream_vectors(g, cs.n_vec, s);
    const uint64_t nq0 = stream_vectors(g, cs.n_vec, grp * 32u);
    // the lane's vectors q = s + j W: their mu and output, by pointer steps of W vectors
    const uint4 *mvp = reinterpret_cast<const uint4 *>(a.mu + cs.elem0 * K::bytes) + s;
    uint4 *ovp = reinterpret_cast<uint4 *>(a.ids ? a.out + unit * a.page_elems * K::bytes
                                                 : a.out + cs.elem0 * K::bytes) + s;
    // sigma row of the chunk and the channel of the lane's vector (advanced by W V mod HD)
    const float *rsrow = a.rsig + sigma_row(g, k) * g.HD;
    uint32_t ch = (uint32_t)(((uint64_t)s * V) % g.HD);
    const uint32_t chstep = (uint32_t)(((uint64_t)g.W * V) % g.HD);
    const float kS = (float)(100.0 * 16777216.0 / (double)((1u << m) - K::N));
    const float inv_total = (g.w_n + g.w_w) ? 1.0f / ((float)(g.w_n + g.w_w) * 16777216.0f) : 0.0f;
    const uint32_t lt = lanemask_lt();
    bool bad_mu = false;

    // The word ring: 4 blocks of 64 words. Block b sits at ring[(64 b) mod 256];
    // when the read pointer enters block b, block b + 3 is requested and the
    // wait leaves only the two newest requests (b + 2, b + 3) in flight, so
    // blocks b and b + 1 have landed (one step reads at most 32 words).
    auto request = [&](uint32_t blk) {
        const uint32_t w0 = blk * kBlock + 4u * lane;
        if (lane < kBlock / 4 && w0 < nwp4) cp_async16(ring + (w0 & (kRing - 1)), words + w0);
        cp_async_commit();
    };
    request(0);
    request(1);
    request(2);
    request(3);
    cp_async_wait2();
    __syncwarp();
    uint32_t rp = 0;        // next word to consume (warp-uniform)

    uint32_t *stage = ring + kRing;              // [4 words][32 lanes]
    // One vector of every lane's stream. TAIL: the group's last vector, which
    // the streams past the chunk's end (the higher lanes) do not have.
    auto vector = [&](auto tail, uint64_t j) {
        constexpr bool TAIL = decltype(tail)::value;
        const bool active = !TAIL || j < nq;
        // mu of this vector into the lane's stage column; the next vector is
        // only prefetched into L2
        uint4 muv = make_uint4(0, 0, 0, 0);
        if (active) {
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(muv.x), "=r"(muv.y), "=r"(muv.z), "=r"(muv.w) : "l"(mvp));
        }
        if (j + 1 < nq) asm volatile("prefetch.global.L2 [%0];" ::"l"(mvp + g.W));
        stage[0 * 32 + lane] = muv.x;
        stage[1 * 32 + lane] = muv.y;
        stage[2 * 32 + lane] = muv.z;
        stage[3 * 32 + lane] = muv.w;
        {
            // a non-finite mu code anywhere in the vector (rare): report it and
            // model those elements with mu = +0 (SKV v1 format §4). A part of
            // t is zero exactly where a code's exponent field is all ones.
            constexpr uint32_t E = BITS == 16 ? 0x7F807F80u : 0x7F7F7F7Fu;
            constexpr uint32_t ONE = BITS == 16 ? 0x00010001u : 0x01010101u;
            constexpr uint32_t TOP = BITS == 16 ? 0x80008000u : 0x80808080u;
            auto nonfinite = [&](uint32_t w) { const uint32_t t = (w & E) ^ E; return (t - ONE) & ~t & TOP; };
            const uint32_t nf = nonfinite(muv.x) | nonfinite(muv.y) | nonfinite(muv.z) | nonfinite(muv.w);
            if (__any_sync(0xFFFFFFFFu, nf != 0u)) {
#pragma unroll 1
                for (uint32_t e = 0; e < V; ++e) {
                    const uint32_t i = ((e / (32u / BITS)) * 32u + lane) * (32u / BITS) + e % (32u / BITS);
                    const uint32_t c = BITS == 16 ? (uint32_t)reinterpret_cast<uint16_t *>(stage)[i]
                                                  : (uint32_t)reinterpret_cast<uint8_t *>(stage)[i];
                    if (!K::finite(c)) {
                        bad_mu = true;
                        if (BITS == 16) reinterpret_cast<uint16_t *>(stage)[i] = 0;
                        else reinterpret_cast<uint8_t *>(stage)[i] = 0;
                    }
                }
                __syncwarp();
            }
        }
        const float *rse = rsrow + ch;
        ch += chstep;
        if (ch >= g.HD) ch -= g.HD;
        // the lane's codes: word w of the vector at stage[32 w + lane], PER codes a word
        constexpr uint32_t PER = 32u / BITS;
#pragma unroll 1
        for (uint32_t wi = 0; wi < 4u; ++wi, rse += PER) {
            uint32_t *sw = stage + wi * 32u + lane;
            // the word's PER values of 1/sigma in one vector load (one gather
            // per word instead of per code: the lanes' channels lie 32 or 64
            // bytes apart, so each scalar load touched 32 sectors); aligned,
            // since a vector's channel is a multiple of V and rows are HD apart
            float rsv[PER];
            if constexpr (PER == 2) {
                const float2 t = __ldg(reinterpret_cast<const float2 *>(rse));
                rsv[0] = t.x;
                rsv[1] = t.y;
            } else {
                const float4 t = __ldg(reinterpret_cast<const float4 *>(rse));
                rsv[0] = t.x;
                rsv[1] = t.y;
                rsv[2] = t.z;
                rsv[3] = t.w;
            }
#pragma unroll
            for (uint32_t pi = 0; pi < PER; ++pi) {
                uint32_t slot = 0, o = 0, c = 0, f = 1;
                float mu = 0.0f, rs = 1.0f;
                bool miss = false;
                if (active) {
                    const uint32_t mc = BITS == 16 ? (uint32_t)reinterpret_cast<const uint16_t *>(sw)[pi]
                                                   : (uint32_t)reinterpret_cast<const uint8_t *>(sw)[pi];
                    mu = DT == SKV_E4M3 ? sl_value(mc) : K::value(mc);
                    rs = rsv[pi];
                    const uint32_t om = K::ord(mc);
                    const float ph = phat_est<DT>(a, om);
                    slot = (uint32_t)x & (M - 1u);
                    o = find_symbol<DT, EP>(a, kS, inv_total, slot, mu, rs, om, ph, c, f);
                    miss = slot - c >= f;    // c, slot < 2^24: c > slot wraps far above any f
                }
                // misses: first one secant step by every missing lane at once (the
                // exact C(o) and f(o) say how many codes away the slot lies), then
                // the whole warp for each lane still missing, one lane at a time
                uint32_t pending = __ballot_sync(0xFFFFFFFFu, miss);
                if (pending) {
                    if (miss) {
                        float rf;
                        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rf) : "f"((float)f));
                        int dlt = __float2int_rd((float)(int)(slot - c) * rf);
                        dlt = (int)(slot - c) < 0 ? min(dlt, -1) : max(dlt, 1);
                        const uint32_t o2 = (uint32_t)min(max((int)o + dlt, 0), (int)K::N - 1);
                        const uint32_t c2 = cdf_dec<DT, EP>(a, o2, mu, rs);
                        const uint32_t f2 = cdf_dec<DT, EP>(a, o2 + 1u, mu, rs) - c2;
                        o = o2; c = c2; f = f2;
                        miss = slot - c >= f;
                    }
                    pending = __ballot_sync(0xFFFFFFFFu, miss);
                }
                while (pending) {
                    const uint32_t Lm = __ffs(pending) - 1u;
                    pending &= pending - 1u;
                    cooperative_search<DT, EP>(a, Lm, slot, mu, rs, o, c, c + f, o, c, f);
                }
                if (active) {
                    x = (uint64_t)f * (x >> m) + slot - c;
                    // the decoded code replaces its (already read) mu code
                    if (BITS == 16) reinterpret_cast<uint16_t *>(sw)[pi] = (uint16_t)K::code(o);
                    else reinterpret_cast<uint8_t *>(sw)[pi] = (uint8_t)K::code(o);
                }
                // refill in lane order (SKV v1 format §7); a read past the group's
                // words returns stale ring data and is caught by the final checks
                const bool refill = active && x < L;
                const uint32_t ball = __ballot_sync(0xFFFFFFFFu, refill);
                const uint32_t wd = ring[(rp + __popc(ball & lt)) & (kRing - 1)];
                if (refill) x = (x << 32) | wd;
                const uint32_t rp2 = rp + __popc(ball);
                if ((rp2 ^ rp) >= kBlock) {
                    __syncwarp();    // every lane's read of the block being replaced is done
                    request((rp2 / kBlock) + 3u);
                    cp_async_wait2();
                    __syncwarp();
                }
                rp = rp2;
            }
        }
        if (active)
            *ovp = make_uint4(stage[0 * 32 + lane], stage[1 * 32 + lane], stage[2 * 32 + lane], stage[3 * 32 + lane]);
        mvp += g.W;
        ovp += g.W;
    };
    // every lane has its vector j for j < nq_all (the group's last stream has the fewest)
    const uint64_t nq_all = stream_vectors(g, cs.n_vec, grp * 32u + 31u);
    uint64_t j = 0;
    for (; j < nq_all; ++j) vector(std::false_type{}, j);
    for (; j < nq0; ++j) vector(std::true_type{}, j);
    cp_async_wait0();
    corrupt |= (x != L);
    if (lane == 0 && rp != nw) corrupt = true;     // short of, or past, the group's words
    if (__any_sync(0xFFFFFFFFu, corrupt) && lane == 0) set_status(a.status, SKV_ERR_CORRUPT);
    if (__any_sync(0xFFFFFFFFu, bad_mu) && lane == 0) set_status(a.status, SKV_ERR_NONFINITE_MU);
}

// Each CTA stages the Phi pairs, the quantile table and (e4m3) the code
// tables, then each warp decodes groups warp * gridDim.x + blockIdx.x, then
// + warps * gridDim.x, ... in turn with its own word ring (consecutive groups
// go to different CTAs, so a few pages spread over many SMs), on a persistent
// grid of at most one CTA per SM.
template <uint32_t DT, bool EP>
__global__ void __launch_bounds__(DecShape<DT>::warps * 32, DecShape<DT>::ctas) decode_kernel(const DecArgs a) {
    constexpr int kDecWarps = DecShape<DT>::warps;
    stage_decoder_tables<DT>(a.qt, a.phat, a.g.w_h);
    const uint32_t warp = threadIdx.x >> 5;
    uint32_t *ring = reinterpret_cast<uint32_t *>(skv_dec_smem + sm_ring<DT>()) + warp * kWarpSmem;
    const uint64_t n_groups = a.n_units * a.g.G;
    for (uint64_t gid = (uint64_t)warp * gridDim.x + blockIdx.x; gid < n_groups;
         gid += (uint64_t)gridDim.x * kDecWarps) {
        decode_group<DT, EP>(a, gid, ring);
        __syncwarp();
    }
}

// The decoder's search on its own: query i asks for the code of slot
// slots[i] (taken mod M) under mu_codes[i] and sigmas[i], answered exactly as
// decode_group answers it (the same estimate, check and cooperative search),
// with C(o) and f(o). For exhaustive checks of the search against the model.
template <uint32_t DT, bool EP>
__global__ void __launch_bounds__(256) search_kernel(const SearchArgs sa) {
    using K = Codes<DT>;
    constexpr uint32_t M = 1u << K::m;
    stage_decoder_tables<DT>(sa.qt, sa.phat, sa.g.w_h);
    DecArgs a{};
    a.g = sa.g;
    a.phat = sa.phat;
    a.qt = sa.qt;
    a.inv_lo = sa.inv_lo;
    a.inv_hi = sa.inv_hi;
    a.ep = sa.ep;
    a.status = sa.status;
    const Geom &g = sa.g;
    const float kS = (float)(100.0 * 16777216.0 / (double)(M - K::N));
    const float inv_total = (g.w_n + g.w_w) ? 1.0f / ((float)(g.w_n + g.w_w) * 16777216.0f) : 0.0f;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    bool bad_mu = false, bad_sig = false;
    for (uint64_t base = ((uint64_t)blockIdx.x * 8u + warp) * 32u; base < sa.n;
         base += (uint64_t)gridDim.x * 8u * 32u) {
        const uint64_t q = base + lane;
        const bool active = q < sa.n;
        const uint32_t mc = active ? sa.mu_codes[q] & ((1u << (8u * K::bytes)) - 1u) : 0u;
        const float sg = active ? sa.sigmas[q] : 1.0f;
        const bool sok = isfinite(sg) && sg >= 1.17549435e-38f;
        bad_sig |= active && !sok;
        const float rs = sok ? __frcp_rn(sg) : 1.0f;
        const bool fin = K::finite(mc);
        bad_mu |= active && !fin;
        const float mu = fin ? K::value(mc) : 0.0f;
        const uint32_t slot = active ? sa.slots[q] & (M - 1u) : 0u;
        const uint32_t o_mu = K::ord(fin ? mc : 0u);
        const float ph = phat_est<DT>(a, o_mu);
        uint32_t o = 0, c = 0, f = 1;
        bool miss = false;
        if (active) {
            o = find_symbol<DT, EP>(a, kS, inv_total, slot, mu, rs, o_mu, ph, c, f);
            miss = slot - c >= f;
        }
        uint32_t pending = __ballot_sync(0xFFFFFFFFu, miss);
        while (pending) {
            const uint32_t Lm = __ffs(pending) - 1u;
            pending &= pending - 1u;
            cooperative_search<DT, EP>(a, Lm, slot, mu, rs, o, c, c + f, o, c, f);
        }
        if (active) {
            sa.o_out[q] = o;
            sa.c_out[q] = c;
            sa.f_out[q] = f;
        }
    }
    if (bad_sig) set_status(sa.status, SKV_ERR_BAD_SIGMA);
    if (bad_mu) set_status(sa.status, SKV_ERR_NONFINITE_MU);
}

int launch_search_eval(const SearchArgs &sa, cudaStream_t st) {
    if (sa.n == 0) return 0;
    uint64_t blocks = (sa.n + 255u) / 256u;
    if (blocks > 4096u) blocks = 4096u;
    // the tables, no word rings
    const uint32_t smem = sa.g.dtype == SKV_BF16 ? sm_ring<SKV_BF16>() : sm_ring<SKV_E4M3>();
    if (sa.g.dtype == SKV_BF16) {
        if (sa.ep) {
            if (cudaFuncSetAttribute(search_kernel<SKV_BF16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem) != cudaSuccess) return 1;
            search_kernel<SKV_BF16, true><<<(unsigned)blocks, 256, smem, st>>>(sa);
        } else {
            if (cudaFuncSetAttribute(search_kernel<SKV_BF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem) != cudaSuccess) return 1;
            search_kernel<SKV_BF16, false><<<(unsigned)blocks, 256, smem, st>>>(sa);
        }
    } else {
        if (cudaFuncSetAttribute(search_kernel<SKV_E4M3, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess) return 1;
        search_kernel<SKV_E4M3, false><<<(unsigned)blocks, 256, smem, st>>>(sa);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

template <uint32_t DT, bool EP>
static int launch_decode_t(const DecArgs &a, cudaStream_t st) {
    constexpr int W = DecShape<DT>::warps;
    const uint64_t n_groups = a.n_units * a.g.G;
    uint64_t blocks = (n_groups + W - 1) / W;
    if (blocks == 0) return 0;
    if (DecShape<DT>::ctas == 1) {             // persistent: one CTA per SM, at least one group each
        blocks = n_groups;
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 1;
        if (blocks > (uint64_t)sms) blocks = (uint64_t)sms;
    }
    if (cudaFuncSetAttribute(decode_kernel<DT, EP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)dec_smem<DT>()) != cudaSuccess)
        return 1;
    decode_kernel<DT, EP><<<(unsigned)blocks, W * 32, dec_smem<DT>(), st>>>(a);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}

int launch_decode(const DecArgs &a, cudaStream_t st) {
    if (a.g.dtype != SKV_BF16) return launch_decode_t<SKV_E4M3, false>(a, st);
    return a.ep ? launch_decode_t<SKV_BF16, true>(a, st) : launch_decode_t<SKV_BF16, false>(a, st);
}

}  // namespace skv

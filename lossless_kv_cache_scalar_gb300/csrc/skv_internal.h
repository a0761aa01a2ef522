// skv_internal.h -- host/device shared geometry and kernel argument blocks.
//
// Geometry follows SKV v1 format §7: a chunk is one (layer, kv, page of
// tokens_per_chunk tokens) block, contiguous in the canonical layout; it has
// G = W/32 groups of 32 interleaved rANS streams; stream s = 32 g + lane owns
// the 16-byte vectors q with q mod W == s.
#pragma once

#include <cstdint>

#include "skv.h"

#define SKV_HD __host__ __device__ __forceinline__

namespace skv {

struct DtypeInfo {
    uint32_t N;       // codes
    uint32_t m;       // log2 of the total frequency M
    uint32_t V;       // codes per 16-byte vector
    uint32_t bytes;   // bytes per code
};

SKV_HD DtypeInfo dtype_info(uint32_t dtype) {
    DtypeInfo d;
    if (dtype == SKV_BF16) { d.N = 65536u; d.m = 24u; d.V = 8u; d.bytes = 2u; }
    else                   { d.N = 256u;   d.m = 16u; d.V = 16u; d.bytes = 1u; }
    return d;
}

// Everything a kernel needs to walk chunks and streams, precomputed on the host.
struct Geom {
    uint32_t dtype;
    uint32_t n_kv, HD, W, G, Tc;
    uint64_t T;            // tokens per plane
    uint64_t P;            // pages per plane
    uint64_t n_chunks;
    uint64_t n_groups;     // n_chunks * G
    uint64_t n_planes;     // n_layers * n_kv
    uint64_t SB;           // sigma block tokens (0: one sigma row per plane)
    uint64_t n_sblk;       // sigma rows per plane
    uint32_t w_n, w_w, w_h;
    uint32_t hdr_bytes;    // 8 W + pad16(4 G)
    uint64_t cap_words;    // scratch words per group (encoder)
};

SKV_HD uint64_t pad16(uint64_t b) { return (b + 15u) & ~uint64_t(15); }

// Chunk k: its plane, its first global element, and its vector count.
struct ChunkSpan {
    uint64_t plane;
    uint64_t elem0;
    uint64_t n_vec;
};

SKV_HD ChunkSpan chunk_span(const Geom &g, uint64_t k) {
    ChunkSpan c;
    uint64_t page = k % g.P;
    c.plane = k / g.P;
    uint64_t tok0 = page * g.Tc;
    uint64_t ntok = g.T - tok0;
    if (ntok > g.Tc) ntok = g.Tc;
    c.elem0 = (c.plane * g.T + tok0) * g.HD;
    c.n_vec = ntok * g.HD / dtype_info(g.dtype).V;
    return c;
}

// Row of the sigma table (HD entries) that chunk k reads: its plane's row, or
// with sigma blocks the row of the block holding its page (a block is a
// whole number of pages, so one row serves the whole chunk).
SKV_HD uint64_t sigma_row(const Geom &g, uint64_t k) {
    const uint64_t plane = k / g.P, page = k % g.P;
    return plane * g.n_sblk + (g.SB ? page * g.Tc / g.SB : 0);
}

// Number of vectors owned by stream s of a chunk with n_vec vectors.
SKV_HD uint64_t stream_vectors(const Geom &g, uint64_t n_vec, uint32_t s) {
    return n_vec > s ? (n_vec - s + g.W - 1) / g.W : 0;
}

struct SetupArgs {
    Geom g;
    const float *sigma;
    const uint64_t *counts;
    uint32_t *phat;        // N + 1 entries
    float *rsig;           // n_planes * HD
    uint2 *ep;             // bf16 encode only (else NULL): (edge bits, P_hat) per ordinal, N + 1
    int32_t *status;
};

struct EncArgs {
    Geom g;
    const uint8_t *kv;
    const uint8_t *mu;
    const uint32_t *phat;
    const uint2 *ep;       // bf16: (edge bits, P_hat) per ordinal
    const float *rsig;
    uint64_t *states;      // n_groups * 32
    uint32_t *nwords;      // n_groups
    uint32_t *scratch;     // n_groups * cap_words
    int32_t *status;
    unsigned long long *next_group;   // work counter, 0 at launch
};

struct ScanArgs {
    Geom g;
    const uint32_t *nwords;
    uint64_t *offsets;     // n_chunks + 1
    uint64_t out_capacity;
    int32_t *status;
};

struct CompactArgs {
    Geom g;
    const uint64_t *states;
    const uint32_t *nwords;
    const uint32_t *scratch;
    const uint64_t *offsets;
    uint8_t *out;
    uint64_t out_capacity;
};

// Decoder search aids (speed only; the output does not depend on them).
// Quantile table of the Gaussian part G of the mixture in the tail variable
// t = -log2(g): entry i holds (z_i, z_{i+1} - z_i) with z_i = G^-1(2^-(1 + i/32)),
// i = 0..kQuantN; t spans [1, 41], i.e. g down to 2^-41.
constexpr uint32_t kQuantSteps = 32;
constexpr uint32_t kQuantN = 40 * kQuantSteps;
constexpr uint32_t kQuantFloats = 2 * (kQuantN + 1);

struct QuantArgs {
    uint32_t w_n, w_w;
    float *qt;             // kQuantFloats: (z, dz) pairs
};

struct InvArgs {
    Geom g;
    const uint32_t *phat;
    uint16_t *inv_lo;      // M entries: max{o : C_lo(o) <= s}
    uint16_t *inv_hi;      // M entries: max{o : C_hi(o) <= s} (0 if none)
};

// decode_kernel keeps one persistent CTA of 32 warps resident per SM (its launch bounds).
constexpr uint32_t kDecResidentWarps = 32;

struct DecArgs {
    Geom g;
    const uint8_t *stream;
    uint64_t stream_bytes;
    const uint64_t *offsets;
    const uint8_t *mu;
    const uint32_t *phat;
    const float *rsig;
    const float *qt;           // kQuantFloats
    const uint16_t *inv_lo;    // NULL: found by bisection instead
    const uint16_t *inv_hi;
    const uint32_t *ids;   // NULL: all chunks in order; else chunk ids (page mode)
    uint64_t n_units;      // chunks to decode (n_chunks or n_ids)
    uint8_t *out;          // canonical layout, or pages of page_elems codes
    uint64_t page_elems;
    int32_t *status;
    uint64_t origin;       // stream holds the bytes from offset `origin` on (staged decode)
    uint64_t chunk0;       // without ids: unit u decodes chunk chunk0 + u
    const uint2 *ep;       // bf16 (edge bits, P_hat) pairs, or NULL: built from the code bits
    const uint64_t *unit_offsets;   // or NULL: unit u's bytes are [unit_offsets[u], unit_offsets[u+1])
};

// Slot -> code queries through the decoder's own search (checking).
struct SearchArgs {
    Geom g;
    const uint32_t *phat;
    const uint2 *ep;           // or NULL
    const float *qt;
    const uint16_t *inv_lo, *inv_hi;   // or NULL
    uint64_t n;
    const uint32_t *mu_codes;
    const float *sigmas;
    const uint32_t *slots;
    uint32_t *o_out, *c_out, *f_out;
    int32_t *status;
};

struct CdfArgs {
    Geom g;
    const uint32_t *phat;
    uint64_t n;
    const uint32_t *mu_codes;
    const float *sigmas;
    const uint32_t *ords;
    uint32_t *C;
    int32_t *status;
};

}  // namespace skv

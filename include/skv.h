/*
 * skv.h -- C ABI of the GB300 (sm_103a) speculative KV coder.
 *
 * The library entropy-codes every scalar of a KV cache against a predictor
 * and decodes it back bit for bit. The method is the one of the
 * "Speculative KV Coding" wiki (aisparkup.com): both ends hold the
 * predictor's per-element mean mu and a per-(layer, kv, head, channel) scale
 * sigma (pipeline section); each scalar is coded under the mixture
 *     q(x) = 0.95 N(x; mu, sigma^2) + 0.03 N(x; mu, (3 sigma)^2) + 0.02 p_hat(x)
 * with p_hat the empirical marginal of the codes (mixture section); the code
 * length approaches -log2 q(x) (information-theory section of the blog
 * "推测性KV编码：用预测模型实现缓存无损压缩4倍", blog.hotdry.top), and the
 * CDF must be bit-identical at both ends (that blog's deployment section).
 * The integer discretisation and the bitstream are specified by the SKV
 * bitstream format, version 1 (its sections are cited as "SKV v1 format §N").
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers must point to device memory of the
 *    current CUDA device; the caller allocates and frees all memory (inputs,
 *    outputs, workspace). The library never allocates, frees or retains
 *    caller memory.
 *  - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream) and is asynchronous: read outputs and *status
 *    after synchronising that stream.
 *  - The return value reports errors found on the host: argument errors
 *    (SKV_ERR_INVALID_ARG), found before anything is enqueued; launch errors
 *    (SKV_ERR_CUDA), after which work the call enqueued earlier may still run;
 *    and, for the calls that read offsets or sizes in host memory, the
 *    SKV_ERR_CORRUPT or SKV_ERR_CAPACITY results their entries describe.
 *    Data-dependent errors are written by the device to the int32 at
 *    `status` (device memory), which the call first sets to SKV_OK; the
 *    first error found wins. The device never traps.
 *  - Tensor layout is canonical: KV and mu are [n_layers][n_kv][n_tokens]
 *    [n_heads][head_dim] codes, channel fastest, 16-byte aligned; sigma is
 *    float32 [n_layers][n_kv][n_heads][head_dim] (with sigma blocks,
 *    [n_layers][n_kv][n_blocks][n_heads][head_dim]); counts is uint64[N], N =
 *    65536 (bf16) or 256 (e4m3), indexed by code bit pattern.
 */
#ifndef SKV_H
#define SKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SKV_FORMAT_VERSION 1u

/* Code types (SKV v1 format §1). */
enum { SKV_BF16 = 0, SKV_E4M3 = 1 };

/* Status codes: returned by calls (host-detected) or written to *status (device-detected). */
enum {
    SKV_OK = 0,
    SKV_ERR_INVALID_ARG = 1,    /* bad layout, pointer, alignment, size or chunk id      */
    SKV_ERR_CUDA = 2,           /* a CUDA call or launch failed                           */
    SKV_ERR_NONFINITE_MU = 3,   /* some mu code is NaN or infinite (modelled as 0)         */
    SKV_ERR_BAD_SIGMA = 4,      /* some sigma is non-finite or below 2^-126                */
    SKV_ERR_EMPTY_MARGINAL = 5, /* w_marginal > 0 but the counts sum to 0                  */
    SKV_ERR_CAPACITY = 6,       /* the encoded stream does not fit out_capacity            */
    SKV_ERR_CORRUPT = 7,        /* bitstream or offsets inconsistent (decode)              */
    SKV_ERR_TIMEOUT = 8         /* reserved: a bounded device wait ran out                 */
};

/*
 * What is coded and how it is cut (SKV v1 format §4 and §7).
 *  version            SKV_FORMAT_VERSION
 *  dtype              SKV_BF16 or SKV_E4M3
 *  n_layers, n_kv     planes; n_kv is 2 for K and V
 *  n_heads, head_dim  HD = n_heads * head_dim channels; HD * bytes_per_code % 16 == 0
 *  n_tokens           T (may be 0), at most 2^40; n_layers * n_kv * T * HD (the
 *                     scalars) at most 2^48 and the sigma table at most 2^40
 *                     entries, so that no size the library computes overflows
 *  tokens_per_chunk   page length T_c >= 1; a chunk is one (layer, kv, page) and
 *                     decodes independently (the random-access unit)
 *  streams_per_chunk  W = 32 * G, G in 1..8: interleaved rANS streams per chunk
 *  w_narrow, w_wide, w_marginal  integer mixture weights, sum 100 (the wiki's
 *                     0.95 / 0.03 / 0.02 are 95 / 3 / 2)
 *  sigma_block_tokens B: 0 gives one sigma per (layer, kv, head, channel) for all
 *                     tokens, the calibrated-once, frozen scale of the wiki's
 *                     predictor-choice section. B > 0 (a multiple of
 *                     tokens_per_chunk) gives one sigma per block of B tokens:
 *                     sigma is then [n_layers][n_kv][ceil(n_tokens / B)][n_heads]
 *                     [head_dim] and token t uses block t / B; this is the
 *                     position-aware sigma the blog's limitations section leaves
 *                     to future work. The bitstream format does not change.
 */
typedef struct skv_layout {
    uint32_t version;
    uint32_t dtype;
    uint32_t n_layers;
    uint32_t n_kv;
    uint32_t n_heads;
    uint32_t head_dim;
    uint64_t n_tokens;
    uint32_t tokens_per_chunk;
    uint32_t streams_per_chunk;
    uint32_t w_narrow;
    uint32_t w_wide;
    uint32_t w_marginal;
    uint32_t sigma_block_tokens; /* 0, or a multiple of tokens_per_chunk (see below) */
} skv_layout;

/* Library build/format version: returns SKV_FORMAT_VERSION. */
uint32_t skv_version(void);

/* Name of a status code ("OK", "CORRUPT", ...); never NULL. */
const char *skv_status_string(int32_t status);

/*
 * Fill *lay with the given shape and the defaults: tokens_per_chunk 256,
 * streams_per_chunk 64, weights 95/3/2 (the wiki's mixture section).
 * Returns SKV_ERR_INVALID_ARG if lay is NULL or the shape is invalid.
 */
int32_t skv_layout_init(skv_layout *lay, uint32_t dtype, uint32_t n_layers, uint32_t n_kv,
                        uint32_t n_heads, uint32_t head_dim, uint64_t n_tokens);

/* Host-side validation of a layout: SKV_OK or SKV_ERR_INVALID_ARG. */
int32_t skv_layout_check(const skv_layout *lay);

/* Number of chunks n = n_layers * n_kv * ceil(n_tokens / tokens_per_chunk). */
int32_t skv_num_chunks(const skv_layout *lay, uint64_t *n_chunks);

/*
 * Upper bound on the encoded size in bytes (SKV v1 format §8): an
 * out_capacity of this size never gives SKV_ERR_CAPACITY. About 1.56x the
 * raw bf16 bytes and 2.1x the raw e4m3 bytes, reached only by data the model
 * predicts very badly.
 */
int32_t skv_max_encoded_bytes(const skv_layout *lay, uint64_t *bytes);

/*
 * Device workspace bytes for a call on this layout, by op:
 *   1  skv_encode: the tables plus one worst-case word slot per stream group
 *      (about the size of skv_max_encoded_bytes);
 *   0  skv_decode / skv_decode_chunks, minimum: the P_hat, 1/sigma and
 *      quantile tables (< 1 MB for these shapes);
 *   2  skv_decode / skv_decode_chunks with the outlier inverse tables as well
 *      (+ 4 * 2^m bytes: 64 MiB for bf16, 256 KiB for e4m3), which make far
 *      outliers cost one lookup instead of a bisection, and for bf16 the
 *      512 KiB (edge, P_hat) pair table of the exact test. A decode call uses
 *      these tables whenever ws_bytes is at least this size; the decoded
 *      output is the same either way.
 * The workspace must be 256-byte aligned and not used by another call in flight.
 */
int32_t skv_workspace_bytes(const skv_layout *lay, int32_t op, uint64_t *bytes);

/*
 * Encode a whole KV cache (the encoder of the wiki's pipeline section).
 *  kv, mu        device, codes in canonical layout (uint16 bf16 / uint8 e4m3), 16-byte aligned
 *  sigma         device float32 [n_layers][n_kv][n_heads][head_dim], or per sigma
 *                block (see skv_layout)
 *  counts        device uint64[N], the marginal histogram (may be NULL iff w_marginal == 0);
 *                its sum must be below 2^63
 *  out           device, out_capacity bytes, 16-byte aligned: receives the chunks back to back
 *  offsets       device uint64[n_chunks + 1]: offsets[k] = byte start of chunk k,
 *                offsets[n_chunks] = total encoded bytes
 *  status        device int32
 *  workspace     device, ws_bytes >= skv_workspace_bytes(lay, 1)
 * Device errors: NONFINITE_MU, BAD_SIGMA, EMPTY_MARGINAL, CAPACITY (offsets
 * are still complete; chunks that do not fit are not written).
 */
int32_t skv_encode(const skv_layout *lay, const void *kv, const void *mu, const float *sigma,
                   const uint64_t *counts, void *out, uint64_t out_capacity, uint64_t *offsets,
                   int32_t *status, void *workspace, uint64_t ws_bytes, void *stream);

/*
 * Decode a whole bitstream back to KV codes (the decoder of the wiki's
 * pipeline section: bits plus (mu, sigma) restore KV_full exactly).
 *  bitstream     device, bitstream_bytes bytes, 16-byte aligned
 *  offsets       device uint64[n_chunks + 1] as written by skv_encode
 *  mu, sigma, counts   exactly as given to skv_encode
 *  kv_out        device, codes in canonical layout, 16-byte aligned
 *  workspace     device, ws_bytes >= skv_workspace_bytes(lay, 0) (or op 2, faster)
 * Device errors: CORRUPT (the chunk's output is then unspecified),
 * NONFINITE_MU, BAD_SIGMA, EMPTY_MARGINAL.
 */
int32_t skv_decode(const skv_layout *lay, const void *bitstream, uint64_t bitstream_bytes,
                   const uint64_t *offsets, const void *mu, const float *sigma,
                   const uint64_t *counts, void *kv_out, int32_t *status, void *workspace,
                   uint64_t ws_bytes, void *stream);

/*
 * Random-access decode of selected chunks (pages) of a full bitstream, for
 * the offload and long-context uses the wiki lists (uses section).
 *  chunk_ids     device uint32[n_ids], each < n_chunks (else SKV_ERR_INVALID_ARG on *status)
 *  pages_out     device, n_ids * tokens_per_chunk * HD codes, 16-byte aligned; chunk
 *                chunk_ids[i] is written at pages_out + i * tokens_per_chunk * HD codes,
 *                in its own [token][head][channel] order (a shorter last page leaves
 *                the rest of its slot untouched)
 * Other arguments as skv_decode.
 */
int32_t skv_decode_chunks(const skv_layout *lay, const void *bitstream, uint64_t bitstream_bytes,
                          const uint64_t *offsets, const void *mu, const float *sigma,
                          const uint64_t *counts, const uint32_t *chunk_ids, uint32_t n_ids,
                          void *pages_out, int32_t *status, void *workspace, uint64_t ws_bytes,
                          void *stream);

/*
 * Random access without per-call set-up. skv_decode_prepare builds the
 * decoder's tables (P_hat, 1/sigma, quantile and, with a workspace of
 * skv_workspace_bytes(lay, 2), the outlier inverse tables) into the workspace
 * once; skv_decode_chunks_prepared then decodes pages exactly as
 * skv_decode_chunks does, reading those tables, for as many calls as the
 * tables stay valid: the same layout, sigma, counts, workspace and ws_bytes,
 * and no other call using that workspace in between. This serves the page
 * access the wiki's uses section describes (offload, long context), where a
 * few pages are wanted at a time and the set-up would dominate.
 * skv_decode_prepare writes BAD_SIGMA / EMPTY_MARGINAL to *status; check it
 * before decoding (the decode call resets *status). Arguments as in
 * skv_decode_chunks; the workspace is only read by the decode call.
 */
int32_t skv_decode_prepare(const skv_layout *lay, const float *sigma, const uint64_t *counts,
                           int32_t *status, void *workspace, uint64_t ws_bytes, void *stream);
int32_t skv_decode_chunks_prepared(const skv_layout *lay, const void *bitstream,
                                   uint64_t bitstream_bytes, const uint64_t *offsets, const void *mu,
                                   const uint32_t *chunk_ids, uint32_t n_ids, void *pages_out,
                                   int32_t *status, const void *workspace, uint64_t ws_bytes,
                                   void *stream);

/*
 * Decode a whole cache whose bitstream sits in host memory: the offload use of
 * the wiki's uses section (KV kept compressed off the GPU and brought back
 * over the host link). The chunks are copied in batches into two halves of a
 * device staging buffer on copy_stream while the previous batch decodes on
 * stream, so transfer and decode overlap; each batch is the longest run of
 * whole chunks (in chunk order) whose bytes fit one half. The result is the
 * same as skv_decode's on a device copy of the stream.
 *  host_bitstream  host memory (page-locked, e.g. cudaHostAlloc, for the copies to
 *                  overlap), bitstream_bytes bytes: the stream skv_encode wrote
 *  host_offsets    host uint64[n_chunks + 1]: the offsets (used to plan the batches)
 *  offsets         device uint64[n_chunks + 1]: the same values (read by the decoder)
 *  staging         device, staging_bytes, 16-byte aligned; each half must hold the
 *                  largest chunk (else SKV_ERR_INVALID_ARG). Halves large enough for
 *                  a few hundred chunks keep every SM busy.
 *  stream, copy_stream  decode and copy streams (cudaStream_t as void*), distinct
 *                  for overlap; the call returns once everything is enqueued.
 * Other arguments and device errors as skv_decode. Host-detected: offsets that
 * are not ascending from 0 or pass bitstream_bytes return SKV_ERR_CORRUPT and
 * nothing is enqueued. host_bitstream and staging must stay untouched until
 * stream has finished.
 */
int32_t skv_decode_offload(const skv_layout *lay, const void *host_bitstream, uint64_t bitstream_bytes,
                           const uint64_t *host_offsets, const uint64_t *offsets, const void *mu,
                           const float *sigma, const uint64_t *counts, void *kv_out, int32_t *status,
                           void *workspace, uint64_t ws_bytes, void *staging, uint64_t staging_bytes,
                           void *stream, void *copy_stream);

/*
 * Random-access page decode from host memory: the pages (chunks) listed in
 * host_chunk_ids are copied from the host bitstream into the staging buffer
 * on copy_stream (one copy per page) and decoded on stream, with the tables
 * skv_decode_prepare built in the workspace (as skv_decode_chunks_prepared).
 * The KV stays compressed in host memory and only the pages a request needs
 * cross the link (the offload use of the wiki's uses section).
 *  host_bitstream, host_offsets  host, as skv_encode wrote them
 *  host_chunk_ids  host uint32[n_ids], each < n_chunks (else SKV_ERR_INVALID_ARG)
 *  pages_out       device, as skv_decode_chunks
 *  staging         device, 256-byte aligned: 4 n_ids and 8 (n_ids + 1) bytes (each
 *                  rounded up to 256) plus the listed pages' bytes, else
 *                  SKV_ERR_INVALID_ARG; it must not be reused until stream has
 *                  finished this call's work
 * Offsets that descend, pass bitstream_bytes or are not 16-byte multiples
 * return SKV_ERR_CORRUPT. Device errors as skv_decode_chunks_prepared.
 * Host buffers: host_offsets is read only during the call. host_chunk_ids and
 * the listed pages of host_bitstream are also the sources of asynchronous
 * copies on copy_stream: from pageable memory CUDA stages them before the call
 * returns, but from pinned memory they are read when copy_stream runs, so a
 * pinned host_chunk_ids or host_bitstream must stay unchanged until
 * copy_stream has passed this call's copies (e.g. until stream has finished).
 */
int32_t skv_decode_pages_host(const skv_layout *lay, const void *host_bitstream, uint64_t bitstream_bytes,
                              const uint64_t *host_offsets, const void *mu, const uint32_t *host_chunk_ids,
                              uint32_t n_ids, void *pages_out, int32_t *status, const void *workspace,
                              uint64_t ws_bytes, void *staging, uint64_t staging_bytes, void *stream,
                              void *copy_stream);

/*
 * The batch plan skv_decode_offload follows (host only, no CUDA call): cut
 * chunks 0..n_chunks-1 into runs of whole chunks of at most batch_bytes bytes
 * and (if max_chunks > 0) at most max_chunks chunks each, in order, each run
 * as long as it can be. skv_decode_offload takes max_chunks = a whole number
 * of decoder waves (the chunks whose warps fit on the GPU at once). batch_first[i] = first chunk
 * of batch i, batch_first[n_batches] = n_chunks; pass max_batches = 0 (and
 * batch_first = NULL) to get only *n_batches. SKV_ERR_INVALID_ARG if a chunk
 * is larger than batch_bytes or max_batches < n_batches + 1; SKV_ERR_CORRUPT
 * if the offsets descend.
 */
int32_t skv_offload_plan(const uint64_t *host_offsets, uint64_t n_chunks, uint64_t batch_bytes,
                         uint64_t max_chunks, uint64_t *batch_first, uint64_t max_batches,
                         uint64_t *n_batches);

/*
 * Evaluate the model's cumulative frequency C(o) (SKV v1 format §5) for n
 * independent queries: C[i] = C(ords[i]) for predictor code mu_codes[i] and
 * scale sigmas[i], under the weights of lay and the marginal counts. For
 * checking the model kernel against an independent implementation.
 *  mu_codes (uint32, code in the low bits), sigmas (float32), ords (uint32, 0..N),
 *  C_out (uint32): device arrays of n entries. workspace >= skv_workspace_bytes(lay, 0).
 * Device errors: NONFINITE_MU, BAD_SIGMA, EMPTY_MARGINAL.
 */
int32_t skv_cdf_eval(const skv_layout *lay, const uint64_t *counts, uint64_t n,
                     const uint32_t *mu_codes, const float *sigmas, const uint32_t *ords,
                     uint32_t *C_out, int32_t *status, void *workspace, uint64_t ws_bytes,
                     void *stream);

/*
 * Histogram of codes: the counts behind p_hat, the empirical marginal of the
 * wiki's mixture section. counts[b] += the number of i < n with codes[i] == b
 * (bit pattern; every pattern is counted, NaN codes included), over N = 65536
 * (bf16) or 256 (e4m3) bins.
 *  dtype       SKV_BF16 or SKV_E4M3
 *  codes       device, n codes (uint16 / uint8), aligned to the code size; any
 *              flat view of a cache (a whole cache, one layer, one page)
 *  counts      device uint64[N], 8-byte aligned; zeroed first unless accumulate != 0,
 *              so per-layer or per-rank histograms can be summed in place
 * No device errors (status is not used). The bf16 kernel keeps the codes of
 * magnitude below 2^65 in 192 KB of shared-memory bins per SM and adds any
 * others straight to counts, so it is exact for every input.
 */
int32_t skv_histogram(uint32_t dtype, const void *codes, uint64_t n, uint64_t *counts,
                      int32_t accumulate, void *stream);

/*
 * Calibrate sigma once from the first t_cal tokens and freeze it: the
 * per-(kv, head, channel) scale of the wiki's predictor-choice section and of
 * the blog's predictor-engineering section, taken per layer as well. The
 * blog's information-theory section gives the optimum Gaussian scale as the
 * residual's mean square about mu, so for each (layer, kv, channel) -- and,
 * when lay->sigma_block_tokens = B > 0, for each block of B tokens, from the
 * first t_cal tokens of that block:
 *     r  = fl64(value(kv) - value(mu))   over those tokens in ascending order,
 *                                         elements with both codes finite and
 *                                         (if mask != NULL) a nonzero mask byte
 *     S  = sum of fl64(r * r) in binary64, added in that order
 *     sigma = fl32(sqrt(fl64(S / count)))  (IEEE round to nearest at each step)
 * clamped into [2^-126, FLT_MAX] so that it is always a valid coding sigma
 * (no counted element gives 2^-126). Values are in code units (for e4m3, the
 * stored code's value, before any per-tensor scale).
 *  kv, mu      device codes in canonical layout
 *  mask        device uint8, canonical layout like kv, or NULL (count every element):
 *              leaves outliers out of the calibration, as a clean calibration set would
 *  t_cal       1 <= t_cal <= n_tokens, and t_cal <= B with sigma blocks (a shorter
 *              last block uses all of its tokens)
 *  sigma       device float32 [n_layers][n_kv][n_heads][head_dim], or
 *              [n_layers][n_kv][n_blocks][n_heads][head_dim] with sigma blocks (output)
 * No device errors. Bit-exact: the same inputs always give the same sigma.
 */
int32_t skv_calibrate_sigma(const skv_layout *lay, const void *kv, const void *mu, const uint8_t *mask,
                            uint64_t t_cal, float *sigma, void *stream);

/*
 * Encode and decode with the cache in host memory (the offload use of the
 * wiki's uses section, end to end): batches of layers_per_batch layers go
 * through two halves of a device staging buffer, host-to-device copies on
 * copy_stream and device-to-host copies on copy_out_stream overlapping each
 * other and the kernels on stream (three distinct streams). The
 * bitstream is byte for byte skv_encode's (chunks code independently, and a
 * batch is a run of whole chunks). Both calls return when everything has
 * landed in host memory; host buffers should be page-locked for the copies to
 * overlap. Device errors go to *status as in skv_encode / skv_decode.
 *  skv_host_staging_bytes  device staging both calls need: op 1 encode, 0 decode,
 *                          2 decode with the outlier inverse tables (faster);
 *                          decode uses them whenever staging_bytes allows
 *  skv_encode_host  host_kv, host_mu: codes in canonical layout (host);
 *                   host_out: out_capacity bytes (host); host_offsets: uint64[n_chunks + 1]
 *                   (host, written); returns SKV_ERR_CAPACITY if the stream does not fit
 *  skv_decode_host  host_bits / host_offsets as skv_encode_host wrote them; host_kv_out
 *                   (host, canonical layout); offsets that descend, pass bitstream_bytes or
 *                   give a batch more bytes than its half holds return SKV_ERR_CORRUPT
 * sigma and counts are device arrays as for skv_encode.
 */
int32_t skv_host_staging_bytes(const skv_layout *lay, uint32_t layers_per_batch, int32_t op,
                               uint64_t *bytes);
int32_t skv_encode_host(const skv_layout *lay, const void *host_kv, const void *host_mu, const float *sigma,
                        const uint64_t *counts, void *host_out, uint64_t out_capacity,
                        uint64_t *host_offsets, int32_t *status, void *staging, uint64_t staging_bytes,
                        uint32_t layers_per_batch, void *stream, void *copy_stream, void *copy_out_stream);
int32_t skv_decode_host(const skv_layout *lay, const void *host_bits, uint64_t bitstream_bytes,
                        const uint64_t *host_offsets, const void *host_mu, const float *sigma,
                        const uint64_t *counts, void *host_kv_out, int32_t *status, void *staging,
                        uint64_t staging_bytes, uint32_t layers_per_batch, void *stream, void *copy_stream,
                        void *copy_out_stream);

/*
 * Lower quantised KV codes from 2b to b bits (the progressive quantisation of
 * PM-KVQ, which the third page's PM-KVQ section describes next to the coder;
 * a lossy step outside the lossless path). mode:
 *   SKV_RQ_ERS  Equivalent Right Shift: zero point kept, scale_out = fl32((2^b + 1)
 *               scale_in), code round(q / (2^b + 1)) -- the same as dequantising
 *               with scale_in and requantising with scale_out, done with integer
 *               adds and shifts;
 *   SKV_RQ_DRS  Direct Right Shift: q >> b, scale_out = 2^b scale_in;
 *   SKV_RQ_MRS  Modified Right Shift (round instead of truncate):
 *               min((q + 2^(b-1)) >> b, 2^b - 1), scale_out = 2^b scale_in.
 *  b           1, 2, 4 or 8 (2 -> 1, 4 -> 2, 8 -> 4, 16 -> 8 bits)
 *  in          device, n codes of 2b bits packed from the least significant bit
 *              (code i in bits [2b i, 2b i + 2b) of the byte string), 16-byte aligned
 *  out         device, n b / 8 bytes of b-bit codes packed the same way, 16-byte aligned
 *  n           a multiple of 8 / b
 *  scale_in, scale_out  device float32, one per group of `group` consecutive codes
 * No device errors.
 */
enum { SKV_RQ_ERS = 0, SKV_RQ_DRS = 1, SKV_RQ_MRS = 2 };
int32_t skv_requantize(uint32_t mode, uint32_t b, const void *in, uint64_t n, void *out,
                       const float *scale_in, float *scale_out, uint64_t group, void *stream);

/*
 * Measurement aid (the pages describe no such call): one launch of an
 * arithmetic issue-rate probe, for the arithmetic roofline of the coder's
 * kernels. kind 0..15: one instruction class of the operation count in the
 * SKV v1 format's section 9 (0 binary32 add/mul/fma, 1 binary32 min/max,
 * 2 integer add, 3 logic (lop3), 4 shift, 5 integer min/max, 6 integer
 * multiply-add, 7 multiply-high, 8 32x32->64 multiply, 9 float/integer
 * conversion, 10 rcp/lg2 approximation, 11 popc, 12 ballot (with its setp),
 * 13 shared-memory load, 14 L1-resident global load, 15 shared-memory store);
 * *ops receives the launch's 32-bit operations (the class's weight per
 * instruction). kind 16..19: the whole operation table of bf16 encode, bf16
 * decode, e4m3 encode, e4m3 decode, issued with full instruction-level
 * parallelism; *ops receives the scalars modelled (each scalar's operations
 * are the table's counts). Every SM runs 8 CTAs of 256 threads, each thread
 * 8 independent chains. *ops is written on the host at once; time the launch
 * on `stream` (CUDA events) for the rate.
 * sink: device uint32, written only if the chains hit one unlikely value.
 */
int32_t skv_peak_probe(int32_t kind, uint32_t iters, uint32_t *sink, uint64_t *ops, void *stream);

/*
 * The operation count of the SKV v1 format's section 9 as this library holds
 * it (the pages describe no such table; it defines the arithmetic roofline).
 * table: 0 bf16 encode, 1 bf16 decode, 2 e4m3 encode, 3 e4m3 decode.
 * counts[c] receives the instructions of class c per scalar and weights[c]
 * its 32-bit operations per instruction, for the n = 16 classes of
 * skv_peak_probe. Host only, no device work; INVALID_ARG for another n.
 */
int32_t skv_op_table(int32_t table, uint32_t *counts, uint32_t *weights, uint32_t n);

/*
 * The decoder's slot-to-code search on its own, for exhaustive checks: query
 * i returns the code ordinal o with C(o) <= s < C(o+1) for s = slots[i] mod M,
 * under predictor code mu_codes[i] and scale sigmas[i], found exactly as
 * skv_decode finds it (the same estimate, exact test and cooperative search,
 * the same tables: with a workspace of skv_workspace_bytes(lay, 2) the
 * (edge, P_hat) pairs and the outlier inverse tables too), with c_out = C(o)
 * and f_out = C(o+1) - C(o). All arrays device, n entries (uint32, float32).
 * Device errors: NONFINITE_MU, BAD_SIGMA, EMPTY_MARGINAL.
 */
int32_t skv_search_eval(const skv_layout *lay, const uint64_t *counts, uint64_t n, const uint32_t *mu_codes,
                        const float *sigmas, const uint32_t *slots, uint32_t *o_out, uint32_t *c_out,
                        uint32_t *f_out, int32_t *status, void *workspace, uint64_t ws_bytes, void *stream);

/*
 * Decode without any caller-provided scratch (the pages describe no such
 * call; it serves deployment only). Same contract and outputs as skv_decode,
 * minus the workspace arguments. It is meant for callers that cannot call
 * cudaMalloc or lend a workspace: a host program whose memory pool owns all
 * device memory and gives this library no allocator, or a latency-critical
 * path where allocating (and the device-wide synchronisation that freeing
 * brings) is not allowed.
 *
 * Its scratch is a fixed device array of SKV_NOALLOC_SCRATCH_BYTES inside the
 * library, held by every GPU that loads the library until the process exits.
 * Layouts whose minimum decode scratch (skv_workspace_bytes(lay, 0, ...): the
 * P_hat and quantile tables plus 4 bytes per sigma entry, i.e. per (layer, kv,
 * sigma block, channel)) exceeds it are rejected with SKV_ERR_INVALID_ARG
 * before anything is enqueued; for bf16, 1 MiB covers up to 193,920 sigma
 * entries, e.g. 80 planes (40 layers, K and V) of 2,048 channels with one
 * sigma per channel, or fewer planes when the layout has several sigma blocks.
 * The bf16 decoder's optional tables (the (edge, P_hat) pairs and the outlier
 * inverse tables, tens of MiB) do not fit, so its far outliers are found by
 * bisection (same output, slower); an e4m3 layout's full workspace is small
 * and, when it fits, the call uses it whole.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture. The
 * address is kept for the life of the process: after a cudaDeviceReset the
 * library's device array (and that address) no longer exist, so do not call
 * this entry point again in the same process after a reset. Every call
 * on a device shares the one array and each call rewrites all of it that it
 * reads, so nothing carries over between calls; calls that overlap on the GPU
 * (on different streams, or from several host threads) race on it and must be
 * serialised by the caller. No memory is allocated or freed.
 */
#define SKV_NOALLOC_SCRATCH_BYTES (1u << 20)
int32_t skv_decode_noalloc(const skv_layout *lay, const void *bitstream, uint64_t bitstream_bytes,
                           const uint64_t *offsets, const void *mu, const float *sigma,
                           const uint64_t *counts, void *kv_out, int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SKV_H */

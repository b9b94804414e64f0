/*
 * polykv.h -- C ABI of libpolykv: one shared, asymmetrically compressed KV
 * pool written once and read by N concurrent agents, on one GB300 (sm_103a).
 *
 * The operations follow "PolyKV: A Shared Asymmetrically-Compressed KV Cache
 * Pool for Multi-Agent LLM Inference" (arXiv 2604.24971), abstract: a
 * compressed cache is written once and read by N independent agents; keys are
 * int8 q8_0; values are rotated by a Fast Walsh-Hadamard Transform (FWHT) and
 * quantized to 3-bit Lloyd-Max codes with centroids tuned to N(0,1).
 *
 * Conventions for every call:
 *   - All tensors are caller-owned. Device pointers must point to memory of
 *     the current CUDA device; the library allocates no device memory itself.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Device work is enqueued asynchronously on it; the call returns
 *     once the launch is issued. Asynchronous faults surface on the caller's
 *     next synchronisation, as with any CUDA launch.
 *   - Every call returns a polykv_status and never throws across the ABI.
 *     On failure nothing is enqueued, and polykv_last_error() returns a
 *     message for the calling host thread.
 *   - fp16 / bf16 tensors are passed as raw 16-bit storage (uint16_t
 *     bit patterns); the pool's in_dtype says which.
 *   - Device pointers passed to encode/attend must be 16-byte aligned.
 */
#ifndef POLYKV_H
#define POLYKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define POLYKV_API __attribute__((visibility("default")))
#else
#define POLYKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct polykv_pool polykv_pool; /* opaque host handle */

typedef enum {
    POLYKV_OK = 0,
    POLYKV_E_INVAL = 1,            /* bad argument: null pointer, shape, alignment */
    POLYKV_E_UNSUPPORTED = 2,      /* valid but not implemented (e.g. head_dim not 64/128) */
    POLYKV_E_BUFFER_TOO_SMALL = 3, /* dev_buf or workspace smaller than required */
    POLYKV_E_CUDA = 4,             /* a CUDA launch or query failed */
    POLYKV_E_TIMEOUT = 5,          /* a bounded device-side wait gave up */
    POLYKV_E_STATE = 6             /* call order violated (e.g. attend beyond encoded tokens) */
} polykv_status;

typedef enum { POLYKV_F16 = 0, POLYKV_BF16 = 1 } polykv_dtype;

/* Pool geometry. head_dim must be 64 or 128 (a multiple of the 32-element
 * q8_0 block and a power of two for the FWHT). */
typedef struct {
    int32_t n_layers;
    int32_t n_kv_heads;
    int32_t head_dim;
    int64_t capacity_tokens; /* tokens the pool can hold per (layer, kv head) */
    polykv_dtype in_dtype;   /* dtype of K, V and queries handed to the calls */
} polykv_pool_desc;

/* Where the pool's fields live inside dev_buf (byte offsets from dev_buf).
 * With U = n_layers * n_kv_heads units and C = capacity_rounded tokens,
 * unit u = layer * n_kv_heads + kv_head, token t:
 *   k_codes  int8    [U][C][head_dim]        at k_codes_off + (u*C + t)*head_dim
 *   k_scales fp16    [U][C][head_dim/32]     at k_scales_off + 2*((u*C + t)*head_dim/32 + block)
 *   v_codes  uint8   [U][C/32][head_dim][12] per group of 32 consecutive tokens and coordinate j,
 *                                            one little-endian 96-bit string holding the 3-bit codes
 *                                            of the group's tokens, token t at bits 3(t%32)..3(t%32)+2
 *                                            (3 bits per code, 3*head_dim/8 bytes per token)
 *   v_norms  fp16    [U][C]                  ||v|| of the unrotated value vector
 */
typedef struct {
    int64_t capacity_rounded; /* capacity_tokens rounded up to a multiple of 128 */
    size_t k_codes_off;
    size_t k_scales_off;
    size_t v_codes_off;
    size_t v_norms_off;
    size_t status_off;        /* uint32 status word (see polykv_pool_status) */
    size_t v_nmax_off;        /* float [U]: running max of ||v|| per unit (kept by encode) */
    size_t header_bytes;      /* [status_off, header_bytes) is cleared by the first encode */
    size_t total_bytes;
} polykv_pool_regions;

/* Create a pool handle over caller-provided device memory.
 * Defined by the abstract's "writes a compressed cache once": the pool is
 * one flat buffer shared by all readers.
 *   desc            geometry (copied; not retained).
 *   dev_buf         device buffer of at least *required_bytes bytes, 256-byte
 *                   aligned, owned by the caller for the life of the handle.
 *                   NULL = query mode: only *required_bytes is set and
 *                   *out is left untouched.
 *   dev_buf_bytes   size of dev_buf.
 *   out             receives the handle (host memory owned by the library;
 *                   release with polykv_free). May be NULL in query mode.
 *   required_bytes  receives the bytes the pool needs (may be NULL when
 *                   dev_buf is not NULL).
 * Enqueues no device work; the pool's contents are undefined until encoded
 * (the first polykv_encode clears the pool header on its stream).
 * Errors: E_INVAL (null desc, non-positive sizes, misaligned dev_buf),
 * E_UNSUPPORTED (head_dim not 64/128), E_BUFFER_TOO_SMALL. */
POLYKV_API polykv_status polykv_pool_create(const polykv_pool_desc* desc, void* dev_buf, size_t dev_buf_bytes,
                                 polykv_pool** out, size_t* required_bytes);

/* Byte offsets of the pool's fields inside dev_buf (host only). */
POLYKV_API polykv_status polykv_pool_get_regions(const polykv_pool* pool, polykv_pool_regions* out);

/* Encode ("write the pool"): quantize keys to q8_0 and values to FWHT + 3-bit
 * Lloyd-Max codes for pool tokens [t0, t0 + n_tokens).
 * Defined by the abstract's asymmetric compression: keys int8 q8_0 (32-element
 * blocks along head_dim, fp16 scale s = fp16(max|x| / 127), codes
 * round-half-away(x / s) in [-127, 127]); values: u = H v / ||v|| with H the
 * Sylvester Hadamard matrix (the normalized FWHT scaled by sqrt(d)/||v||),
 * code = number of Lloyd-Max decision boundaries <= u, ||v|| stored as fp16.
 *   k, v      device, in_dtype bits, [n_layers][n_kv_heads][n_tokens][head_dim]
 *             contiguous.
 *   t0        first pool token written; must be <= the number of tokens
 *             already encoded (appending or overwriting, no gaps).
 *   n_tokens  >= 0; t0 + n_tokens <= capacity_tokens. 0 is a no-op.
 * One kernel launch on `stream`. Ordering against attend calls on the same
 * pool is the caller's job (same stream or events): one writer, then readers.
 * The encode also raises the per-unit maximum of ||v|| kept in the pool header
 * (attention uses it to scale fp16 operands); the first encode into a pool
 * clears that header first (a cudaMemsetAsync on `stream`).
 * Non-finite keys: a 32-element block holding an infinity or a NaN gets a
 * non-finite scale and all-zero codes (attention over such a pool is
 * undefined). Non-finite values are not supported.
 * Errors: E_INVAL, E_STATE (t0 beyond the encoded prefix), E_CUDA. */
POLYKV_API polykv_status polykv_encode(polykv_pool* pool, const void* k, const void* v, int64_t t0, int64_t n_tokens,
                            void* stream);

/* Bytes of device workspace polykv_attend needs for these arguments. The
 * workspace holds per-split softmax partials; it may be reused by calls that
 * are ordered on the GPU, and must not be shared by calls that may overlap. */
POLYKV_API polykv_status polykv_attend_workspace_size(const polykv_pool* pool, int32_t n_agents, int32_t n_q_heads,
                                           int64_t n_ctx, size_t* bytes);

/* Multi-agent decode attention over pool tokens [0, n_ctx).
 * Defined by the abstract's "multi-reader concurrent agent access": every
 * agent's decode query attends over the same compressed pool. Output
 *   out[l][a][hq][:] = sum_t softmax_t(scale * q . k_hat_t) v_hat_t
 * with k_hat the dequantized q8_0 key, v_hat = (||v||_fp16 / d) H C[code]
 * (H C[code] is the inverse normalized FWHT up to the 1/sqrt(d) factors) and
 * q head hq reading kv head hq / (n_q_heads / n_kv_heads).
 *   q         device, in_dtype bits, [n_layers][n_agents][n_q_heads][head_dim].
 *   out       device, float32, same shape as q.
 *   n_agents  >= 1; n_q_heads a positive multiple of n_kv_heads.
 *   n_ctx     1 <= n_ctx <= tokens encoded so far.
 *   softmax_scale  <= 0 selects 1/sqrt(head_dim).
 *   workspace device buffer of >= polykv_attend_workspace_size bytes,
 *             16-byte aligned (may be NULL when that size is 0).
 * Errors: E_INVAL, E_STATE, E_BUFFER_TOO_SMALL, E_UNSUPPORTED, E_CUDA. */
POLYKV_API polykv_status polykv_attend(const polykv_pool* pool, const void* q, float* out, int32_t n_agents,
                            int32_t n_q_heads, int64_t n_ctx, float softmax_scale, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Extensions of an attend call (zero-initialise and set what is used). */
typedef struct {
    /* Private per-agent suffix: each agent's own uncompressed recent tokens, attended together with
     * the pool under ONE softmax. in_dtype bits, [n_layers][n_agents][n_kv_heads][suffix_len][head_dim]
     * contiguous, device, 16-byte aligned. suffix_len = 0 disables it. At most 16 query heads per
     * kv head. */
    const void* suffix_k;
    const void* suffix_v;
    int64_t suffix_len;
    /* Query-chunk mode: each agent brings chunk_len query tokens, each with its own key and value
     * (in_dtype bits, chunk_k / chunk_v [n_layers][n_agents][n_kv_heads][chunk_len][head_dim]
     * contiguous, device, 16-byte aligned). Query token c of an agent attends the whole pool plus
     * that agent's chunk tokens 0..c (causal inside the chunk), under one softmax. q and out are then
     * [n_layers][n_agents][chunk_len][n_q_heads][head_dim]. chunk_len = 0 disables it; it cannot be
     * combined with a suffix. At most 16 query heads per kv head. */
    const void* chunk_k;
    const void* chunk_v;
    int64_t chunk_len;
} polykv_attend_ext;

/* Workspace bytes for polykv_attend_ex with these arguments (ext may be NULL). */
POLYKV_API polykv_status polykv_attend_ex_workspace_size(const polykv_pool* pool, int32_t n_agents, int32_t n_q_heads,
                                                         int64_t n_ctx, const polykv_attend_ext* ext, size_t* bytes);

/* polykv_attend with extensions. In chunk mode the output for query token c of agent a is
 *   out[l][a][c][hq] = sum over pool tokens t < n_ctx and chunk tokens c' <= c of softmax(scale * q.k) v
 * (the agent's chunk keys/values used as given); E_UNSUPPORTED if a suffix is also given.
 * With a suffix the output is
 *   out[l][a][hq] = sum over pool tokens t < n_ctx and suffix tokens s of softmax(scale * q.k) v
 * where pool keys/values are dequantized as in polykv_attend and suffix keys/values are used as
 * given. Errors as polykv_attend, plus E_INVAL for a bad suffix and E_UNSUPPORTED for more than 16
 * query heads per kv head. ext may be NULL (then identical to polykv_attend). */
POLYKV_API polykv_status polykv_attend_ex(const polykv_pool* pool, const void* q, float* out, int32_t n_agents,
                                          int32_t n_q_heads, int64_t n_ctx, float softmax_scale,
                                          const polykv_attend_ext* ext, void* workspace, size_t workspace_bytes,
                                          void* stream);

/* polykv_attend without a caller workspace (an addition of this library; the paper has no
 * counterpart). For callers that cannot allocate device memory when they attend -- code running
 * while a CUDA graph is captured elsewhere in the process, embeddings without an allocator, or
 * hosts with a fixed memory budget -- the split partials go to a 16 MiB array that is part of the
 * library's device module (held on every GPU that loads the library until the process exits).
 * Arguments and output are those of polykv_attend; nothing is allocated. Arguments that would
 * need more than 16 MiB of partials return POLYKV_E_BUFFER_TOO_SMALL with a message (the
 * Llama-3-8B shape with 15 agents needs about 12.7 MB on a 152-SM GB300, at any context length:
 * the partials grow with the SM count and the number of kv-head units, not with n_ctx).
 * The first call in a CUDA context looks up the array's device address (cudaGetSymbolAddress)
 * and caches it with the context's unique id; a call in another context looks it up again. The
 * cached address does not survive cudaDeviceReset: the next call (in the new primary context)
 * makes a fresh lookup. Make the first call in a context before any stream capture. All calls share the one array:
 * calls that may overlap on the GPU (other streams, other host threads) race on it and must be
 * ordered by the caller. The array keeps the last call's partials; every call writes each slot it
 * reads, so nothing needs clearing between calls. */
POLYKV_API polykv_status polykv_attend_static_ws(const polykv_pool* pool, const void* q, float* out,
                                                 int32_t n_agents, int32_t n_q_heads, int64_t n_ctx,
                                                 float softmax_scale, void* stream);

/* Read and clear the pool's device status word (synchronises `stream`).
 * Bit 0: a kernel gave up on a bounded device-side wait (about 2 s) and its
 * results are invalid; the call then returns POLYKV_E_TIMEOUT. *flags gets the
 * raw word. The word is cleared by the first encode into the pool.
 * Errors: E_INVAL, E_CUDA, E_TIMEOUT. */
POLYKV_API polykv_status polykv_pool_status(const polykv_pool* pool, void* stream, uint32_t* flags);

/* Release a handle (host memory only; dev_buf stays the caller's). NULL is OK. */
POLYKV_API polykv_status polykv_free(polykv_pool* pool);

/* The fp32 codebook embedded in the library: 8 ascending Lloyd-Max centroids
 * for N(0,1) and the 7 decision boundaries (c_i + c_{i+1}) * 0.5 in fp32.
 * Host only; either pointer may be NULL. */
POLYKV_API polykv_status polykv_codebook(float centroids[8], float boundaries[7]);

/* Message for the last failed call on this host thread ("" if none). */
POLYKV_API const char* polykv_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* POLYKV_H */

// C ABI of libpolykv: argument validation, pool layout, dispatch to kernels.
// Host code only. The operations are those of "PolyKV: A Shared
// Asymmetrically-Compressed KV Cache Pool for Multi-Agent LLM Inference"
// (abstract): write one compressed pool once, let N agents attend over it.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "polykv_internal.cuh"

struct polykv_pool {
    polykv_pool_desc desc;
    polykv::PoolView view;
    polykv_pool_regions regions;
    int64_t encoded;  // tokens [0, encoded) hold encoded data (as issued)
};

namespace polykv {

static thread_local char g_err[512] = "";

polykv_status set_error(polykv_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static polykv_status compute_regions(const polykv_pool_desc* d, polykv_pool_regions* r) {
    if (!d) return set_error(POLYKV_E_INVAL, "desc is NULL");
    if (d->n_layers <= 0 || d->n_kv_heads <= 0 || d->capacity_tokens <= 0)
        return set_error(POLYKV_E_INVAL, "n_layers, n_kv_heads and capacity_tokens must be positive");
    if (d->in_dtype != POLYKV_F16 && d->in_dtype != POLYKV_BF16)
        return set_error(POLYKV_E_INVAL, "in_dtype must be POLYKV_F16 or POLYKV_BF16");
    if (d->head_dim != 64 && d->head_dim != 128)
        return set_error(POLYKV_E_UNSUPPORTED, "head_dim %d (supported: 64, 128)", d->head_dim);
    if (d->capacity_tokens > ((int64_t)1 << 40)) return set_error(POLYKV_E_INVAL, "capacity_tokens too large");
    const int64_t cap = (d->capacity_tokens + kTokenAlign - 1) / kTokenAlign * kTokenAlign;
    const size_t units = (size_t)d->n_layers * (size_t)d->n_kv_heads;
    const size_t hd = (size_t)d->head_dim;
    const size_t toks = units * (size_t)cap;
    size_t off = 0;
    r->capacity_rounded = cap;
    r->status_off = off;
    r->v_nmax_off = off + 256;
    off = align_up(off + 256 + units * sizeof(float), 256);
    r->header_bytes = off;
    r->k_codes_off = off;
    off = align_up(off + toks * hd, 256);
    r->k_scales_off = off;
    off = align_up(off + toks * (hd / kQ8Block) * 2, 256);
    r->v_codes_off = off;
    off = align_up(off + toks * (3 * hd / 8), 256);
    r->v_norms_off = off;
    off = align_up(off + toks * 2, 256);
    r->total_bytes = off;
    return POLYKV_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Which attention kernel serves a call: the warp-level kernel when a kv head
// has few query rows (head_dim 64 with up to 16, 128 with up to 8), the
// tensor-core kernel for head_dim 128 and more rows, the CUDA-core kernel
// otherwise. The environment variable POLYKV_ATTEND_PATH=simt|tc|warp
// overrides (tc and warp only where supported) so the paths can be checked
// against each other on the same shapes.
enum class AttendPath { Simt, Tc, Warp };

static AttendPath attend_path(const PoolView& p, int rows) {
    const bool tc_ok = attend_tc_supported(p, rows);
    const bool warp_ok = attend_warp_supported(p, rows);
    const char* e = getenv("POLYKV_ATTEND_PATH");
    if (e && strcmp(e, "simt") == 0) return AttendPath::Simt;
    if (e && strcmp(e, "tc") == 0 && tc_ok) return AttendPath::Tc;
    if (e && strcmp(e, "warp") == 0 && warp_ok) return AttendPath::Warp;
    if (warp_ok) return AttendPath::Warp;
    return tc_ok ? AttendPath::Tc : AttendPath::Simt;
}

static size_t attend_workspace(const PoolView& p, int rows, int64_t n_ctx) {
    switch (attend_path(p, rows)) {
        case AttendPath::Warp: return attend_warp_workspace(p, rows, n_ctx);
        case AttendPath::Tc: return attend_tc_workspace(p, rows, n_ctx);
        default: return attend_simt_workspace(p, rows, n_ctx);
    }
}

static polykv_status launch_pool_attend(const PoolView& p, polykv_dtype dt, const void* q, float* out, int n_agents,
                                        int n_q_heads, int64_t n_ctx, float scale, void* ws, size_t ws_bytes,
                                        cudaStream_t st, const SuffixArgs* sfx = nullptr) {
    const int rows = n_agents * (n_q_heads / p.H);
    switch (attend_path(p, rows)) {
        case AttendPath::Warp:
            return launch_attend_warp(p, dt, q, out, n_agents, n_q_heads, n_ctx, scale, ws, ws_bytes, st, sfx);
        case AttendPath::Tc:
            return launch_attend_tc(p, dt, q, out, n_agents, n_q_heads, n_ctx, scale, ws, ws_bytes, st, sfx);
        default:
            return launch_attend_simt(p, dt, q, out, n_agents, n_q_heads, n_ctx, scale, ws, ws_bytes, st, sfx);
    }
}

}  // namespace polykv

using namespace polykv;

extern "C" {

polykv_status polykv_pool_create(const polykv_pool_desc* desc, void* dev_buf, size_t dev_buf_bytes,
                                 polykv_pool** out, size_t* required_bytes) {
    polykv_pool_regions r;
    const polykv_status st = compute_regions(desc, &r);
    if (st != POLYKV_OK) return st;
    if (required_bytes) *required_bytes = r.total_bytes;
    if (!dev_buf) return POLYKV_OK;  // query mode
    if (!out) return set_error(POLYKV_E_INVAL, "out is NULL");
    if ((reinterpret_cast<uintptr_t>(dev_buf) & 255u) != 0)
        return set_error(POLYKV_E_INVAL, "dev_buf must be 256-byte aligned");
    if (dev_buf_bytes < r.total_bytes)
        return set_error(POLYKV_E_BUFFER_TOO_SMALL, "dev_buf has %zu bytes, pool needs %zu", dev_buf_bytes,
                         r.total_bytes);
    polykv_pool* p = new (std::nothrow) polykv_pool;
    if (!p) return set_error(POLYKV_E_INVAL, "host allocation failed");
    p->desc = *desc;
    p->regions = r;
    p->encoded = 0;
    char* base = static_cast<char*>(dev_buf);
    p->view.kq = reinterpret_cast<int8_t*>(base + r.k_codes_off);
    p->view.ks = reinterpret_cast<__half*>(base + r.k_scales_off);
    p->view.vc = reinterpret_cast<uint8_t*>(base + r.v_codes_off);
    p->view.vn = reinterpret_cast<__half*>(base + r.v_norms_off);
    p->view.status = reinterpret_cast<uint32_t*>(base + r.status_off);
    p->view.nmax = reinterpret_cast<float*>(base + r.v_nmax_off);
    p->view.L = desc->n_layers;
    p->view.H = desc->n_kv_heads;
    p->view.d = desc->head_dim;
    p->view.cap = r.capacity_rounded;
    *out = p;
    g_err[0] = 0;
    return POLYKV_OK;
}

polykv_status polykv_pool_get_regions(const polykv_pool* pool, polykv_pool_regions* out) {
    if (!pool || !out) return set_error(POLYKV_E_INVAL, "pool and out must be non-NULL");
    *out = pool->regions;
    return POLYKV_OK;
}

polykv_status polykv_encode(polykv_pool* pool, const void* k, const void* v, int64_t t0, int64_t n_tokens,
                            void* stream) {
    if (!pool) return set_error(POLYKV_E_INVAL, "pool is NULL");
    if (n_tokens < 0 || t0 < 0) return set_error(POLYKV_E_INVAL, "t0 and n_tokens must be >= 0");
    if (t0 + n_tokens > pool->desc.capacity_tokens)
        return set_error(POLYKV_E_INVAL, "t0 + n_tokens = %lld exceeds capacity %lld", (long long)(t0 + n_tokens),
                         (long long)pool->desc.capacity_tokens);
    if (t0 > pool->encoded)
        return set_error(POLYKV_E_STATE, "t0 = %lld leaves a gap after the %lld encoded tokens", (long long)t0,
                         (long long)pool->encoded);
    if (n_tokens == 0) return POLYKV_OK;
    if (!k || !v) return set_error(POLYKV_E_INVAL, "k and v must be non-NULL");
    if (!aligned16(k) || !aligned16(v)) return set_error(POLYKV_E_INVAL, "k and v must be 16-byte aligned");
    if (pool->encoded == 0) {
        // first write into this pool: clear the header (status word, per-unit norm maxima)
        const cudaError_t e = cudaMemsetAsync(pool->view.status, 0, pool->regions.header_bytes - pool->regions.status_off,
                                              static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "encode: header clear: %s", cudaGetErrorString(e));
    }
    const polykv_status st =
        launch_encode(pool->view, pool->desc.in_dtype, k, v, t0, n_tokens, static_cast<cudaStream_t>(stream));
    if (st != POLYKV_OK) return st;
    if (t0 + n_tokens > pool->encoded) pool->encoded = t0 + n_tokens;
    return POLYKV_OK;
}

static polykv_status check_attend_args(const polykv_pool* pool, int32_t n_agents, int32_t n_q_heads, int64_t n_ctx) {
    if (!pool) return set_error(POLYKV_E_INVAL, "pool is NULL");
    if (n_agents < 1) return set_error(POLYKV_E_INVAL, "n_agents must be >= 1");
    if (n_q_heads < 1 || n_q_heads % pool->desc.n_kv_heads != 0)
        return set_error(POLYKV_E_INVAL, "n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)", n_q_heads,
                         pool->desc.n_kv_heads);
    if (n_ctx < 1) return set_error(POLYKV_E_INVAL, "n_ctx must be >= 1");
    if (n_ctx > pool->encoded)
        return set_error(POLYKV_E_STATE, "n_ctx = %lld exceeds the %lld encoded tokens", (long long)n_ctx,
                         (long long)pool->encoded);
    if ((int64_t)n_agents * (n_q_heads / pool->desc.n_kv_heads) > (1 << 20))
        return set_error(POLYKV_E_UNSUPPORTED, "too many query rows per kv head");
    return POLYKV_OK;
}

polykv_status polykv_attend_workspace_size(const polykv_pool* pool, int32_t n_agents, int32_t n_q_heads,
                                           int64_t n_ctx, size_t* bytes) {
    const polykv_status st = check_attend_args(pool, n_agents, n_q_heads, n_ctx);
    if (st != POLYKV_OK) return st;
    if (!bytes) return set_error(POLYKV_E_INVAL, "bytes is NULL");
    const int rows = n_agents * (n_q_heads / pool->desc.n_kv_heads);
    *bytes = attend_workspace(pool->view, rows, n_ctx);
    return POLYKV_OK;
}

polykv_status polykv_attend(const polykv_pool* pool, const void* q, float* out, int32_t n_agents, int32_t n_q_heads,
                            int64_t n_ctx, float softmax_scale, void* workspace, size_t workspace_bytes,
                            void* stream) {
    const polykv_status st = check_attend_args(pool, n_agents, n_q_heads, n_ctx);
    if (st != POLYKV_OK) return st;
    if (!q || !out) return set_error(POLYKV_E_INVAL, "q and out must be non-NULL");
    if (!aligned16(q) || !aligned16(out) || (workspace && !aligned16(workspace)))
        return set_error(POLYKV_E_INVAL, "q, out and workspace must be 16-byte aligned");
    const int rows = n_agents * (n_q_heads / pool->desc.n_kv_heads);
    const size_t need = attend_workspace(pool->view, rows, n_ctx);
    if (need > 0 && !workspace) return set_error(POLYKV_E_INVAL, "workspace is NULL but %zu bytes are needed", need);
    const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)pool->desc.head_dim);
    return launch_pool_attend(pool->view, pool->desc.in_dtype, q, out, n_agents, n_q_heads, n_ctx, scale, workspace,
                              workspace_bytes, static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------------------------
// Attention without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run attention: code that
// runs while a CUDA graph is being captured elsewhere in the process, allocator-less embedding
// layers, or hosts whose memory budget is fixed up front. For them the split partials live in a
// file-scope device array instead. The array is part of the library's module, so every GPU that
// loads the library holds it until the process exits; its size is therefore kept modest and
// fixed: 16 MiB, enough for the Llama-3-8B shape (32 layers x 8 kv heads, 15 agents x 4 query
// heads, any context length on a 152-SM GB300: about 12.7 MB).
namespace polykv {
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_attend_scratch[kStaticScratchBytes];
struct ScratchAddr {
    unsigned long long ctx_id;   // unique id of the context the address was looked up in (0: none)
    void* ptr;
};
static ScratchAddr g_scratch_addr[128] = {};
static std::mutex g_scratch_mu;

// Unique id of the calling thread's current CUDA context (0 if none), via cuCtxGetCurrent and
// cuCtxGetId from the driver, looked up once (no link-time dependency on libcuda). Ids, unlike
// context handles, are never reused within a process.
static polykv_status current_ctx_id(unsigned long long* id) {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_cur || !get_id) return set_error(POLYKV_E_CUDA, "attend_static: cuCtxGetCurrent/cuCtxGetId not available");
    CUcontext ctx = nullptr;
    if (get_cur(&ctx) != CUDA_SUCCESS) return set_error(POLYKV_E_CUDA, "attend_static: cuCtxGetCurrent failed");
    *id = 0;
    if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return set_error(POLYKV_E_CUDA, "attend_static: cuCtxGetId failed");
    return POLYKV_OK;
}

// Device address of the scratch array in the current device's current context. Host code only
// sees a host-side stand-in for the symbol, so the address is looked up on the first call in a
// context and cached with that context's id. A call made in another context (the primary context
// re-created after cudaDeviceReset, or a context the caller made current) looks it up again: the
// module, and so the array, is loaded anew in every context.
static polykv_status static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "attend_static: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 128) return set_error(POLYKV_E_UNSUPPORTED, "attend_static: device %d", dev);
    unsigned long long id = 0;
    polykv_status st = current_ctx_id(&id);
    if (st != POLYKV_OK) return st;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr& a = g_scratch_addr[dev];
    if (id == 0 || !a.ptr || a.ctx_id != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attend_scratch);   // makes the primary context current if none is
        if (e != cudaSuccess || !p)
            return set_error(POLYKV_E_CUDA, "attend_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        if (id == 0) {
            st = current_ctx_id(&id);
            if (st != POLYKV_OK) return st;
            if (id == 0) return set_error(POLYKV_E_CUDA, "attend_static: no current CUDA context");
        }
        a.ctx_id = id;
        a.ptr = p;
    }
    *out = a.ptr;
    return POLYKV_OK;
}
}  // namespace polykv

polykv_status polykv_attend_static_ws(const polykv_pool* pool, const void* q, float* out, int32_t n_agents,
                                      int32_t n_q_heads, int64_t n_ctx, float softmax_scale, void* stream) {
    const polykv_status st = check_attend_args(pool, n_agents, n_q_heads, n_ctx);
    if (st != POLYKV_OK) return st;
    if (!q || !out) return set_error(POLYKV_E_INVAL, "q and out must be non-NULL");
    if (!aligned16(q) || !aligned16(out)) return set_error(POLYKV_E_INVAL, "q and out must be 16-byte aligned");
    const int rows = n_agents * (n_q_heads / pool->desc.n_kv_heads);
    const size_t need = attend_workspace(pool->view, rows, n_ctx);
    if (need > kStaticScratchBytes)
        return set_error(POLYKV_E_BUFFER_TOO_SMALL,
                         "attend_static: these arguments need %zu bytes of scratch, the built-in array holds %zu; "
                         "use polykv_attend with a caller workspace",
                         need, kStaticScratchBytes);
    void* ws = nullptr;
    const polykv_status s2 = static_scratch(&ws);
    if (s2 != POLYKV_OK) return s2;
    const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)pool->desc.head_dim);
    return launch_pool_attend(pool->view, pool->desc.in_dtype, q, out, n_agents, n_q_heads, n_ctx, scale, ws,
                              kStaticScratchBytes, static_cast<cudaStream_t>(stream));
}

polykv_status polykv_pool_status(const polykv_pool* pool, void* stream, uint32_t* flags) {
    if (!pool || !flags) return set_error(POLYKV_E_INVAL, "pool and flags must be non-NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, pool->view.status, sizeof(h), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(pool->view.status, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "status read: %s", cudaGetErrorString(e));
    *flags = h;
    if (h & 1u) return set_error(POLYKV_E_TIMEOUT, "a kernel gave up waiting on a bounded device-side wait");
    return POLYKV_OK;
}

static size_t suffix_bytes(const polykv_pool* pool, int32_t n_agents, int32_t n_q_heads) {
    const size_t rows = (size_t)pool->desc.n_layers * (size_t)n_agents * (size_t)n_q_heads;
    return sizeof(float) * rows * ((size_t)pool->desc.head_dim + 2);
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Query-chunk mode runs the pool part with the chunk position folded into the agent index
// (agents x chunk_len "virtual agents", the same row layout as q [L][A][C][Hq][d]).
static polykv_status chunk_agents(const polykv_pool* pool, int32_t n_agents, int32_t n_q_heads,
                                  const polykv_attend_ext* ext, int64_t* agents) {
    if (ext->suffix_len != 0) return set_error(POLYKV_E_UNSUPPORTED, "chunk mode cannot be combined with a suffix");
    if (ext->chunk_len < 0) return set_error(POLYKV_E_INVAL, "chunk_len must be >= 0");
    const int64_t av = (int64_t)n_agents * ext->chunk_len;
    if (av * (n_q_heads / pool->desc.n_kv_heads) > (1 << 20))
        return set_error(POLYKV_E_UNSUPPORTED, "chunk mode: too many query rows per kv head");
    *agents = av;
    return POLYKV_OK;
}

polykv_status polykv_attend_ex_workspace_size(const polykv_pool* pool, int32_t n_agents, int32_t n_q_heads,
                                              int64_t n_ctx, const polykv_attend_ext* ext, size_t* bytes) {
    const polykv_status st = check_attend_args(pool, n_agents, n_q_heads, n_ctx);
    if (st != POLYKV_OK) return st;
    if (!bytes) return set_error(POLYKV_E_INVAL, "bytes is NULL");
    int64_t agents = n_agents;
    if (ext && ext->chunk_len != 0) {
        const polykv_status cs = chunk_agents(pool, n_agents, n_q_heads, ext, &agents);
        if (cs != POLYKV_OK) return cs;
    }
    const int rows = (int)(agents * (n_q_heads / pool->desc.n_kv_heads));
    size_t b = attend_workspace(pool->view, rows, n_ctx);
    if (ext && (ext->suffix_len > 0 || ext->chunk_len > 0)) b = align256(b) + suffix_bytes(pool, (int32_t)agents, n_q_heads);
    *bytes = b;
    return POLYKV_OK;
}

polykv_status polykv_attend_ex(const polykv_pool* pool, const void* q, float* out, int32_t n_agents,
                               int32_t n_q_heads, int64_t n_ctx, float softmax_scale, const polykv_attend_ext* ext,
                               void* workspace, size_t workspace_bytes, void* stream) {
    if (!ext || (ext->suffix_len == 0 && ext->chunk_len == 0))
        return polykv_attend(pool, q, out, n_agents, n_q_heads, n_ctx, softmax_scale, workspace, workspace_bytes,
                             stream);
    const polykv_status st = check_attend_args(pool, n_agents, n_q_heads, n_ctx);
    if (st != POLYKV_OK) return st;
    if (ext->chunk_len != 0) {
        int64_t av = 0;
        const polykv_status cs = chunk_agents(pool, n_agents, n_q_heads, ext, &av);
        if (cs != POLYKV_OK) return cs;
        if (!q || !out || !workspace) return set_error(POLYKV_E_INVAL, "q, out and workspace must be non-NULL");
        if (!aligned16(q) || !aligned16(out) || !aligned16(workspace))
            return set_error(POLYKV_E_INVAL, "q, out and workspace must be 16-byte aligned");
        if (!ext->chunk_k || !ext->chunk_v || !aligned16(ext->chunk_k) || !aligned16(ext->chunk_v))
            return set_error(POLYKV_E_INVAL, "chunk_k and chunk_v must be non-NULL and 16-byte aligned");
        if (n_q_heads / pool->desc.n_kv_heads > 16)
            return set_error(POLYKV_E_UNSUPPORTED, "chunk: more than 16 query heads per kv head");
        const int rows = (int)(av * (n_q_heads / pool->desc.n_kv_heads));
        const size_t pool_ws = attend_workspace(pool->view, rows, n_ctx);
        const size_t need = align256(pool_ws) + suffix_bytes(pool, (int32_t)av, n_q_heads);
        if (workspace_bytes < need)
            return set_error(POLYKV_E_BUFFER_TOO_SMALL, "attend_ex: workspace %zu < %zu bytes", workspace_bytes, need);
        const size_t nrows = (size_t)pool->desc.n_layers * (size_t)av * (size_t)n_q_heads;
        SuffixArgs chk;
        chk.q = q;
        chk.k = ext->chunk_k;
        chk.v = ext->chunk_v;
        chk.len = ext->chunk_len;
        chk.chunk = ext->chunk_len;
        chk.acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(pool_ws));
        chk.ml = chk.acc + nrows * (size_t)pool->desc.head_dim;
        const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)pool->desc.head_dim);
        return launch_pool_attend(pool->view, pool->desc.in_dtype, q, out, (int)av, n_q_heads, n_ctx, scale,
                                  workspace, pool_ws, static_cast<cudaStream_t>(stream), &chk);
    }
    if (!q || !out || !workspace) return set_error(POLYKV_E_INVAL, "q, out and workspace must be non-NULL");
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace))
        return set_error(POLYKV_E_INVAL, "q, out and workspace must be 16-byte aligned");
    if (ext->suffix_len < 0) return set_error(POLYKV_E_INVAL, "suffix_len must be >= 0");
    if (!ext->suffix_k || !ext->suffix_v || !aligned16(ext->suffix_k) || !aligned16(ext->suffix_v))
        return set_error(POLYKV_E_INVAL, "suffix_k and suffix_v must be non-NULL and 16-byte aligned");
    if (n_q_heads / pool->desc.n_kv_heads > 16)
        return set_error(POLYKV_E_UNSUPPORTED, "suffix: more than 16 query heads per kv head");
    const int rows = n_agents * (n_q_heads / pool->desc.n_kv_heads);
    const size_t pool_ws = attend_workspace(pool->view, rows, n_ctx);
    const size_t need = align256(pool_ws) + suffix_bytes(pool, n_agents, n_q_heads);
    if (workspace_bytes < need)
        return set_error(POLYKV_E_BUFFER_TOO_SMALL, "attend_ex: workspace %zu < %zu bytes", workspace_bytes, need);
    const size_t nrows = (size_t)pool->desc.n_layers * (size_t)n_agents * (size_t)n_q_heads;
    SuffixArgs sfx;
    sfx.q = q;
    sfx.k = ext->suffix_k;
    sfx.v = ext->suffix_v;
    sfx.len = ext->suffix_len;
    sfx.acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(pool_ws));
    sfx.ml = sfx.acc + nrows * (size_t)pool->desc.head_dim;
    const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / sqrtf((float)pool->desc.head_dim);
    return launch_pool_attend(pool->view, pool->desc.in_dtype, q, out, n_agents, n_q_heads, n_ctx, scale, workspace,
                              pool_ws, static_cast<cudaStream_t>(stream), &sfx);
}

polykv_status polykv_free(polykv_pool* pool) {
    delete pool;
    return POLYKV_OK;
}

polykv_status polykv_codebook(float centroids[8], float boundaries[7]) {
    if (centroids)
        for (int i = 0; i < 8; ++i) centroids[i] = centroid_of(i);
    if (boundaries) {
        const float b[7] = {-kB6, -kB5, -kB4, 0.0f, kB4, kB5, kB6};
        for (int i = 0; i < 7; ++i) boundaries[i] = b[i];
    }
    return POLYKV_OK;
}

const char* polykv_last_error(void) { return g_err; }

}  // extern "C"

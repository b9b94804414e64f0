// Internal definitions shared by the libpolykv translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "polykv.h"

namespace polykv {

// SM count of the current device (read per call: cheap, and right for every device of a process)
inline int device_sm_count() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    return v;
}

constexpr int kQ8Block = 32;       // q8_0 block length along head_dim
constexpr int kTokenAlign = 128;   // pool capacity is rounded to this many tokens

// 8-level Lloyd-Max quantizer for a unit Gaussian (Max 1960; the N(0,1)
// codebook named in the PolyKV abstract), centroids rounded to fp32.
constexpr float kC4 = 0.245094178944f;
constexpr float kC5 = 0.756005281206f;
constexpr float kC6 = 1.343909278505f;
constexpr float kC7 = 2.151945704537f;
// decision boundaries: midpoints formed in fp32 from the fp32 centroids
constexpr float kB4 = (kC4 + kC5) * 0.5f;
constexpr float kB5 = (kC5 + kC6) * 0.5f;
constexpr float kB6 = (kC6 + kC7) * 0.5f;

// Device view of a pool laid out in one caller buffer.
struct PoolView {
    int8_t* kq;        // [U][cap][d]
    __half* ks;        // [U][cap][d/32]
    uint8_t* vc;       // [U][cap/32][d][12]: per 32-token group and coordinate, one 12-byte code string
    __half* vn;        // [U][cap]
    uint32_t* status;  // status word (bit 0: a bounded device wait gave up)
    float* nmax;       // [U] running maximum of ||v|| per unit
    int L, H, d;
    int64_t cap;
};

polykv_status set_error(polykv_status st, const char* fmt, ...);

polykv_status launch_encode(const PoolView& p, polykv_dtype dt, const void* k, const void* v, int64_t t0,
                            int64_t n_tokens, cudaStream_t stream);

// Private per-agent suffix (uncompressed keys/values [L][A][H][len][d]) and its partials
// (acc [L][A][Hq][d] in the original basis, (m, l) [L][A][Hq][2]).
struct SuffixArgs {
    const void* q;
    const void* k;
    const void* v;
    int64_t len;
    float* acc;
    float* ml;
    int64_t chunk = 0;   // > 0: query-chunk mode (len = chunk, causal; the attend's n_agents counts agents x chunk)
};
polykv_status launch_attend_suffix(const SuffixArgs& a, polykv_dtype dt, int L, int A, int H, int Hq, int D,
                                   float scale, cudaStream_t st);

// number of token splits used by the CUDA-core attention path
int attend_simt_splits(const PoolView& p, int rows, int64_t n_ctx);
size_t attend_simt_workspace(const PoolView& p, int rows, int64_t n_ctx);
polykv_status launch_attend_simt(const PoolView& p, polykv_dtype dt, const void* q, float* out, int n_agents,
                                 int n_q_heads, int64_t n_ctx, float scale, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, const SuffixArgs* sfx = nullptr);

// Where the pool partials are. nc == 0: CUDA-core splits, slot = unit * n_slots + split, R rows
// per slot. nc > 0: the tensor-core partition of (segment = unit x row group, tile) over nc CTAs,
// slot = segment + CTA, RS rows per slot, nrg row groups of 64 rows per unit.
struct MergeLayout {
    int nrg = 1, RS = 0;
    int64_t nt = 0, tt = 0;
    int nc = 0;
};
polykv_status launch_attend_merge(const float* ws_acc, const float* ws_ml, float* out, int U, int H, int A, int Hq,
                                  int R, int n_slots, const MergeLayout& ml, int D, cudaStream_t st,
                                  const float* sfx_acc = nullptr, const float* sfx_ml = nullptr);

// tensor-core attention path (head_dim 128, any row count in groups of 64 rows per kv head)
bool attend_tc_supported(const PoolView& p, int rows);
size_t attend_tc_workspace(const PoolView& p, int rows, int64_t n_ctx);
polykv_status launch_attend_tc(const PoolView& p, polykv_dtype dt, const void* q, float* out, int n_agents,
                               int n_q_heads, int64_t n_ctx, float scale, void* ws, size_t ws_bytes,
                               cudaStream_t stream, const SuffixArgs* sfx = nullptr);

// warp-level attention path for few rows per kv head (head_dim 64 with up to 16 rows, 128 with up to 8)
bool attend_warp_supported(const PoolView& p, int rows);
size_t attend_warp_workspace(const PoolView& p, int rows, int64_t n_ctx);
polykv_status launch_attend_warp(const PoolView& p, polykv_dtype dt, const void* q, float* out, int n_agents,
                                 int n_q_heads, int64_t n_ctx, float scale, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, const SuffixArgs* sfx = nullptr);

__host__ __device__ inline float centroid_of(int code) {
    // ascending codes 0..7 -> -c7 .. -c4, c4 .. c7
    const float mag[4] = {kC4, kC5, kC6, kC7};
    return code >= 4 ? mag[code - 4] : -mag[3 - code];
}

}  // namespace polykv

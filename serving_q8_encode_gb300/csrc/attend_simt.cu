// Multi-agent decode attention over the shared pool on CUDA cores (any number
// of query rows; the general path and the one used when few rows share a kv
// head).
//
// PolyKV abstract ("PolyKV: A Shared Asymmetrically-Compressed KV Cache Pool
// for Multi-Agent LLM Inference"): N agents read one compressed pool. Each
// CTA owns one (layer, kv head, token split) and ALL query rows that read
// that kv head (agents x GQA group), so every pool byte is fetched once per
// split for all agents. Keys are dequantized in registers (int8 code times
// the block's fp16 scale, applied to the 32-wide partial dot product); the
// online softmax runs in base 2; values are accumulated in the ROTATED basis
// as (p * ||v||) * centroid[code]. Because the inverse transform is linear, the
// merge kernel applies one inverse FWHT per output row instead of one per
// value vector:  o = (1/d) H (sum_t p_t n_t C[code_t]) / sum_t p_t.
#include <algorithm>
#include <cmath>

#include "polykv_internal.cuh"
#include "merge_row.cuh"

namespace polykv {
namespace {

constexpr int kTT = 64;        // tokens per tile
constexpr int kThreads = 128;
constexpr int kMaxRowsPerCta = 64;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float centroid_signed(uint32_t code) {
    const uint32_t idx = code >= 4 ? code - 4 : 3 - code;
    const float m = idx == 0 ? kC4 : (idx == 1 ? kC5 : (idx == 2 ? kC6 : kC7));
    return code >= 4 ? m : -m;
}

__device__ __forceinline__ float q_to_float(uint16_t bits, bool bf16) {
    return bf16 ? __uint_as_float((uint32_t)bits << 16) : __half2float(__ushort_as_half(bits));
}

template <int D, int RMAX>
struct SimtSmem {
    static constexpr int kQs = D * RMAX;            // [D][RMAX]
    static constexpr int kSc = RMAX * (kTT + 1);    // [RMAX][kTT+1]
    static constexpr int kVh = kTT * (D + 4);       // [kTT][D+4]
    static constexpr int kFloats = kQs + kSc + kVh + 3 * RMAX + kTT;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

// grid: (split, unit = layer*H + kv_head, row chunk); block: 128 threads.
template <int D, int RMAX, bool BF16>
__global__ void __launch_bounds__(kThreads) attend_partial_simt(PoolView p, const uint16_t* __restrict__ q, int A,
                                                                int Hq, int R, int64_t n_ctx, int64_t split_len,
                                                                int n_splits, float scale_log2, float* __restrict__ ws_acc,
                                                                float* __restrict__ ws_ml) {
    using S = SimtSmem<D, RMAX>;
    extern __shared__ float4 smem4[];
    float* smem = reinterpret_cast<float*>(smem4);
    float* qs = smem;                 // [D][RMAX]
    float* sc = qs + S::kQs;          // [RMAX][kTT+1]
    float* vh = sc + S::kSc;          // [kTT][D+4]
    float* m_s = vh + S::kVh;
    float* l_s = m_s + RMAX;
    float* al_s = l_s + RMAX;
    float* nvs = al_s + RMAX;         // [kTT] norms of the tile's tokens (0 past the split)

    const int tid = threadIdx.x;
    const int split = blockIdx.x;
    const int unit = blockIdx.y;
    const int row0 = blockIdx.z * RMAX;
    const int nrows = min(RMAX, R - row0);
    const int layer = unit / p.H, kvh = unit % p.H;
    const int G = Hq / p.H;

    // ---- query rows of this kv head, transposed to [j][r], fp32
    for (int i = tid; i < D * RMAX; i += kThreads) {
        const int r = i / D, j = i % D;
        float val = 0.0f;
        if (r < nrows) {
            const int gr = row0 + r;
            const int a = gr / G, g = gr % G;
            val = q_to_float(q[(((int64_t)layer * A + a) * Hq + kvh * G + g) * D + j], BF16);
        }
        qs[j * RMAX + r] = val;
    }
    if (tid < RMAX) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.0f;
    }

    const int64_t t_begin = (int64_t)split * split_len;
    const int64_t t_end = (t_begin + split_len < n_ctx) ? t_begin + split_len : n_ctx;
    const int64_t ubase = (int64_t)unit * p.cap;

    // PV mapping: column quad cq, row group rg
    constexpr int NCQ = D / 4;
    constexpr int NRG = kThreads / NCQ;
    constexpr int ROWS = (RMAX + NRG - 1) / NRG;
    const int cq = tid % NCQ, rg = tid / NCQ;
    float acc[ROWS][4];
#pragma unroll
    for (int i = 0; i < ROWS; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = 0.0f;

    __syncthreads();

    for (int64_t tile = t_begin; tile < t_end; tile += kTT) {
        // ---- A: scores, thread = (token, row half)
        {
            constexpr int RH = RMAX / 2;
            const int t = tid % kTT, rh = tid / kTT;
            const int64_t tok = tile + t;
            const bool valid = tok < t_end;
            float score[RH];
#pragma unroll
            for (int i = 0; i < RH; ++i) score[i] = 0.0f;
            if (valid) {
                const uint4* krow = reinterpret_cast<const uint4*>(p.kq + (ubase + tok) * D);
                const __half* srow = p.ks + (ubase + tok) * (D / kQ8Block);
#pragma unroll
                for (int b = 0; b < D / kQ8Block; ++b) {
                    float part[RH];
#pragma unroll
                    for (int i = 0; i < RH; ++i) part[i] = 0.0f;
#pragma unroll
                    for (int w16 = 0; w16 < 2; ++w16) {
                        const uint4 kr = krow[b * 2 + w16];
                        const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float kf = (float)(int8_t)((kw[e >> 2] >> (8 * (e & 3))) & 0xFF);
                            const int j = b * 32 + w16 * 16 + e;
                            const float* qj = qs + j * RMAX + rh * RH;
#pragma unroll
                            for (int i = 0; i < RH; i += 4) {
                                const float4 q4 = *reinterpret_cast<const float4*>(qj + i);
                                part[i] = fmaf(q4.x, kf, part[i]);
                                part[i + 1] = fmaf(q4.y, kf, part[i + 1]);
                                part[i + 2] = fmaf(q4.z, kf, part[i + 2]);
                                part[i + 3] = fmaf(q4.w, kf, part[i + 3]);
                            }
                        }
                    }
                    const float sb = __half2float(srow[b]);
#pragma unroll
                    for (int i = 0; i < RH; ++i) score[i] = fmaf(sb, part[i], score[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < RH; ++i) {
                const int r = rh * RH + i;
                if (r < nrows) sc[r * (kTT + 1) + t] = valid ? score[i] * scale_log2 : -INFINITY;
            }
        }
        // ---- C: centroids of the value tile in the rotated basis, vh[t][j] = C[code]; each token's
        // norm is applied to its probability in B. The tile (64 tokens, 64-aligned) is two 32-token
        // groups of the pool, one 12-byte string per (group, coordinate).
        {
            if (tid < kTT) {
                const int64_t tok = tile + tid;
                nvs[tid] = tok < t_end ? __half2float(p.vn[ubase + tok]) : 0.0f;
            }
            const int64_t gbase = (ubase + tile) / 32;
            for (int it = tid; it < 2 * D; it += kThreads) {
                const int h = it / D, j = it % D;
                const uint32_t* src = reinterpret_cast<const uint32_t*>(p.vc + ((gbase + h) * D + j) * 12);
                const uint32_t w[3] = {src[0], src[1], src[2]};
                float* col = vh + (32 * h) * (D + 4) + j;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int bit = 3 * k, wi = bit >> 5, off = bit & 31;
                    uint32_t c = w[wi] >> off;
                    if (off > 29) c |= w[wi + 1] << (32 - off);
                    col[k * (D + 4)] = centroid_signed(c & 7u);
                }
            }
        }
        __syncthreads();
        // ---- B: online softmax per row (base 2), warp per row
        {
            const int warp = tid / 32, lane = tid % 32;
            for (int r = warp; r < nrows; r += kThreads / 32) {
                float* row = sc + r * (kTT + 1);
                const float x0 = row[lane], x1 = row[lane + 32];
                float mt = fmaxf(x0, x1);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                const float m_old = m_s[r];
                const float m_new = fmaxf(m_old, mt);
                float p0 = 0.f, p1 = 0.f, alpha = 1.f;
                if (m_new != -INFINITY) {
                    p0 = exp2f(x0 - m_new);
                    p1 = exp2f(x1 - m_new);
                    alpha = exp2f(m_old - m_new);
                }
                float sum = p0 + p1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                row[lane] = p0 * nvs[lane];   // the value operand carries no norm (see C)
                row[lane + 32] = p1 * nvs[lane + 32];
                if (lane == 0) {
                    l_s[r] = l_s[r] * alpha + sum;
                    m_s[r] = m_new;
                    al_s[r] = alpha;
                }
            }
        }
        __syncthreads();
        // ---- D: acc[r][:] = acc * alpha + sum_t p[r][t] * vh[t][:]
        {
#pragma unroll
            for (int i = 0; i < ROWS; ++i) {
                const int r = rg * ROWS + i;
                if (r < nrows) {
                    const float a = al_s[r];
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[i][c] *= a;
                }
            }
            const int tmax = (t_end - tile < kTT) ? (int)(t_end - tile) : kTT;
            for (int t = 0; t < tmax; ++t) {
                const float4 vv = reinterpret_cast<const float4*>(vh + t * (D + 4))[cq];
#pragma unroll
                for (int i = 0; i < ROWS; ++i) {
                    const int r = rg * ROWS + i;
                    if (r < nrows) {
                        const float pr = sc[r * (kTT + 1) + t];
                        acc[i][0] = fmaf(pr, vv.x, acc[i][0]);
                        acc[i][1] = fmaf(pr, vv.y, acc[i][1]);
                        acc[i][2] = fmaf(pr, vv.z, acc[i][2]);
                        acc[i][3] = fmaf(pr, vv.w, acc[i][3]);
                    }
                }
            }
        }
        __syncthreads();
    }

    // ---- partials: acc [U][S][R][D], (m, l) [U][S][R][2]
    const int64_t pbase = ((int64_t)unit * n_splits + split) * R;
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
        const int r = rg * ROWS + i;
        if (r < nrows)
            reinterpret_cast<float4*>(ws_acc + (pbase + row0 + r) * D)[cq] =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
    if (tid < nrows) {
        ws_ml[(pbase + row0 + tid) * 2] = m_s[tid];
        ws_ml[(pbase + row0 + tid) * 2 + 1] = l_s[tid];
    }
}

// One warp per (unit, row): log-sum-exp merge of the splits, normalisation,
// one inverse FWHT of the row (o = (1/d) H acc / l), fp32 output.
// Partials of unit u live in slots u*n_slots + k. With nc > 0 the slots come
// from a contiguous cut of the (unit, tile) list into nc ranges (tt tiles,
// nt per unit) and unit u has one piece per range that overlaps it;
// otherwise every unit has n_slots pieces.
//
// The kernel is bound by load latency (the partials were just written and
// sit in L2), so each lane issues the loads of up to kMergeBatch pieces, and
// of the suffix partial, before it uses any of them, with one vector load
// per piece, and folds each batch into a running maximum.
constexpr int kMergeBatch = 4;
constexpr int kMergeWarps = 8;

// First tile-range index overlapping tile position x of the (unit, tile) list
// cut into nc ranges of tt tiles: floor((x * nc - 1) / tt) for x >= 1. Uses
// 32-bit division when the product fits, which is the usual case.
__device__ __forceinline__ int64_t merge_range_of(int64_t x, int nc, int64_t tt) {
    const int64_t num = x * nc - 1;
    if (num <= 0xFFFFFFFFll && tt <= 0xFFFFFFFFll) return (int64_t)((uint32_t)num / (uint32_t)tt);
    return num / tt;
}

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) attend_merge(const float* __restrict__ ws_acc,
                                                                 const float* __restrict__ ws_ml,
                                                                 float* __restrict__ out, int U, int H, int A, int Hq,
                                                                 int R, int n_slots, MergeLayout lay,
                                                                 const float* __restrict__ sfx_acc,
                                                                 const float* __restrict__ sfx_ml) {
    constexpr int EPL = D / 32;  // elements per lane
    using V = MergeVec<D>;
    const int64_t wid = (int64_t)blockIdx.x * kMergeWarps + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    // launched as a programmatic dependent of the partial kernel: wait until its writes are visible
    // (a no-op for an ordinary launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (wid >= (int64_t)U * R) return;
    const int unit = (int)(wid / R), r = (int)(wid % R);
    const int G = Hq / H;
    const int layer = unit / H, kvh = unit % H;
    const int a = r / G, g = r % G;

    // partial rows of this output row: pr(s) = first + s * stride, s < pieces
    int pieces = n_slots;
    int64_t first = (int64_t)unit * n_slots * R + r, stride = R;
    if (lay.nc > 0) {
        const int64_t seg = (int64_t)unit * lay.nrg + r / lay.RS;
        const int64_t lo = merge_range_of(seg * lay.nt + 1, lay.nc, lay.tt);
        const int64_t hi = merge_range_of(seg * lay.nt + lay.nt, lay.nc, lay.tt);
        pieces = (int)(hi - lo + 1);
        first = (seg + lo) * lay.RS + r % lay.RS;
        stride = lay.RS;
    }
    const int64_t orow = ((int64_t)layer * A + a) * Hq + kvh * G + g;   // output / suffix row

    // the suffix partial is independent of the pieces: start its loads first
    float2 sml = make_float2(-INFINITY, 0.0f);
    typename V::T sv{};
    if (sfx_ml) {
        sml = reinterpret_cast<const float2*>(sfx_ml)[orow];
        sv = reinterpret_cast<const typename V::T*>(sfx_acc + orow * D)[lane];
    }

    float M = -INFINITY, L = 0.0f;
    float o[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o[e] = 0.0f;
    for (int s0 = 0; s0 < pieces; s0 += kMergeBatch) {
        float2 ml[kMergeBatch];
        typename V::T v[kMergeBatch];
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
            ml[i] = make_float2(-INFINITY, 0.0f);
            if (s0 + i < pieces) {
                const int64_t pr = first + (int64_t)(s0 + i) * stride;
                ml[i] = reinterpret_cast<const float2*>(ws_ml)[pr];
                v[i] = reinterpret_cast<const typename V::T*>(ws_acc + pr * D)[lane];
            }
        }
        float Mn = M;
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) Mn = fmaxf(Mn, ml[i].x);
        if (Mn == -INFINITY) continue;
        const float c = exp2f(M - Mn);  // 0 while nothing has been merged
        L *= c;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] *= c;
#pragma unroll
        for (int i = 0; i < kMergeBatch; ++i) {
            if (ml[i].x == -INFINITY) continue;
            const float w = exp2f(ml[i].x - Mn);
            L = fmaf(w, ml[i].y, L);
            float x[EPL];
            V::to(v[i], x);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] = fmaf(w, x[e], o[e]);
        }
        M = Mn;
    }
    finish_row<D>(o, M, L, sml, sv, lane);
    reinterpret_cast<typename V::T*>(out + orow * D)[lane] = V::from(o);
}

// Merge for the tensor-core partition: blockIdx.x is a segment (kv-head unit x row group of up to 64
// rows), blockIdx.y a block of 16 of its rows, two rows per warp. The segment's pieces are the slots
// s + c for the CTAs c whose contiguous tile ranges overlap the segment (at most two for segments
// longer than a CTA's range, the usual case). Index arithmetic is done once per block, and a warp
// issues the loads of all its rows' first two pieces (and suffix partials) before using any, so the
// whole merge costs about one memory round trip per warp.
constexpr int kMergeRowsPerWarp = 2;
template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) attend_merge_tc(const float* __restrict__ ws_acc,
                                                                    const float* __restrict__ ws_ml,
                                                                    float* __restrict__ out, int H, int A, int Hq,
                                                                    int Rtot, MergeLayout lay,
                                                                    const float* __restrict__ sfx_acc,
                                                                    const float* __restrict__ sfx_ml) {
    constexpr int EPL = D / 32;
    constexpr int RW = kMergeRowsPerWarp;
    using V = MergeVec<D>;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int s = blockIdx.x;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int unit = s / lay.nrg, rg = s - unit * lay.nrg;
    const int layer = unit / H, kvh = unit - layer * H;
    const int G = Hq / H;
    const int rows = min(lay.RS, Rtot - rg * lay.RS);
    const int64_t x0 = (int64_t)s * lay.nt;                      // the segment's first tile
    const int lo = (int)(((x0 + 1) * lay.nc - 1) / lay.tt);      // CTA holding its first tile
    const int hi = (int)(((x0 + lay.nt) * lay.nc - 1) / lay.tt); // CTA holding its last tile
    const int pieces = hi - lo + 1;
    const int rbase = blockIdx.y * (kMergeWarps * RW) + warp * RW;

    float2 ml[RW][2], sml[RW];
    typename V::T v[RW][2], sv[RW];
    int64_t orow[RW];
#pragma unroll
    for (int k = 0; k < RW; ++k) {
        const int r = rbase + k;
        orow[k] = 0;
        sml[k] = make_float2(-INFINITY, 0.0f);
        ml[k][0] = ml[k][1] = make_float2(-INFINITY, 0.0f);
        if (r < rows) {
            const int R0 = rg * lay.RS + r;
            const int a = R0 / G, g = R0 - a * G;
            orow[k] = ((int64_t)layer * A + a) * Hq + kvh * G + g;
            if (sfx_ml) {
                sml[k] = reinterpret_cast<const float2*>(sfx_ml)[orow[k]];
                sv[k] = reinterpret_cast<const typename V::T*>(sfx_acc + orow[k] * D)[lane];
            }
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (i < pieces) {
                    const int64_t pr = (int64_t)(s + lo + i) * lay.RS + r;
                    ml[k][i] = reinterpret_cast<const float2*>(ws_ml)[pr];
                    v[k][i] = reinterpret_cast<const typename V::T*>(ws_acc + pr * D)[lane];
                }
        }
    }
#pragma unroll
    for (int k = 0; k < RW; ++k) {
        const int r = rbase + k;
        if (r >= rows) continue;
        float M = fmaxf(ml[k][0].x, ml[k][1].x), L = 0.0f;
        float o[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = 0.0f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (ml[k][i].x == -INFINITY) continue;
            const float w = exp2f(ml[k][i].x - M);
            L = fmaf(w, ml[k][i].y, L);
            float x[EPL];
            V::to(v[k][i], x);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] = fmaf(w, x[e], o[e]);
        }
        for (int i = 2; i < pieces; ++i) {   // segments split over more than two CTAs
            const int64_t pr = (int64_t)(s + lo + i) * lay.RS + r;
            const float2 mi = reinterpret_cast<const float2*>(ws_ml)[pr];
            if (mi.x == -INFINITY) continue;
            float x[EPL];
            V::to(reinterpret_cast<const typename V::T*>(ws_acc + pr * D)[lane], x);
            const float Mn = fmaxf(M, mi.x);
            const float c = exp2f(M - Mn), w = exp2f(mi.x - Mn);
            L = fmaf(w, mi.y, L * c);
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[e] = fmaf(w, x[e], o[e] * c);
            M = Mn;
        }
        finish_row<D>(o, M, L, sml[k], sv[k], lane);
        reinterpret_cast<typename V::T*>(out + orow[k] * D)[lane] = V::from(o);
    }
}

template <int D, int RMAX, bool BF16>
polykv_status run_simt(const PoolView& p, const void* q, float* out, int A, int Hq, int R, int64_t n_ctx,
                       float scale, float* ws, int n_splits, int64_t split_len, cudaStream_t st,
                       const SuffixArgs* sfx) {
    using S = SimtSmem<D, RMAX>;
    auto kern = attend_partial_simt<D, RMAX, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kBytes);
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "attend: smem attribute: %s", cudaGetErrorString(e));
    const int U = p.L * p.H;
    float* ws_acc = ws;
    float* ws_ml = ws + (size_t)U * n_splits * R * D;
    dim3 grid(n_splits, U, (R + RMAX - 1) / RMAX);
    kern<<<grid, kThreads, S::kBytes, st>>>(p, static_cast<const uint16_t*>(q), A, Hq, R, n_ctx, split_len, n_splits,
                                            scale * kLog2e, ws_acc, ws_ml);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "attend partial launch: %s", cudaGetErrorString(e));
    if (sfx) {
        const polykv_status ss = launch_attend_suffix(*sfx, BF16 ? POLYKV_BF16 : POLYKV_F16, p.L, A, p.H, Hq, D, scale, st);
        if (ss != POLYKV_OK) return ss;
    }
    return launch_attend_merge(ws_acc, ws_ml, out, U, p.H, A, Hq, R, n_splits, MergeLayout(), D, st,
                               sfx ? sfx->acc : nullptr, sfx ? sfx->ml : nullptr);
}

template <int D, bool BF16>
polykv_status dispatch_rows(const PoolView& p, const void* q, float* out, int A, int Hq, int R, int64_t n_ctx,
                            float scale, float* ws, int n_splits, int64_t split_len, cudaStream_t st,
                            const SuffixArgs* sfx) {
    if (R <= 8) return run_simt<D, 8, BF16>(p, q, out, A, Hq, R, n_ctx, scale, ws, n_splits, split_len, st, sfx);
    if (R <= 16) return run_simt<D, 16, BF16>(p, q, out, A, Hq, R, n_ctx, scale, ws, n_splits, split_len, st, sfx);
    if (R <= 32) return run_simt<D, 32, BF16>(p, q, out, A, Hq, R, n_ctx, scale, ws, n_splits, split_len, st, sfx);
    return run_simt<D, kMaxRowsPerCta, BF16>(p, q, out, A, Hq, R, n_ctx, scale, ws, n_splits, split_len, st, sfx);
}

int64_t split_length(const PoolView& p, int rows, int64_t n_ctx) {
    const int U = p.L * p.H;
    const int chunks = (rows + kMaxRowsPerCta - 1) / kMaxRowsPerCta;
    const int64_t want_ctas = 4 * 152;
    int64_t s = (want_ctas + (int64_t)U * chunks - 1) / ((int64_t)U * chunks);
    const int64_t tiles = (n_ctx + kTT - 1) / kTT;
    s = std::max<int64_t>(1, std::min<int64_t>(s, tiles));
    const int64_t per = (n_ctx + s - 1) / s;
    return ((per + kTT - 1) / kTT) * kTT;
}

}  // namespace

polykv_status launch_attend_merge(const float* ws_acc, const float* ws_ml, float* out, int U, int H, int A, int Hq,
                                  int R, int n_slots, const MergeLayout& lay, int D, cudaStream_t st,
                                  const float* sfx_acc, const float* sfx_ml) {
    const int64_t warps = (int64_t)U * R;
    const unsigned blocks = (unsigned)((warps + kMergeWarps - 1) / kMergeWarps);
    // programmatic dependent launch: the merge's CTAs may be scheduled while the partial kernel's last
    // CTAs finish; each waits (griddepcontrol.wait) for the partials before reading them
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(32 * kMergeWarps);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (lay.nc > 0 && lay.RS > 8) {
        // many rows per segment and few pieces (the tensor-core partition): two rows per warp
        constexpr int rows_per_block = kMergeWarps * kMergeRowsPerWarp;
        cfg.gridDim = dim3((unsigned)((int64_t)U * lay.nrg), (unsigned)((lay.RS + rows_per_block - 1) / rows_per_block));
        e = D == 128 ? cudaLaunchKernelEx(&cfg, attend_merge_tc<128>, ws_acc, ws_ml, out, H, A, Hq, R, lay, sfx_acc, sfx_ml)
                     : cudaLaunchKernelEx(&cfg, attend_merge_tc<64>, ws_acc, ws_ml, out, H, A, Hq, R, lay, sfx_acc, sfx_ml);
    } else {
        e = D == 128 ? cudaLaunchKernelEx(&cfg, attend_merge<128>, ws_acc, ws_ml, out, U, H, A, Hq, R, n_slots, lay,
                                          sfx_acc, sfx_ml)
                     : cudaLaunchKernelEx(&cfg, attend_merge<64>, ws_acc, ws_ml, out, U, H, A, Hq, R, n_slots, lay,
                                          sfx_acc, sfx_ml);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "attend merge launch: %s", cudaGetErrorString(e));
    return POLYKV_OK;
}

int attend_simt_splits(const PoolView& p, int rows, int64_t n_ctx) {
    const int64_t len = split_length(p, rows, n_ctx);
    return (int)((n_ctx + len - 1) / len);
}

size_t attend_simt_workspace(const PoolView& p, int rows, int64_t n_ctx) {
    const size_t S = (size_t)attend_simt_splits(p, rows, n_ctx);
    const size_t U = (size_t)p.L * p.H;
    return sizeof(float) * U * S * (size_t)rows * ((size_t)p.d + 2);
}

polykv_status launch_attend_simt(const PoolView& p, polykv_dtype dt, const void* q, float* out, int n_agents,
                                 int n_q_heads, int64_t n_ctx, float scale, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, const SuffixArgs* sfx) {
    const int R = n_agents * (n_q_heads / p.H);
    const int64_t len = split_length(p, R, n_ctx);
    const int S = (int)((n_ctx + len - 1) / len);
    if (ws_bytes < attend_simt_workspace(p, R, n_ctx))
        return set_error(POLYKV_E_BUFFER_TOO_SMALL, "attend: workspace %zu < %zu bytes", ws_bytes,
                         attend_simt_workspace(p, R, n_ctx));
    float* w = static_cast<float*>(ws);
    const bool bf = dt == POLYKV_BF16;
    if (p.d == 128)
        return bf ? dispatch_rows<128, true>(p, q, out, n_agents, n_q_heads, R, n_ctx, scale, w, S, len, stream, sfx)
                  : dispatch_rows<128, false>(p, q, out, n_agents, n_q_heads, R, n_ctx, scale, w, S, len, stream, sfx);
    if (p.d == 64)
        return bf ? dispatch_rows<64, true>(p, q, out, n_agents, n_q_heads, R, n_ctx, scale, w, S, len, stream, sfx)
                  : dispatch_rows<64, false>(p, q, out, n_agents, n_q_heads, R, n_ctx, scale, w, S, len, stream, sfx);
    return set_error(POLYKV_E_UNSUPPORTED, "attend: head_dim %d", p.d);
}

}  // namespace polykv

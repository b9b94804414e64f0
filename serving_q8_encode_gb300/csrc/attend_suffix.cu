// Private per-agent keys/values attended together with the shared compressed pool under ONE
// softmax: a suffix of uncompressed recent tokens, or (query-chunk mode) a chunk of query tokens
// that each carry their own key/value, seen causally.
//
// Each agent appends its own recent tokens after the shared context; those
// are not part of the compressed pool (the PolyKV abstract's pool is the shared
// context written once). For every (layer, agent, kv head) this kernel scores
// the agent's G query heads against its suffix keys and accumulates the suffix
// values in the ORIGINAL basis, producing one online-softmax partial (running
// max m in log2 units, sum l, unnormalised accumulator) per query head. The
// merge kernel combines it with the pool partials (whose accumulators are in
// the rotated basis) after the pool part's inverse FWHT.
#include <cmath>

#include "polykv_internal.cuh"

namespace polykv {
namespace {

constexpr int kSfxTile = 128;   // suffix tokens per tile (one per thread for the scores)
constexpr int kSfxThreads = 128;

__device__ __forceinline__ float bits_to_float(uint16_t b, bool bf16) {
    return bf16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
}

// Shared-memory tile of the suffix: keys with rows padded by 16 bytes (a thread reads its token's row;
// the padding spreads eight consecutive rows over distinct banks) and values unpadded (a thread reads
// one column; consecutive threads read consecutive 2-byte elements).
template <int D>
struct SfxTileSmem {
    static constexpr int kKRow = 2 * D + 16;
    static constexpr int kKBytes = kSfxTile * kKRow;
    static constexpr int kVBytes = kSfxTile * 2 * D;
    static constexpr int kBytes = kKBytes + kVBytes;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// grid: one block per (layer, agent, kv head); block: 128 threads. Each 128-token tile of the agent's
// keys and values is copied into shared memory with coalesced 16-byte asynchronous copies; the scores
// (thread = token) and the value accumulation (thread = head dim) then read shared memory only.
template <int D, int GMAX, bool BF16>
__global__ void __launch_bounds__(kSfxThreads) suffix_partial(const uint16_t* __restrict__ q,
                                                              const uint16_t* __restrict__ sk,
                                                              const uint16_t* __restrict__ sv, int A, int H, int Hq,
                                                              int64_t S, float scale_log2, float* __restrict__ acc_out,
                                                              float* __restrict__ ml_out) {
    using T = SfxTileSmem<D>;
    extern __shared__ __align__(16) unsigned char sfx_smem[];
    __shared__ __align__(16) float qs[GMAX][D];
    __shared__ __align__(16) float ps[kSfxTile][GMAX];   // probabilities, token-major
    __shared__ float red[4][GMAX];
    __shared__ float m_s[GMAX], l_s[GMAX], al_s[GMAX];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = Hq / H;
    const int unit = blockIdx.x;                    // (layer * A + a) * H + h
    const int h = unit % H;
    const int la = unit / H;                        // layer * A + a
    const uint16_t* kbase = sk + (int64_t)unit * S * D;
    const uint16_t* vbase = sv + (int64_t)unit * S * D;
    const uint32_t ks_u = (uint32_t)__cvta_generic_to_shared(sfx_smem);
    const uint32_t vs_u = ks_u + T::kKBytes;
    const uint16_t* Vs = reinterpret_cast<const uint16_t*>(sfx_smem + T::kKBytes);

    for (int i = tid; i < GMAX * D; i += kSfxThreads) {
        const int g = i / D, j = i % D;
        qs[g][j] = g < G ? bits_to_float(q[((int64_t)la * Hq + h * G + g) * D + j], BF16) : 0.0f;
    }
    if (tid < GMAX) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.0f;
    }
    constexpr int CPT = (D + kSfxThreads - 1) / kSfxThreads;   // accumulator columns per thread
    float acc[GMAX][CPT];
#pragma unroll
    for (int g = 0; g < GMAX; ++g)
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[g][c] = 0.0f;

    constexpr int kChunksPerRow = D / 8;            // 16-byte chunks per key or value row
    for (int64_t t0 = 0; t0 < S; t0 += kSfxTile) {
        const int tmax = (int)((S - t0) < kSfxTile ? (S - t0) : kSfxTile);
        // ---- the tile's keys and values into shared memory (rows past the suffix are not copied)
        for (int c = tid; c < tmax * kChunksPerRow; c += kSfxThreads) {
            const int row = c / kChunksPerRow, col = c - row * kChunksPerRow;
            const int64_t goff = (t0 + row) * D + col * 8;
            cp_async16(ks_u + (uint32_t)(row * T::kKRow + col * 16), kbase + goff);
            cp_async16(vs_u + (uint32_t)(row * 2 * D + col * 16), vbase + goff);
        }
        cp_async_wait_all();
        __syncthreads();

        // ---- scores: thread = token
        const bool valid = tid < tmax;
        float x[GMAX];
#pragma unroll
        for (int g = 0; g < GMAX; ++g) x[g] = 0.0f;
        if (valid) {
            const unsigned char* krow = sfx_smem + tid * T::kKRow;
#pragma unroll 4
            for (int c = 0; c < kChunksPerRow; ++c) {
                const uint4 w = *reinterpret_cast<const uint4*>(krow + 16 * c);
                const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                float kf[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kf[2 * e] = bits_to_float((uint16_t)(wv[e] & 0xFFFFu), BF16);
                    kf[2 * e + 1] = bits_to_float((uint16_t)(wv[e] >> 16), BF16);
                }
#pragma unroll
                for (int g = 0; g < GMAX; ++g) {
                    const float4 qa = *reinterpret_cast<const float4*>(&qs[g][8 * c]);
                    const float4 qb = *reinterpret_cast<const float4*>(&qs[g][8 * c + 4]);
                    float s = x[g];
                    s = fmaf(qa.x, kf[0], s);
                    s = fmaf(qa.y, kf[1], s);
                    s = fmaf(qa.z, kf[2], s);
                    s = fmaf(qa.w, kf[3], s);
                    s = fmaf(qb.x, kf[4], s);
                    s = fmaf(qb.y, kf[5], s);
                    s = fmaf(qb.z, kf[6], s);
                    s = fmaf(qb.w, kf[7], s);
                    x[g] = s;
                }
            }
        }
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            x[g] = valid ? x[g] * scale_log2 : -INFINITY;
            float v = x[g];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) red[warp][g] = v;
        }
        __syncthreads();
        if (tid < GMAX) {
            const float mt = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
            const float mo = m_s[tid];
            const float mn = fmaxf(mo, mt);
            al_s[tid] = mo == -INFINITY ? 0.0f : exp2f(mo - mn);
            m_s[tid] = mn;
        }
        __syncthreads();
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            const float p = valid ? exp2f(x[g] - m_s[g]) : 0.0f;
            ps[tid][g] = p;
            float v = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[warp][g] = v;
        }
        __syncthreads();
        if (tid < GMAX) l_s[tid] = l_s[tid] * al_s[tid] + red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];
        // ---- values: thread = column
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const int j = tid + c * kSfxThreads;
            if (j < D) {
#pragma unroll
                for (int g = 0; g < GMAX; ++g) acc[g][c] *= al_s[g];
#pragma unroll 4
                for (int tt = 0; tt < tmax; ++tt) {
                    const float vv = bits_to_float(Vs[tt * D + j], BF16);
#pragma unroll
                    for (int g4 = 0; g4 < GMAX; g4 += 4) {
                        const float4 p4 = *reinterpret_cast<const float4*>(&ps[tt][g4]);
                        acc[g4][c] = fmaf(p4.x, vv, acc[g4][c]);
                        acc[g4 + 1][c] = fmaf(p4.y, vv, acc[g4 + 1][c]);
                        acc[g4 + 2][c] = fmaf(p4.z, vv, acc[g4 + 2][c]);
                        acc[g4 + 3][c] = fmaf(p4.w, vv, acc[g4 + 3][c]);
                    }
                }
            }
        }
        __syncthreads();   // the tile's shared memory is reused by the next tile's copies
    }
    // partial per query head hq = h*G + g of agent a
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int j = tid + c * kSfxThreads;
        if (j < D)
            for (int g = 0; g < G && g < GMAX; ++g) acc_out[((int64_t)la * Hq + h * G + g) * D + j] = acc[g][c];
    }
    if (tid < G) {
        ml_out[((int64_t)la * Hq + h * G + tid) * 2] = m_s[tid];
        ml_out[((int64_t)la * Hq + h * G + tid) * 2 + 1] = l_s[tid];
    }
}

// ---------------------------------------------------------------- query-chunk mode
// Each agent's chunk of C query tokens carries its own keys/values; query token c sees the agent's
// chunk tokens 0..c (plus the pool, merged later). One block per (layer, agent, kv head, block of 32
// query rows r = c * G + g); chunk keys/values go through shared memory in tiles of 64 tokens; one
// warp owns 8 rows (one online-softmax state each), a lane one token of the tile for the scores and
// D/32 head dims for the accumulator. The partial (running max in log2 units, sum, unnormalised
// accumulator in the original basis) goes to the same slots as a suffix partial, with the chunk
// position folded into the agent index (a' = a * C + c).
constexpr int kChT = 64;
constexpr int kChRows = 32;
constexpr int kChThreads = 128;

template <int D>
constexpr size_t chunk_smem_bytes() {
    return sizeof(float) * ((size_t)kChT * (D + 1) + (size_t)kChT * D + (size_t)kChRows * D + 4 * kChT);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kChThreads) chunk_partial(const uint16_t* __restrict__ q,
                                                            const uint16_t* __restrict__ ck,
                                                            const uint16_t* __restrict__ cv, int H, int Hq, int64_t C,
                                                            float scale_log2, float* __restrict__ acc_out,
                                                            float* __restrict__ ml_out) {
    extern __shared__ float chs[];
    float* Ks = chs;                       // [kChT][D + 1]
    float* Vs = Ks + kChT * (D + 1);       // [kChT][D]
    float* Qs = Vs + kChT * D;             // [kChRows][D]
    float* Ps = Qs + kChRows * D;          // [4 warps][kChT]
    constexpr int RW = kChRows / 4;        // rows per warp
    constexpr int DPL = D / 32;            // accumulator dims per lane
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = Hq / H;
    const int64_t unit = blockIdx.x;       // (layer * A + a) * H + h
    const int h = (int)(unit % H);
    const int64_t la = unit / H;           // layer * A + a
    const int64_t rows = C * G;
    const int64_t r0 = (int64_t)blockIdx.y * kChRows;
    const uint16_t* kb = ck + unit * C * D;
    const uint16_t* vb = cv + unit * C * D;

    for (int i = tid; i < kChRows * D; i += kChThreads) {
        const int64_t r = r0 + i / D;
        float x = 0.0f;
        if (r < rows) {
            const int64_t c = r / G;
            const int g = (int)(r % G);
            x = bits_to_float(q[((la * C + c) * Hq + h * G + g) * D + i % D], BF16);
        }
        Qs[i] = x;
    }
    float m[RW], l[RW], acc[RW][DPL];
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.0f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[i][e] = 0.0f;
    }
    const int64_t r_last = (r0 + kChRows < rows ? r0 + kChRows : rows) - 1;
    const int64_t c_max = r_last / G;
    for (int64_t t0 = 0; t0 <= c_max; t0 += kChT) {
        __syncthreads();
        for (int i = tid; i < kChT * D; i += kChThreads) {
            const int tk = i / D, dd = i % D;
            const bool ok = t0 + tk < C;
            Ks[tk * (D + 1) + dd] = ok ? bits_to_float(kb[(t0 + tk) * D + dd], BF16) : 0.0f;
            Vs[tk * D + dd] = ok ? bits_to_float(vb[(t0 + tk) * D + dd], BF16) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RW; ++i) {
            const int ri = warp * RW + i;
            const int64_t r = r0 + ri;
            if (r >= rows) continue;               // warp-uniform
            const int64_t c = r / G;
            if (t0 > c) continue;                  // no visible token in this tile (warp-uniform)
            const float* qr = Qs + ri * D;
            float x0 = 0.0f, x1 = 0.0f;
#pragma unroll 8
            for (int dd = 0; dd < D; ++dd) {
                x0 = fmaf(qr[dd], Ks[lane * (D + 1) + dd], x0);
                x1 = fmaf(qr[dd], Ks[(lane + 32) * (D + 1) + dd], x1);
            }
            x0 = (t0 + lane <= c) ? x0 * scale_log2 : -INFINITY;
            x1 = (t0 + lane + 32 <= c) ? x1 * scale_log2 : -INFINITY;
            float tmax = fmaxf(x0, x1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
            const float mn = fmaxf(m[i], tmax);
            const float alpha = m[i] == -INFINITY ? 0.0f : exp2f(m[i] - mn);
            const float p0 = exp2f(x0 - mn), p1 = exp2f(x1 - mn);
            float ps = p0 + p1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            l[i] = l[i] * alpha + ps;
            m[i] = mn;
            Ps[warp * kChT + lane] = p0;
            Ps[warp * kChT + lane + 32] = p1;
            __syncwarp();
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[i][e] *= alpha;
            const int tmaxk = (int)((c - t0 + 1) < kChT ? (c - t0 + 1) : kChT);
            for (int tk = 0; tk < tmaxk; ++tk) {
                const float pp = Ps[warp * kChT + tk];
#pragma unroll
                for (int e = 0; e < DPL; ++e) acc[i][e] = fmaf(pp, Vs[tk * D + lane * DPL + e], acc[i][e]);
            }
            __syncwarp();
        }
    }
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        const int64_t r = r0 + warp * RW + i;
        if (r >= rows) continue;
        const int64_t c = r / G;
        const int g = (int)(r % G);
        const int64_t orow = (la * C + c) * Hq + h * G + g;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc_out[orow * D + lane * DPL + e] = acc[i][e];
        if (lane == 0) {
            ml_out[orow * 2] = m[i];
            ml_out[orow * 2 + 1] = l[i];
        }
    }
}

template <int D, bool BF16>
polykv_status run_chunk(const SuffixArgs& a, int L, int A_virtual, int H, int Hq, float scale, cudaStream_t st) {
    const int G = Hq / H;
    const int64_t C = a.chunk;
    const int64_t A = A_virtual / C;
    const int64_t nblk_rows = (C * G + kChRows - 1) / kChRows;
    if (nblk_rows > 65535) return set_error(POLYKV_E_UNSUPPORTED, "chunk: %lld query rows per kv head", (long long)(C * G));
    const dim3 grid((unsigned)((int64_t)L * A * H), (unsigned)nblk_rows);
    constexpr size_t smem = chunk_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(chunk_partial<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "chunk: smem attribute: %s", cudaGetErrorString(e));
    chunk_partial<D, BF16><<<grid, kChThreads, smem, st>>>(
        static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k), static_cast<const uint16_t*>(a.v), H, Hq,
        C, scale * 1.4426950408889634f, a.acc, a.ml);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "chunk launch: %s", cudaGetErrorString(e));
    return POLYKV_OK;
}

template <int D, int GMAX, bool BF16>
polykv_status launch_suffix_partial(const SuffixArgs& a, int L, int A, int H, int Hq, float sl, cudaStream_t st) {
    constexpr int smem = SfxTileSmem<D>::kBytes;
    auto kern = suffix_partial<D, GMAX, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "suffix: smem attribute: %s", cudaGetErrorString(e));
    const unsigned blocks = (unsigned)((int64_t)L * A * H);
    kern<<<blocks, kSfxThreads, smem, st>>>(static_cast<const uint16_t*>(a.q), static_cast<const uint16_t*>(a.k),
                                            static_cast<const uint16_t*>(a.v), A, H, Hq, a.len, sl, a.acc, a.ml);
    e = cudaGetLastError();
    if (e != cudaSuccess) return set_error(POLYKV_E_CUDA, "suffix launch: %s", cudaGetErrorString(e));
    return POLYKV_OK;
}

template <int D, bool BF16>
polykv_status run_suffix(const SuffixArgs& a, int L, int A, int H, int Hq, float scale, cudaStream_t st) {
    const int G = Hq / H;
    const float sl = scale * 1.4426950408889634f;
    if (G <= 4) return launch_suffix_partial<D, 4, BF16>(a, L, A, H, Hq, sl, st);
    return launch_suffix_partial<D, 16, BF16>(a, L, A, H, Hq, sl, st);
}

}  // namespace

polykv_status launch_attend_suffix(const SuffixArgs& a, polykv_dtype dt, int L, int A, int H, int Hq, int D,
                                   float scale, cudaStream_t st) {
    const bool bf = dt == POLYKV_BF16;
    if (a.chunk > 0) {
        if (D == 128) return bf ? run_chunk<128, true>(a, L, A, H, Hq, scale, st) : run_chunk<128, false>(a, L, A, H, Hq, scale, st);
        if (D == 64) return bf ? run_chunk<64, true>(a, L, A, H, Hq, scale, st) : run_chunk<64, false>(a, L, A, H, Hq, scale, st);
        return set_error(POLYKV_E_UNSUPPORTED, "chunk: head_dim %d", D);
    }
    if (D == 128) return bf ? run_suffix<128, true>(a, L, A, H, Hq, scale, st) : run_suffix<128, false>(a, L, A, H, Hq, scale, st);
    if (D == 64) return bf ? run_suffix<64, true>(a, L, A, H, Hq, scale, st) : run_suffix<64, false>(a, L, A, H, Hq, scale, st);
    return set_error(POLYKV_E_UNSUPPORTED, "suffix: head_dim %d", D);
}

}  // namespace polykv
